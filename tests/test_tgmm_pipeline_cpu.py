"""The tgmm kernels' pipeline protocols (tgmm.cu, and the SM-pair tgmm_2sm.cu), modelled on the
CPU with pipeline_model.py: a TMA producer filling STAGES operand stages per 64-row chunk, one
MMA warp accumulating each output tile into one of two TMEM accumulators, and four epilogue warps
draining them.  In the pair kernel both CTAs' producers fill their halves of a stage, whose bytes
complete on the leader's full barrier; the leader's MMA commits go to both CTAs, and both CTAs'
epilogue warps free an accumulator on the leader's barrier.  Tiles of an empty group use no
chunk and no accumulator: the producer, the MMA warp and the epilogue must all skip them, or the
accumulator ring falls out of step.  Every wait must pass on the phase it
means, every arrival land in its phase, and every schedule run to its end, for ragged groups with
empty ones among them."""

import os
import random
import re

import pytest

import pipeline_model as model
from pipeline_model import Barrier, ring, wait_full

CSRC = os.path.join(os.path.dirname(__file__), "..", "moe_grouped_matrix_gb300", "csrc")


def stages(src="tgmm.cu"):
    m = re.search(r"constexpr int STAGES = (\d+);", open(os.path.join(CSRC, src)).read())
    assert m
    return int(m.group(1))


def roles(chunks, n_stages, epilogue_skips_empty=True):
    """chunks: the 64-row chunk count of each work item's group, in the CTA's order."""
    full, empty = ring("full", n_stages, 1), ring("empty", n_stages, 1)
    accf, acce = ring("accf", 2, 1), ring("acce", 2, 4)

    def producer():
        s = 0
        for c in chunks:
            for _ in range(c):
                yield wait_full(empty[s % n_stages], s // n_stages - 1)
                yield ("async", None, full[s % n_stages], s // n_stages)
                s += 1

    def mma():
        s = t = 0
        for c in chunks:
            if c == 0:
                continue  # the epilogue writes zeros; no accumulator is used
            yield wait_full(acce[t % 2], t // 2 - 1)
            for _ in range(c):
                yield wait_full(full[s % n_stages], s // n_stages)
                yield ("async", "mma", empty[s % n_stages], s // n_stages)
                s += 1
            yield ("async", "mma", accf[t % 2], t // 2)
            t += 1

    def epilogue():
        t = 0
        for c in chunks:
            if c == 0 and epilogue_skips_empty:
                continue
            yield wait_full(accf[t % 2], t // 2)
            yield ("arrive", acce[t % 2], t // 2)
            t += 1

    return [producer(), mma()] + [epilogue() for _ in range(4)]


def pair_roles(chunks, n_stages):
    full = [Barrier(f"full{s}", 3) for s in range(n_stages)]  # the leader's: arm + both halves
    empty = [ring(f"empty[cta{c}]", n_stages, 1) for c in range(2)]
    accf = [ring(f"accf[cta{c}]", 2, 1) for c in range(2)]
    acce = ring("acce", 2, 8)

    def producer(cta):
        s = 0
        for c in chunks:
            for _ in range(c):
                yield wait_full(empty[cta][s % n_stages], s // n_stages - 1)
                if cta == 0:
                    yield ("arrive", full[s % n_stages], s // n_stages)
                yield ("async", None, full[s % n_stages], s // n_stages)
                s += 1

    def mma():
        s = t = 0
        for c in chunks:
            if c == 0:
                continue  # the epilogues write zeros; no accumulator is used
            yield wait_full(acce[t % 2], t // 2 - 1)
            for _ in range(c):
                yield wait_full(full[s % n_stages], s // n_stages)
                for cta in range(2):
                    yield ("async", "mma", empty[cta][s % n_stages], s // n_stages)
                s += 1
            for cta in range(2):
                yield ("async", "mma", accf[cta][t % 2], t // 2)
            t += 1

    def epilogue(cta):
        t = 0
        for c in chunks:
            if c == 0:
                continue
            yield wait_full(accf[cta][t % 2], t // 2)
            yield ("arrive", acce[t % 2], t // 2)
            t += 1

    return [producer(0), producer(1), mma()] + [epilogue(c) for c in (0, 1) for _ in range(4)]


def ragged(seed, items=24):
    rng = random.Random(seed)
    return [rng.choice((0, 0, 1, 2, 3, 5, 9)) for _ in range(items)]


def test_shipped_protocol_with_empty_groups():
    n = stages()
    for seed in range(60):
        errors = model.run(roles(ragged(seed), n), seed)
        assert not errors, (seed, errors[:3])


def test_pair_kernel_protocol_with_empty_groups():
    n = stages("tgmm_2sm.cu")
    for seed in range(40):
        errors = model.run(pair_roles(ragged(seed), n), seed)
        assert not errors, (seed, errors[:3])


@pytest.mark.parametrize("n_stages", [1, 2, 4])
def test_any_stage_count_keeps_the_protocol(n_stages):
    # one producer and one MMA warp, each in order: no depth aliases
    for seed in range(20):
        assert not model.run(roles(ragged(seed), n_stages), seed)


def test_an_epilogue_that_waits_on_empty_tiles_is_caught():
    found = []
    for seed in range(20):
        chunks = ragged(seed)
        chunks[3] = 0  # at least one empty group
        found += model.run(roles(chunks, stages(), epilogue_skips_empty=False), seed)
    assert "deadlock" in found or any("passed at" in e for e in found), found[:3]
