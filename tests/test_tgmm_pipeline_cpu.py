"""The tgmm kernel's pipeline protocol (tgmm.cu), modelled on the CPU with pipeline_model.py: a
TMA producer filling STAGES operand stages per 64-row chunk, one MMA warp accumulating each
output tile into one of two TMEM accumulators, and four epilogue warps draining them.  Tiles of
an empty group use no chunk and no accumulator: the producer, the MMA warp and the epilogue must
all skip them, or the accumulator ring falls out of step.  Every wait must pass on the phase it
means, every arrival land in its phase, and every schedule run to its end, for ragged groups with
empty ones among them."""

import os
import random
import re

import pytest

import pipeline_model as model
from pipeline_model import ring, wait_full

SRC = os.path.join(os.path.dirname(__file__), "..", "moe_grouped_matrix_gb300", "csrc", "tgmm.cu")


def stages():
    m = re.search(r"constexpr int STAGES = (\d+);", open(SRC).read())
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


def ragged(seed, items=24):
    rng = random.Random(seed)
    return [rng.choice((0, 0, 1, 2, 3, 5, 9)) for _ in range(items)]


def test_shipped_protocol_with_empty_groups():
    n = stages()
    for seed in range(60):
        errors = model.run(roles(ragged(seed), n), seed)
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
