"""The bf16 forward kernels' pipeline protocols, modelled on the CPU with pipeline_model.py.

One-SM kernels (gemm_bf16.cu, gemm_bf16_swap.cu): a TMA producer fills STAGES operand stages,
one MMA warp accumulates each tile into one of two TMEM accumulators, four epilogue warps drain
them.

SM-pair kernels (gemm_bf16_2sm.cu, gemm_bf16_2sm_swap.cu): both CTAs' producers copy their halves
of a stage, and both copies complete on the leader's full barrier, which only the leader arms
(expect_tx of both halves' bytes, so a follower copy may land before the leader arms it); the
leader's MMA warp commits each stage to both CTAs' empty barriers and each tile to both CTAs'
accumulator-full barriers; the four epilogue warps of both CTAs free an accumulator on the
leader's barrier.  The follower's producer waits on its own empty barriers only.

Every wait must pass on the phase it means, every arrival land in its phase (a follower copy in
the leader's current phase, in particular), and every schedule run to its end."""

import os
import random
import re

import pytest

import pipeline_model as model
from pipeline_model import Barrier, ring, wait_full

CSRC = os.path.join(os.path.dirname(__file__), "..", "moe_grouped_matrix_gb300", "csrc")


def stages(name):
    m = re.search(r"constexpr int STAGES = (\d+);", open(os.path.join(CSRC, name)).read())
    assert m, name
    return int(m.group(1))


def one_sm_roles(chunks, n_stages):
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
        s = 0
        for t, c in enumerate(chunks):
            yield wait_full(acce[t % 2], t // 2 - 1)
            for _ in range(c):
                yield wait_full(full[s % n_stages], s // n_stages)
                yield ("async", "mma", empty[s % n_stages], s // n_stages)
                s += 1
            yield ("async", "mma", accf[t % 2], t // 2)

    def epilogue():
        for t in range(len(chunks)):
            yield wait_full(accf[t % 2], t // 2)
            yield ("arrive", acce[t % 2], t // 2)

    return [producer(), mma()] + [epilogue() for _ in range(4)]


def pair_roles(chunks, n_stages):
    # the leader's full barriers: its arm (arrive + expect_tx) and the two halves' bytes
    full = [Barrier(f"full{s}", 3) for s in range(n_stages)]
    empty = [ring(f"empty[cta{c}]", n_stages, 1) for c in range(2)]
    accf = [ring(f"accf[cta{c}]", 2, 1) for c in range(2)]
    acce = ring("acce", 2, 8)  # the leader's, one arrival per epilogue warp of both CTAs

    def producer(cta):
        s = 0
        for c in chunks:
            for _ in range(c):
                yield wait_full(empty[cta][s % n_stages], s // n_stages - 1)
                if cta == 0:
                    yield ("arrive", full[s % n_stages], s // n_stages)
                yield ("async", None, full[s % n_stages], s // n_stages)
                s += 1

    def mma():  # the leader's
        s = 0
        for t, c in enumerate(chunks):
            yield wait_full(acce[t % 2], t // 2 - 1)
            for _ in range(c):
                yield wait_full(full[s % n_stages], s // n_stages)
                for cta in range(2):  # one commit, multicast to both CTAs
                    yield ("async", "mma", empty[cta][s % n_stages], s // n_stages)
                s += 1
            for cta in range(2):
                yield ("async", "mma", accf[cta][t % 2], t // 2)

    def epilogue(cta):
        for t in range(len(chunks)):
            yield wait_full(accf[cta][t % 2], t // 2)
            yield ("arrive", acce[t % 2], t // 2)

    return [producer(0), producer(1), mma()] + [epilogue(c) for c in (0, 1) for _ in range(4)]


def tiles(seed, n=20):
    rng = random.Random(seed)
    return [rng.choice((1, 2, 3, 8, 16)) for _ in range(n)]


@pytest.mark.parametrize("src", ["gemm_bf16.cu", "gemm_bf16_swap.cu"])
def test_one_sm_kernels(src):
    n = stages(src)
    for seed in range(30):
        errors = model.run(one_sm_roles(tiles(seed), n), seed)
        assert not errors, (src, seed, errors[:3])


@pytest.mark.parametrize("src", ["gemm_bf16_2sm.cu", "gemm_bf16_2sm_swap.cu"])
def test_pair_kernels(src):
    n = stages(src)
    for seed in range(30):
        errors = model.run(pair_roles(tiles(seed), n), seed)
        assert not errors, (src, seed, errors[:3])


def test_a_follower_producer_without_its_empty_wait_is_caught():
    # a control: a pair whose follower producer skipped its own empty wait would copy into a
    # stage the MMAs may still read, and its bytes would land in the wrong phase
    n = stages("gemm_bf16_2sm.cu")
    found = []
    for seed in range(20):
        chunks = tiles(seed)
        gens = pair_roles(chunks, n)
        follower = gens[1]

        def eager(g=follower):
            for op in g:
                if op[0] == "wait":
                    continue  # no wait at all
                yield op

        gens[1] = eager()
        found += model.run(gens, seed)
    assert any("landed in phase" in e for e in found) or "deadlock" in found, found[:3]
