"""The e4m3 tensor-core kernel's pipeline protocol (gemm_fp8.cuh), modelled on the CPU with
pipeline_model.py, for each kind of launch it has:
- weights read natively (e4m3, e5m2, e2m1: two 128-k sub-tiles a step, no rewrite), where the
  producer reuses a raw stage once the step-done barrier of the step RAWST before completes;
- weights rewritten in shared memory (int8: one sub-tile a step; int4, uint4: two);
- activations as e4m3 rows or as the split pass's planes (a TMA copy into the operand ring, and a
  token-scale warp), or split inside the kernel (four split warps between a bf16 row ring and the
  operand ring).
Every wait must pass on the phase it means, every arrival land in its phase, and every schedule
run to its end. The ring depths are those of the kernel's configuration, whose formulas the test
checks in the source first."""

import os

import pytest

import pipeline_model as model
from pipeline_model import ring, wait_full

SRC = os.path.join(os.path.dirname(__file__), "..", "moe_grouped_matrix_gb300", "csrc", "gemm_fp8.cuh")


def test_the_modelled_depths_are_the_kernel_s_own():
    text = open(SRC).read()
    for line in ("static constexpr int QPS = F == WFmt::kInt8 ? 1 : 2;",
                 "static constexpr int RAWST = 4;",
                 "static constexpr int CST = kConv ? 2 : 0;",
                 "static constexpr int NACC = QPS == 2 ? 4 : 8;",
                 "static constexpr int RTS = kA8 ? 0 : 2, BST = kA8 ? 4 : 2, NSC = 8;",
                 "static constexpr int NDONE = NACC;",
                 "static constexpr int kConvWarps = kA8 ? 1 : 4;",
                 "static constexpr int kWConvWarps = kConv ? (kA8 ? 8 : 4) : 0;",
                 "static constexpr int kIssuers = 2;"):
        assert line in text, line


def config(qps, conv, a8, issuers=2, cst=None):
    nacc = 4 if qps == 2 else 8
    return dict(RAWST=4, CST=(2 if conv else 0) if cst is None else cst, NACC=nacc, NDONE=nacc,
                RTS=0 if a8 else 2, BST=4 if a8 else 2, NSC=8, SPLITW=1 if a8 else 4,
                WCONV=(8 if a8 else 4) if conv else 0, ISS=issuers, conv=conv, a8=a8)


def roles(c, steps):
    RAWST, CST, NACC, NDONE, RTS, BST, NSC = (c[x] for x in ("RAWST", "CST", "NACC", "NDONE", "RTS", "BST", "NSC"))
    conv, a8, ISS, SPLITW, WCONV = c["conv"], c["a8"], c["ISS"], c["SPLITW"], c["WCONV"]
    assert conv or RAWST == NDONE  # the kernel's own static_assert
    rawfull, rawempty = ring("rawfull", RAWST, 1), ring("rawempty", RAWST, max(WCONV, 1))
    convfull, stepdone = ring("convfull", max(CST, 1), max(WCONV, 1)), ring("stepdone", NDONE, 1)
    rfull, rempty = ring("rfull", max(RTS, 1), 1), ring("rempty", max(RTS, 1), SPLITW)
    bfull = ring("bfull", BST, 1 if a8 else SPLITW)
    sfull, sempty = ring("sfull", NSC, SPLITW), ring("sempty", NSC, 4)
    acce = ring("acce", NACC, 4)

    def step_done(j, depth):
        if j >= depth:
            yield wait_full(stepdone[(j - depth) % NDONE], (j - depth) // NDONE)

    def producer():
        for j in range(steps):
            # raw stage j % RAWST is free once its last reader is done: the rewrite, or the MMAs
            # of step j - RAWST (the step-done barrier of the same index, previous phase)
            free = rawempty[j % RAWST] if conv else stepdone[j % RAWST]
            yield wait_full(free, j // RAWST - 1)
            yield ("async", None, rawfull[j % RAWST], j // RAWST)
            if a8:
                yield from step_done(j, BST)
                yield ("async", None, bfull[j % BST], j // BST)
            else:
                yield wait_full(rempty[j % RTS], j // RTS - 1)
                yield ("async", None, rfull[j % RTS], j // RTS)

    def issuer(mine):
        for j in range(steps):
            if j % ISS != mine:
                continue
            yield wait_full(acce[j % NACC], j // NACC - 1)
            if conv:
                yield wait_full(convfull[j % CST], j // CST)
            else:
                yield wait_full(rawfull[j % RAWST], j // RAWST)
            yield wait_full(bfull[j % BST], j // BST)
            yield ("async", f"issuer{mine}", stepdone[j % NACC], j // NACC)

    def epilogue():
        for j in range(steps):
            yield wait_full(stepdone[j % NACC], j // NACC)
            yield wait_full(sfull[j % NSC], j // NSC)
            yield ("arrive", acce[j % NACC], j // NACC)
            yield ("arrive", sempty[j % NSC], j // NSC)

    def token_scales():  # e4m3 rows or split-pass planes: one warp
        for j in range(steps):
            yield wait_full(sempty[j % NSC], j // NSC - 1)
            yield ("async", None, sfull[j % NSC], j // NSC)

    def split_warp():  # the split inside the kernel: bf16 rows in, operand rows and scales out
        for j in range(steps):
            yield wait_full(rfull[j % RTS], j // RTS)
            yield from step_done(j, BST)
            yield wait_full(sempty[j % NSC], j // NSC - 1)
            yield ("arrive", rempty[j % RTS], j // RTS)
            yield ("arrive", bfull[j % BST], j // BST)
            yield ("arrive", sfull[j % NSC], j // NSC)

    def rewrite():
        for j in range(steps):
            yield wait_full(rawfull[j % RAWST], j // RAWST)
            yield from step_done(j, CST)
            yield ("arrive", rawempty[j % RAWST], j // RAWST)
            yield ("arrive", convfull[j % CST], j // CST)

    gens = [producer()] + [issuer(i) for i in range(ISS)] + [epilogue() for _ in range(4)]
    gens += [token_scales()] if a8 else [split_warp() for _ in range(SPLITW)]
    gens += [rewrite() for _ in range(WCONV)]
    return gens


KINDS = {
    "native, e4m3 or split-pass rows": config(2, False, True),
    "native, split in the kernel": config(2, False, False),
    "int8 rewrite, e4m3 or split-pass rows": config(1, True, True),
    "int8 rewrite, split in the kernel": config(1, True, False),
    "4-bit rewrite, e4m3 or split-pass rows": config(2, True, True),
    "4-bit rewrite, split in the kernel": config(2, True, False),
}


@pytest.mark.parametrize("kind", sorted(KINDS))
def test_shipped_rings_never_alias(kind):
    for seed in range(30):
        errors = model.run(roles(KINDS[kind], 29), seed)
        assert not errors, (kind, seed, errors[:3])


def test_more_issuers_than_the_rewrite_ring_is_caught():
    # the same kernel with 3 issuers: the 2-deep rewrite ring is then shallower than the issuer
    # count, and the model must see waits pass early
    found = [e for seed in range(30) for e in model.run(roles(config(1, True, True, issuers=3), 29), seed)]
    assert any("convfull" in e and "passed at" in e for e in found), found[:3]
