"""The fp16-weight kernel's pipeline protocol (gemm_f16w.cu), modelled on the CPU: its roles and
mbarrier rings as the kernel runs them, under many random schedules (pipeline_model.py). Every
wait must pass on the phase it means, every arrival land in its phase, and every schedule run to
its end. The ring depths are read from the kernel source. The rule the model bears out: a ring the MMA issuers wait on must be at least as deep as
there are issuers. Negative controls show that the check catches shallower rings, among them the
layout that returned wrong sums (3 A stages and 5 accumulator slots for MXFP8 with 4 MMA
issuers)."""

import os
import re

import pytest

import pipeline_model as model
from pipeline_model import ring, wait_full

SRC = os.path.join(os.path.dirname(__file__), "..", "moe_grouped_matrix_gb300", "csrc", "gemm_f16w.cu")


def constants():
    text = open(SRC).read()
    out = {}
    for name in ("RAWST", "CST", "BST", "NACC", "NDONE", "NSC", "kIssuers", "kConvWarps", "BT"):
        m = re.search(rf"constexpr (?:int|uint32_t) {name} = (\d+);", text)
        assert m, name
        out[name] = int(m.group(1))
    # MX_NACC = A_COL0 / MX_SLOT_COLS with A_COL0 = NACC * SLOT_COLS and MX_SLOT_COLS = 4 * BT
    slot_cols = int(re.search(r"constexpr int SLOT_COLS = (\d+);", text).group(1))
    assert re.search(r"constexpr int MX_NACC = A_COL0 / MX_SLOT_COLS;", text)
    out["MX_NACC"] = out["NACC"] * slot_cols // (4 * out["BT"])
    return out


def roles(c, steps, spr, nacc, cst):
    """The kernel's roles over `steps` steps of one CTA (spr steps per raw box)."""
    RAWST, BST, NDONE, NSC = c["RAWST"], c["BST"], c["NDONE"], c["NSC"]
    ISS, CONV = c["kIssuers"], c["kConvWarps"]
    rawfull, rawempty = ring("rawfull", RAWST, 1), ring("rawempty", RAWST, CONV)
    convfull, stepdone = ring("convfull", cst, CONV), ring("stepdone", NDONE, 1)
    acce, bfull = ring("acce", nacc, 4), ring("bfull", BST, 1)
    sfull, sempty = ring("sfull", NSC, 1), ring("sempty", NSC, 4)
    boxes = (steps + spr - 1) // spr

    def step_done(j, depth):  # wait_step_done(j, depth): the MMAs of step j - depth are complete
        if j >= depth:
            yield wait_full(stepdone[(j - depth) % NDONE], (j - depth) // NDONE)

    def raw_producer():
        for b in range(boxes):
            # the empty wait: phase b / RAWST - 1 complete (b < RAWST: passes at once)
            yield wait_full(rawempty[b % RAWST], b // RAWST - 1)
            yield ("async", None, rawfull[b % RAWST], b // RAWST)

    def b_producer():
        for j in range(steps):
            yield from step_done(j, BST)
            yield ("async", None, bfull[j % BST], j // BST)

    def issuer(mine):
        for j in range(steps):
            if j % ISS != mine:
                continue
            yield wait_full(acce[j % nacc], j // nacc - 1)
            yield wait_full(convfull[j % cst], j // cst)
            yield wait_full(bfull[j % BST], j // BST)
            # the commit arrives once the step's MMAs complete, in issue order per thread
            yield ("async", f"issuer{mine}", stepdone[j % NDONE], j // NDONE)

    def converter():
        for j in range(steps):
            h, box = j % spr, j // spr
            if h == 0:
                yield wait_full(rawfull[box % RAWST], box // RAWST)
            yield from step_done(j, cst)
            if h == spr - 1 or j + 1 == steps:
                yield ("arrive", rawempty[box % RAWST], box // RAWST)
            yield ("arrive", convfull[j % cst], j // cst)

    def epilogue():
        for j in range(steps):
            yield wait_full(stepdone[j % NDONE], j // NDONE)
            yield wait_full(sfull[j % NSC], j // NSC)
            yield ("arrive", acce[j % nacc], j // nacc)
            yield ("arrive", sempty[j % NSC], j // NSC)

    def scale(mine):
        for j in range(steps):
            if j % 2 != mine:
                continue
            yield wait_full(sempty[j % NSC], j // NSC - 1)
            yield ("async", None, sfull[j % NSC], j // NSC)

    gens = [raw_producer(), b_producer()] + [issuer(i) for i in range(ISS)]
    gens += [converter() for _ in range(CONV)] + [epilogue() for _ in range(4)] + [scale(i) for i in range(2)]
    return gens


def run(c, steps, spr, nacc, cst, seed):
    return model.run(roles(c, steps, spr, nacc, cst), seed)


C = constants()


@pytest.mark.parametrize("fmt,spr,nacc", [("int8", 1, C["NACC"]), ("4-bit", 2, C["NACC"]),
                                           ("MXFP8", 1, C["MX_NACC"])])
def test_shipped_rings_never_alias(fmt, spr, nacc):
    for seed in range(40):
        errors = run(C, 37, spr, nacc, C["CST"], seed)
        assert not errors, (fmt, seed, errors[:3])


def test_a_ring_shallower_than_the_issuer_count_is_caught():
    # 3 A stages and 5 accumulator slots with 4 issuers: the issuer of step j + 3 is another
    # warp than step j's, and begins its wait on the shared A-stage barrier a phase early
    found = [e for seed in range(40) for e in run(C, 37, 1, 5, 3, seed)]
    assert any("convfull" in e and "passed at" in e for e in found), found[:3]
    shallow_b = dict(C, BST=C["kIssuers"] - 1)
    found = [e for seed in range(40) for e in run(shallow_b, 37, 1, C["NACC"], C["CST"], seed)]
    assert any("bfull" in e and "passed at" in e for e in found), found[:3]
    found = [e for seed in range(40) for e in run(C, 37, 1, C["kIssuers"] - 1, C["CST"], seed)]
    assert any("acce" in e for e in found), found[:3]


@pytest.mark.parametrize("nacc,cst", [(5, 4), (4, 5), (6, 6)])
def test_depths_at_least_the_issuer_count_need_not_be_multiples(nacc, cst):
    for seed in range(25):
        assert not run(C, 37, 1, nacc, cst, seed)


def test_the_256k_step_layout_needs_fewer_issuers():
    # The 256-k step layout (4 raw stages, 6 activation stages, 3 A stages of 128 columns and 4
    # accumulator slots: all of TMEM) with 4 issuers: its A-stage ring is shallower than the
    # issuer count, and schedules alias and deadlock, as that build's wait timeouts did on the
    # GPU.  With 3 issuers every schedule runs clean.
    layout = dict(C, RAWST=4, BST=6, NDONE=8, NSC=8)
    found = [e for seed in range(40) for e in run(dict(layout, kIssuers=4), 37, 1, 4, 3, seed)]
    assert "deadlock" in found and any("convfull" in e and "passed at" in e for e in found)
    for seed in range(40):
        assert not run(dict(layout, kIssuers=3), 37, 1, 4, 3, seed)
