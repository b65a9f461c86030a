"""The decoding kernel's pipeline protocol (gemm_scaled.cu), modelled on the CPU with
pipeline_model.py, in both of its forms:
- bf16 weights: the TMA producer loads each step's weight tile straight into the operand ring;
- decoded weights (e4m3, MXFP8, NVFP4): the producer fills a raw ring, sixteen decoder warps turn
  each raw tile into a bf16 operand stage in tensor memory, freeing the raw stage as they go.
One MMA warp accumulates SB quant blocks into each of NACC accumulator slots and commits the slot
once; four epilogue warps fold each slot and free it.  Items have any number of quant blocks, so
the last slot of an item may hold fewer than SB.  Every wait must pass on the phase it means,
every arrival land in its phase, and every schedule run to its end."""

import os
import random
import re

import pytest

import pipeline_model as model
from pipeline_model import ring, wait_full

SRC = os.path.join(os.path.dirname(__file__), "..", "moe_grouped_matrix_gb300", "csrc", "gemm_scaled.cu")


def constants():
    text = open(SRC).read()
    out = {}
    for name in ("RSTAGES", "BSTAGES", "SB", "NACC", "kConvWarps"):
        m = re.search(rf"constexpr int {name} = (\d+);", text)
        assert m, name
        out[name] = int(m.group(1))
    assert "static constexpr int kOStages = kE4M3 ? 2 : 3;" in text
    return out


def roles(c, items, decoded, epilogue_per_block=False):
    """items: (quant blocks, steps per block) of each of the CTA's items.  epilogue_per_block: a
    wrong epilogue (for the control) that takes one slot per quant block."""
    R, BS, SB, NACC, CONV = c["RSTAGES"], c["BSTAGES"], c["SB"], c["NACC"], c["kConvWarps"]
    OS = 2 if decoded else 3
    rfull, rempty = ring("rfull", R, 1), ring("rempty", R, CONV)
    ofull, oempty = ring("ofull", OS, CONV if decoded else 1), ring("oempty", OS, 1)
    bfull, bempty = ring("bfull", BS, 1), ring("bempty", BS, 1)
    accf, acce = ring("accf", NACC, 1), ring("acce", NACC, 4)
    steps = sum(nb * spb for nb, spb in items)

    def producer():
        for j in range(steps):
            if decoded:
                yield wait_full(rempty[j % R], j // R - 1)
                yield ("async", None, rfull[j % R], j // R)
            else:
                yield wait_full(oempty[j % OS], j // OS - 1)
                yield ("async", None, ofull[j % OS], j // OS)
            yield wait_full(bempty[j % BS], j // BS - 1)
            yield ("async", None, bfull[j % BS], j // BS)

    def decoder():
        for j in range(steps):
            yield wait_full(rfull[j % R], j // R)
            yield wait_full(oempty[j % OS], j // OS - 1)
            yield ("arrive", rempty[j % R], j // R)
            yield ("arrive", ofull[j % OS], j // OS)

    def mma():
        j = t = 0
        for nb, spb in items:
            for b0 in range(0, nb, SB):
                yield wait_full(acce[t % NACC], t // NACC - 1)
                for _ in range(min(SB, nb - b0) * spb):
                    yield wait_full(ofull[j % OS], j // OS)
                    yield wait_full(bfull[j % BS], j // BS)
                    yield ("async", "mma", oempty[j % OS], j // OS)
                    yield ("async", "mma", bempty[j % BS], j // BS)
                    j += 1
                yield ("async", "mma", accf[t % NACC], t // NACC)
                t += 1

    def epilogue():
        t = 0
        for nb, _ in items:
            for _ in range(0, nb, 1 if epilogue_per_block else SB):
                yield wait_full(accf[t % NACC], t // NACC)
                yield ("arrive", acce[t % NACC], t // NACC)
                t += 1

    gens = [producer(), mma()] + [epilogue() for _ in range(4)]
    if decoded:
        gens += [decoder() for _ in range(CONV)]
    return gens


def mixed_items(seed):
    rng = random.Random(seed)
    return [(rng.choice((1, 2, 3, 4, 5, 9)), rng.choice((1, 2, 4))) for _ in range(6)]


@pytest.mark.parametrize("decoded", [True, False], ids=["decoded weights", "bf16 weights"])
def test_shipped_protocol(decoded):
    c = constants()
    for seed in range(30):
        errors = model.run(roles(c, mixed_items(seed), decoded), seed)
        assert not errors, (decoded, seed, errors[:3])


def test_an_epilogue_out_of_step_with_the_slots_is_caught():
    # the MMA warp commits one slot per SB quant blocks; an epilogue that took one per block
    # would wait on slots that are never committed
    c = constants()
    found = [e for seed in range(10) for e in model.run(roles(c, mixed_items(seed), True, True), seed)]
    assert "deadlock" in found or any("passed at" in e for e in found), found[:3]
