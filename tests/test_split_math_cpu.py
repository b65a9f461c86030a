"""The exactness of the two-term e4m3 split that the fp8 kernels apply to bf16 activations, as
stated in gemm_fp8.cuh and the ABI header, checked on the host statement of the split
(tests/split_statement.py, which the GPU tests compare with the kernels bit for bit).  For a
k step whose largest magnitude is M, with E = floor(log2 M), every bf16 x of the step equals
2^(E-7) (h + l/16) exactly when |x| >= 2^(E-13), and is within 2^(E-21) <= M 2^-21 of it
otherwise (E clamped at -119 for steps below 2^-119)."""

import numpy as np
import pytest

import oracle
from split_statement import e4m3_rne, split_statement


@pytest.fixture(scope="module", autouse=True)
def library():
    oracle.build()


def _reconstruct(bits, step):
    planes, scales = split_statement(bits, step)
    h = oracle.decode(planes[0])
    l = oracle.decode(planes[1])
    s = np.repeat(scales, step, axis=1)[:, :bits.shape[1]].astype(np.float64)
    return s * (h + l / 16)


def _values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("top", [0x3F80, 0x3FFF, 0x4780, 0x0080])  # M = 1, 1.99.., 65536, 2^-126
def test_every_smaller_bf16_magnitude_in_a_step(top):
    # every positive bf16 code up to M, both signs, each step holding M itself: exact from
    # 2^(E-13) up, within M 2^-21 below
    codes = np.arange(1, top + 1, dtype=np.uint16)
    codes = np.concatenate([codes, codes | 0x8000])
    per_row = 255
    rows = -(-codes.size // per_row)
    bits = np.zeros((rows, 256), np.uint16)
    bits[:, 0] = top
    flat = np.zeros(rows * per_row, np.uint16)
    flat[:codes.size] = codes
    bits[:, 1:] = flat.reshape(rows, per_row)
    x = _values(bits)
    rec = _reconstruct(bits, 256)
    M = float(_values(np.array([top], np.uint16))[0])
    # E, clamped at -119: a step whose largest magnitude is below 2^-119 is scaled by 2^-126
    E = max(np.floor(np.log2(M)), -119.0)
    exact = np.abs(x) >= 2.0 ** (E - 13)
    assert np.array_equal(rec[exact], x[exact])
    assert np.all(np.abs(rec - x)[~exact] <= 2.0 ** (E - 21))
    # the bound is reached: the statement is not stronger than it needs to be
    # (bf16 subnormals below a clamped step have too few bits to be rounded)
    if M >= 2.0 ** -119 and (~exact).any():
        assert np.abs(rec - x)[~exact].max() > 2.0 ** (E - 22)


def test_range_2_14_is_not_enough():
    # x between M 2^-14 and 2^(E-13) can be rounded: x / 2^(E-7) is an e4m3 subnormal there
    M = 2.71875                       # E = 1
    x = -0.00018596649169921875       # |x| / M = 2^-13.84, below 2^(E-13) = 2^-12
    bits = np.zeros((1, 256), np.uint16)
    bits[0, :2] = (np.array([M, x], np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert abs(x) >= M * 2.0 ** -14
    rec = _reconstruct(bits, 256)
    assert rec[0, 1] != x and abs(rec[0, 1] - x) <= M * 2.0 ** -21


def test_ties_round_to_the_even_code():
    y = np.array([1.0625, 1.1875, -1.0625, 0.0029296875, 448.0, 500.0], np.float32)
    # 1.0625: 1.0 (0x38) vs 1.125 (0x39); 1.1875: 1.125 vs 1.25 (0x3A); 0.0029296875 = 1.5 x 2^-9:
    # subnormals 1 x 2^-9 (0x01) vs 2 x 2^-9 (0x02); 500 saturates to 448 (0x7E)
    assert e4m3_rne(y).tolist() == [0x38, 0x3A, 0xB8, 0x02, 0x7E, 0x7E]


def test_zero_and_negative_zero_steps():
    bits = np.zeros((2, 384), np.uint16)
    bits[1] = 0x8000
    planes, scales = split_statement(bits, 256)
    assert (planes[:, 0] == 0).all()
    assert (planes[0, 1] == 0x80).all() and (planes[1, 1] == 0).all()  # h = -0, l = +0 (-0 - -0)
    assert (scales == np.float32(2.0 ** -126)).all()                   # e clamped to 8
