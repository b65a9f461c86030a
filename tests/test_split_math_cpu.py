"""The two-level e4m3 split that the fp8 kernels apply to bf16 activations, as stated in
gemm_fp8.cuh and the ABI header, checked on the host statement of the split
(tests/split_statement.py, which the GPU tests compare with the kernels bit for bit).

For a k step whose largest magnitude is M, with E = floor(log2 M), the first level alone equals
every bf16 x of the step exactly when |x| >= 2^(E-13) and is within 2^(E-21) <= M 2^-21 of it
otherwise (E clamped at -119 for steps below 2^-119).  The second level splits what the first
leaves; a step is marked for the kernel's exact path exactly when the two levels together do not
give back every value of the step, or when it holds an infinity or a NaN."""

import numpy as np
import pytest

import oracle
from split_statement import e4m3_rne, reconstruct, split_statement


@pytest.fixture(scope="module", autouse=True)
def library():
    oracle.build()


def _level1(bits, step):
    planes, scales = split_statement(bits, step)
    h = oracle.decode(planes[0])
    l = oracle.decode(planes[1])
    s = np.repeat(scales[:, :, 0], step, axis=1)[:, :bits.shape[1]].astype(np.float64)
    return s * (h + l / 16)


def _values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bits_of(values):
    v = np.asarray(values, np.float32)
    b = (v.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_values(b), v.astype(np.float64)), "values must be bf16 values"
    return b


def _rows_with_every_code_below(top):
    # every positive bf16 code up to M, both signs, each 256-wide row holding M itself first
    codes = np.arange(1, top + 1, dtype=np.uint16)
    codes = np.concatenate([codes, codes | 0x8000])
    per_row = 255
    rows = -(-codes.size // per_row)
    bits = np.zeros((rows, 256), np.uint16)
    bits[:, 0] = top
    flat = np.zeros(rows * per_row, np.uint16)
    flat[:codes.size] = codes
    bits[:, 1:] = flat.reshape(rows, per_row)
    return bits


@pytest.mark.parametrize("top", [0x3F80, 0x3FFF, 0x4780, 0x0080])  # M = 1, 1.99.., 65536, 2^-126
def test_first_level_range_for_every_smaller_bf16_magnitude(top):
    # exact from 2^(E-13) up, within M 2^-21 below
    bits = _rows_with_every_code_below(top)
    x = _values(bits)
    rec = _level1(bits, 256)
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


@pytest.mark.parametrize("top", [0x3F80, 0x3FFF, 0x4780, 0x0080])
def test_two_levels_or_a_mark_for_every_smaller_bf16_magnitude(top):
    # every step is either given back exactly by the two levels or marked, never both
    bits = _rows_with_every_code_below(top)
    planes, scales = split_statement(bits, 256)
    rec, marked = reconstruct(planes, scales, 256)
    x = _values(bits)
    exact_rows = (rec == x).all(axis=1)
    assert np.array_equal(~exact_rows, marked[:, 0])
    # the unmarked steps include every step whose values lie within 2^26 of M
    M = float(_values(np.array([top], np.uint16))[0])
    E = max(np.floor(np.log2(M)), -119.0)
    close = (np.abs(x) >= 2.0 ** (E - 26)) | (x == 0)
    assert not marked[close.all(axis=1), 0].any()


def test_range_2_14_is_not_enough_for_one_level():
    # x between M 2^-14 and 2^(E-13) can be rounded by the first level: x / 2^(E-7) is an e4m3
    # subnormal there; the second level gives it back
    M = 2.71875                       # E = 1
    x = -0.00018596649169921875       # |x| / M = 2^-13.84, below 2^(E-13) = 2^-12
    bits = np.zeros((1, 256), np.uint16)
    bits[0, :2] = _bits_of([M, x])
    assert abs(x) >= M * 2.0 ** -14
    rec1 = _level1(bits, 256)
    assert rec1[0, 1] != x and abs(rec1[0, 1] - x) <= M * 2.0 ** -21
    planes, scales = split_statement(bits, 256)
    rec, marked = reconstruct(planes, scales, 256)
    assert rec[0, 1] == x and not marked.any() and scales[0, 0, 1] > 0


def test_one_large_value_beside_small_ones():
    # 1.0 and 3 * 2^-22: the first level rounds each small value to 2^-20 (+33 %); the second
    # holds the rest, -2^-22, exactly
    bits = np.zeros((2, 256), np.uint16)
    bits[0] = _bits_of([1.0] + [3 * 2.0 ** -22] * 255)
    bits[1] = _bits_of([1.0] + [3 * 2.0 ** -133, -5 * 2.0 ** -133] * 127 + [0.0])  # bf16 subnormals
    x = _values(bits)
    assert _level1(bits, 256)[0, 1] == 2.0 ** -20
    planes, scales = split_statement(bits, 256)
    rec, marked = reconstruct(planes, scales, 256)
    assert np.array_equal(rec, x) and not marked.any()
    assert scales[0, 0, 1] == np.float32(2.0 ** -29)  # the rest's largest magnitude is 2^-22


def test_three_ranges_are_marked():
    # 1.0, values near 2^-30 and values near 2^-60: the second level's range ends 2^13 below its
    # own largest value, so the smallest ones are left over and the step is marked
    v = [1.0] + [1.5 * 2.0 ** -30, 1.25 * 2.0 ** -60] * 127 + [0.0]
    bits = _bits_of(v)[None]
    planes, scales = split_statement(bits, 256)
    rec, marked = reconstruct(planes, scales, 256)
    assert marked[0, 0] and not np.array_equal(rec, _values(bits))
    assert np.signbit(scales[0, 0, 1]) and np.isfinite(scales[0, 0, 0])


def test_random_rows_marked_exactly_when_not_given_back():
    # random magnitudes over 2^-130 .. 2^30 and both signs, 128- and 256-wide steps
    g = np.random.Generator(np.random.PCG64(11))
    for step in (256, 128):
        x = g.standard_normal((64, 1024)) * 2.0 ** g.integers(-130, 31, (64, 1024))
        x[::3] = g.standard_normal((22, 1024))  # plain rows: almost never marked
        bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        planes, scales = split_statement(bits, step)
        rec, marked = reconstruct(planes, scales, step)
        xv = _values(bits)
        steps_exact = (rec == xv).reshape(64, -1, step).all(axis=2)
        assert np.array_equal(~steps_exact, marked)
        assert not marked[::3].any()


def test_non_finite_steps_are_marked():
    bits = np.zeros((3, 512), np.uint16)
    bits[:, :] = _bits_of(np.ones(512))
    bits[0, 5] = 0x7F80   # +inf
    bits[1, 300] = 0xFF80  # -inf
    bits[2, 7] = 0x7FC0   # NaN
    _, scales = split_statement(bits, 256)
    marked = np.signbit(scales[:, :, 1])
    assert marked.tolist() == [[True, False], [False, True], [True, False]]
    assert np.isnan(scales[0, 0, 0]) and np.isnan(scales[1, 1, 0]) and np.isfinite(scales[0, 1, 0])


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
    assert (planes[2:, 1] == 0).all()                                   # no second level
    assert (scales[:, :, 0] == np.float32(2.0 ** -126)).all()          # e clamped to 8
    assert (scales[:, :, 1] == 0).all() and not np.signbit(scales[:, :, 1]).any()


# ------------------------------------------------------------------ the fp16 split (integer weights)
def _rows_of_128(bits256):
    # the 256-wide rows above cut into two 128-wide rows, each led by its step's maximum
    b = bits256.reshape(-1, 128).copy()
    b[1::2, 0] = bits256[:, 0]
    return b


@pytest.mark.parametrize("top", [0x3F80, 0x3FFF, 0x4780, 0x0080, 0x0001])  # M = 1, 1.99.., 65536, 2^-126, 2^-133
def test_fp16_split_range_for_every_smaller_bf16_magnitude(top):
    # with E = floor(log2 M) (at least -112 through the clamp) x is held exactly when
    # |x| >= 2^(E-28) (an fp16 normal), and below that exactly when x is a multiple of fp16's
    # subnormal spacing 2^(E-38); a step holding any other x is marked, and only then
    from split_statement import split_statement_f16
    bits = _rows_of_128(_rows_with_every_code_below(top))
    plane, scales = split_statement_f16(bits, perm=False)
    x = _values(bits)
    back = plane.view(np.float16).astype(np.float64) * scales[:, 0:1, 0].astype(np.float64)
    E = max(int(np.floor(np.log2(_values(np.array([top], np.uint16))[0]))), -112)
    spacing = 2.0 ** (E - 38)
    held = (np.abs(x) >= 2.0 ** (E - 28)) | (np.mod(x, spacing) == 0)
    assert np.array_equal(back == x, held)
    assert np.array_equal(np.signbit(scales[:, 0, 1]), ~held.all(axis=1))


def test_fp16_split_marks_nonfinite_steps_and_orders_four_bit_rows():
    from split_statement import F16_ORDER, split_statement_f16
    rng = np.random.default_rng(5)
    bits = (rng.standard_normal((6, 256)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits[2, 7] = 0x7F80   # +inf
    bits[3, 200] = 0x7FC0  # NaN
    plane, scales = split_statement_f16(bits, perm=False)
    permuted, scales_p = split_statement_f16(bits, perm=True)
    marks = np.signbit(scales[:, :, 1])
    assert marks[2, 0] and not marks[2, 1] and marks[3, 1] and not marks[3, 0]
    assert not marks[[0, 1, 4, 5]].any(), "N(0, 1) steps are held whole"
    assert np.array_equal(scales.view(np.uint32), scales_p.view(np.uint32))
    assert np.array_equal(permuted.reshape(6, 32, 8), plane.reshape(6, 32, 8)[:, :, F16_ORDER])
    # unmarked steps give every value back
    back = plane.view(np.float16).astype(np.float64) * np.repeat(scales[:, :, 0], 128, axis=1)
    ok = ~np.repeat(marks, 128, axis=1)
    assert np.array_equal(back[ok], _values(bits)[ok])
