"""Pins for the CPU oracle (no GPU).

The oracle is checked against things that do not come from itself: hand-worked
values (tests/golden/hand_worked.json), the e4m3fn and bf16 format definitions
(and torch's independent decoders), brute-force dense per-group products written
separately here, and the invariants of the grouped matmul:
  I0 brute force over every composition of m rows into G groups (zeros included)
  I1 rows at or past sum(group_sizes) are zero
  I2 an empty group contributes nothing
  I3 NT on W equals NN on an explicitly transposed W, bit for bit
  I4 tgmm equals the per-group lhs_g^T dout_g; summed over groups it is lhs^T dout
  I5 group_offset selects the expert slice; shards add up to the full result
  I6 integer-valued inputs give exact results
  I7 special cases: one group is a dense matmul, unit scale is no scale,
     power-of-two scales are exact, and mag is the result on |inputs|.
Definitions: page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230",
tpu_inference/kernels/megablox/gmm.py (gmm docstring, _accum, make_group_metadata,
rhs_transform_indices, _zero_uninitialized_memory) and common.py (dtype list).
"""

import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def bf16_bits(x) -> np.ndarray:
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.copy()).view(torch.bfloat16).to(torch.float64).numpy()


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits(rng.standard_normal(shape) * scale)


# ------------------------------------------------------------------ golden
def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["gmm"], ids=lambda c: c["name"])
def test_hand_worked_gmm(case):
    lhs = bf16_bits(case["lhs"])
    if "rhs_e4m3_codes" in case:
        rhs = np.asarray(case["rhs_e4m3_codes"], dtype=np.uint8)
    else:
        rhs = bf16_bits(case["rhs"])
    scale = None if "rhs_scale" not in case else np.asarray(case["rhs_scale"], np.float32)
    bias = None if "rhs_bias" not in case else bf16_bits(case["rhs_bias"])
    ref, mag = oracle.gmm(lhs, rhs, np.asarray(case["group_sizes"]), transpose_rhs=case["transpose_rhs"],
                          group_offset=case["group_offset"], rhs_scale=scale, rhs_bias=bias)
    np.testing.assert_array_equal(ref, np.asarray(case["ref"], np.float64))
    np.testing.assert_array_equal(mag, np.asarray(case["mag"], np.float64))


@pytest.mark.parametrize("case", _golden()["tgmm"], ids=lambda c: c["name"])
def test_hand_worked_tgmm(case):
    ref, mag = oracle.tgmm(bf16_bits(case["lhs"]), bf16_bits(case["dout"]), np.asarray(case["group_sizes"]))
    np.testing.assert_array_equal(ref, np.asarray(case["ref"], np.float64))
    np.testing.assert_array_equal(mag, np.asarray(case["mag"], np.float64))


# ------------------------------------------------------------------ formats
def test_e4m3fn_all_codes_match_format_definition_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(got)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}, "e4m3fn has exactly two NaN codes"
    np.testing.assert_array_equal(got[~nan], lib[~nan])
    assert np.isnan(lib[nan]).all()
    # values fixed by the format: bias 7, 3 mantissa bits, subnormals at 2^-6 * m/8
    assert got[0x38] == 1.0 and got[0x40] == 2.0 and got[0xB8] == -1.0
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9 and got[0x07] == 7 * 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert got[0x00] == 0.0 and np.signbit(got[0x80])


def test_e5m2_all_codes_match_format_definition_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode(codes, oracle.E5M2)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(got)
    assert set(np.flatnonzero(nan)) == {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF}
    np.testing.assert_array_equal(got[~nan], lib[~nan])
    assert np.isnan(lib[nan]).all()
    # bias 15, 2 mantissa bits, IEEE infinities, subnormals at 2^-14 * m/4
    assert got[0x3C] == 1.0 and got[0x40] == 2.0 and got[0xBC] == -1.0
    assert got[0x7C] == np.inf and got[0xFC] == -np.inf
    assert got[0x7B] == 57344.0 and got[0x01] == 2.0 ** -16 and got[0x04] == 2.0 ** -14


def test_int8_all_codes():
    codes = np.arange(-128, 128, dtype=np.int64).astype(np.int8)
    np.testing.assert_array_equal(oracle.decode(codes), np.arange(-128, 128, dtype=np.float64))


# e2m1 (OCP microscaling formats): sign, 2 exponent bits with bias 1, 1 mantissa bit.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_4bit_formats_values_and_nibble_order():
    # byte 0x7A holds element 0 = 0xA (low nibble) and element 1 = 0x7
    b = np.array([0x7A], np.uint8)
    np.testing.assert_array_equal(oracle.decode(b, oracle.INT4), [-6.0, 7.0])
    np.testing.assert_array_equal(oracle.decode(b, oracle.UINT4), [10.0, 7.0])
    np.testing.assert_array_equal(oracle.decode(b, oracle.E2M1), [-1.0, 6.0])
    # all 16 nibbles in both positions
    lo = np.arange(16, dtype=np.uint8)
    both = (lo | (lo[::-1] << 4)).astype(np.uint8)
    for code, table in ((oracle.INT4, [v if v < 8 else v - 16 for v in range(16)]),
                        (oracle.UINT4, list(range(16))), (oracle.E2M1, E2M1_TABLE)):
        got = oracle.decode(both, code).reshape(16, 2)
        np.testing.assert_array_equal(got[:, 0], np.asarray(table, np.float64))
        np.testing.assert_array_equal(got[:, 1], np.asarray(table, np.float64)[::-1])
    assert np.signbit(oracle.decode(np.array([0x08], np.uint8), oracle.E2M1)[0])


def unpack_nibbles(packed: np.ndarray, table) -> np.ndarray:
    """[..., k/2] bytes -> [..., k] values, low nibble first (independent of the oracle)."""
    t = np.asarray(table, np.float64)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.float64)
    out[..., 0::2] = t[packed & 0xF]
    out[..., 1::2] = t[packed >> 4]
    return out


def test_bf16_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(codes)
    lib = bf16_values(codes)
    nan = np.isnan(lib)
    assert (np.isnan(got) == nan).all()
    np.testing.assert_array_equal(got[~nan], lib[~nan])


# ------------------------------------------------------------------ brute force (I0)
def brute_force_gmm(lhs_v, w_v, sizes, transpose_rhs, group_offset=0, scale=None, bias_v=None):
    """Dense per-group products, written independently of the oracle: gather the group's
    rows into a matrix and multiply by the group's weight with numpy (fp64)."""
    m, k = lhs_v.shape
    L = w_v.shape[0]
    n = w_v.shape[1] if transpose_rhs else w_v.shape[2]
    out = np.zeros((m, n))
    start = 0
    for g, s in enumerate(sizes):
        s = max(int(s), 0)
        stop = min(start + s, m)
        if group_offset <= g < group_offset + L and stop > start:
            wg = w_v[g - group_offset]
            wg_nk = wg if transpose_rhs else wg.T  # [n, k]
            rows = lhs_v[start:stop]
            if scale is None:
                res = rows @ wg_nk.T
            else:
                nb = scale.shape[1]
                bs = k // nb
                res = np.zeros((stop - start, n))
                for b in range(nb):
                    res += (rows[:, b * bs:(b + 1) * bs] @ wg_nk[:, b * bs:(b + 1) * bs].T) * scale[g - group_offset, b, 0]
            if bias_v is not None:
                res = res + bias_v[g - group_offset, 0]
            out[start:stop] = res
        start = stop
    return out


def compositions(total, parts):
    for cuts in itertools.combinations_with_replacement(range(total + 1), parts - 1):
        edges = (0,) + cuts + (total,)
        yield [edges[i + 1] - edges[i] for i in range(parts)]


@pytest.mark.parametrize("transpose_rhs", [True, False])
def test_brute_force_every_composition(transpose_rhs):
    rng = np.random.default_rng(7)
    m, k, n, G = 6, 24, 5, 3
    lhs = rand_bf16(rng, (m, k))
    w = rand_bf16(rng, (G, n, k) if transpose_rhs else (G, k, n), 0.25)
    lhs_v, w_v = bf16_values(lhs), bf16_values(w)
    count = 0
    for total in range(m + 1):  # sums below m leave tail rows (I1)
        for sizes in compositions(total, G):
            ref, mag = oracle.gmm(lhs, w, np.array(sizes), transpose_rhs=transpose_rhs)
            np.testing.assert_allclose(ref, brute_force_gmm(lhs_v, w_v, sizes, transpose_rhs), rtol=1e-12, atol=1e-12)
            count += 1
    assert count == sum(len(list(compositions(t, G))) for t in range(m + 1))


def test_brute_force_with_torch_matmul_as_library_routine():
    rng = np.random.default_rng(8)
    m, k, n, G = 40, 64, 24, 4
    sizes = [9, 0, 20, 8]  # sum 37 < m
    lhs = rand_bf16(rng, (m, k))
    w = rand_bf16(rng, (G, n, k), 0.1)
    ref, _ = oracle.gmm(lhs, w, np.array(sizes))
    lt = torch.from_numpy(bf16_values(lhs))
    wt = torch.from_numpy(bf16_values(w))
    start = 0
    for g, s in enumerate(sizes):
        if s:
            exp = torch.matmul(lt[start:start + s], wt[g].T).numpy()
            np.testing.assert_allclose(ref[start:start + s], exp, rtol=1e-12, atol=1e-12)
        start += s
    assert (ref[start:] == 0).all()


def test_scale_and_bias_against_brute_force():
    rng = np.random.default_rng(9)
    m, k, n, G, nb = 20, 64, 12, 3, 4
    sizes = [7, 0, 11]
    lhs = rand_bf16(rng, (m, k))
    w = rand_bf16(rng, (G, n, k), 0.3)
    scale = rng.uniform(-2, 2, (G, nb, 1, n)).astype(np.float32)
    bias = rand_bf16(rng, (G, 1, n))
    ref, _ = oracle.gmm(lhs, w, np.array(sizes), rhs_scale=scale, rhs_bias=bias)
    exp = brute_force_gmm(bf16_values(lhs), bf16_values(w), sizes, True, scale=scale.astype(np.float64),
                          bias_v=bf16_values(bias))
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-12)


def test_e4m3_weights_with_scale_against_brute_force():
    rng = np.random.default_rng(10)
    m, k, n, G, nb = 16, 256, 8, 2, 2
    sizes = [5, 9]
    lhs = rand_bf16(rng, (m, k))
    codes = torch.from_numpy(np.clip(rng.standard_normal((G, n, k)) * 40, -448, 448).astype(np.float32))
    w = codes.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    w_v = torch.from_numpy(w.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scale = rng.uniform(0.5, 2, (G, nb, 1, n)).astype(np.float32) / 448
    ref, _ = oracle.gmm(lhs, w, np.array(sizes), rhs_scale=scale)
    exp = brute_force_gmm(bf16_values(lhs), w_v, sizes, True, scale=scale.astype(np.float64))
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("fmt", ["e5m2", "int8", "int4", "uint4", "e2m1"])
def test_other_weight_formats_against_brute_force(fmt):
    # NT weights [G, n, k] in each stored format, with quant-block scales and bias.
    rng = np.random.default_rng(12)
    m, k, n, G, nb = 20, 64, 8, 3, 2
    sizes = [6, 0, 11]
    lhs = rand_bf16(rng, (m, k))
    if fmt == "e5m2":
        x = torch.from_numpy(np.clip(rng.standard_normal((G, n, k)) * 300, -57344, 57344).astype(np.float32))
        w = x.to(torch.float8_e5m2).view(torch.uint8).numpy()
        w_v = torch.from_numpy(w.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
        code = oracle.E5M2
    elif fmt == "int8":
        w = rng.integers(-128, 128, (G, n, k)).astype(np.int8)
        w_v = w.astype(np.float64)
        code = oracle.INT8
    else:
        w = rng.integers(0, 256, (G, n, k // 2)).astype(np.uint8)
        table = {"int4": [v if v < 8 else v - 16 for v in range(16)], "uint4": list(range(16)),
                 "e2m1": E2M1_TABLE}[fmt]
        w_v = unpack_nibbles(w, table)
        code = {"int4": oracle.INT4, "uint4": oracle.UINT4, "e2m1": oracle.E2M1}[fmt]
    scale = rng.uniform(0.5, 2, (G, nb, 1, n)).astype(np.float32) / 64
    bias = rand_bf16(rng, (G, 1, n))
    ref, _ = oracle.gmm(lhs, w, np.array(sizes), rhs_scale=scale, rhs_bias=bias, rhs_dtype=code)
    exp = brute_force_gmm(bf16_values(lhs), w_v, sizes, True, scale=scale.astype(np.float64),
                          bias_v=bf16_values(bias))
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ invariants
def _case(seed=11, m=48, k=32, n=16, G=5, sizes=(10, 0, 13, 7, 12)):
    rng = np.random.default_rng(seed)
    return (rand_bf16(rng, (m, k)), rand_bf16(rng, (G, n, k), 0.2), np.array(sizes, np.int32), rng)


def test_I1_rows_past_sum_are_zero():
    lhs, w, sizes, _ = _case(sizes=(3, 0, 9, 1, 2))
    ref, mag = oracle.gmm(lhs, w, sizes)
    assert (ref[15:] == 0).all() and (mag[15:] == 0).all()
    assert (np.abs(ref[:15]).sum(axis=1) > 0).all()


def test_I2_inserting_an_empty_group_changes_nothing():
    lhs, w, sizes, rng = _case()
    ref, _ = oracle.gmm(lhs, w, sizes)
    for pos in range(len(sizes) + 1):
        junk = rand_bf16(rng, (1,) + w.shape[1:], 5.0)
        ref2, _ = oracle.gmm(lhs, np.concatenate([w[:pos], junk, w[pos:]]), np.insert(sizes, pos, 0))
        np.testing.assert_array_equal(ref, ref2)


def test_I3_nt_equals_nn_on_transposed_weight_bitwise():
    lhs, w, sizes, _ = _case()
    a, am = oracle.gmm(lhs, w, sizes, transpose_rhs=True)
    b, bm = oracle.gmm(lhs, np.ascontiguousarray(np.swapaxes(w, 1, 2)), sizes, transpose_rhs=False)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(am, bm)


def test_I4_tgmm_is_per_group_product_and_sums_to_dense():
    rng = np.random.default_rng(12)
    m, k, n = 30, 12, 10
    sizes = np.array([4, 0, 17, 9], np.int32)  # sum == m
    lhs, dout = rand_bf16(rng, (m, k)), rand_bf16(rng, (m, n))
    ref, _ = oracle.tgmm(lhs, dout, sizes)
    lv, dv = bf16_values(lhs), bf16_values(dout)
    start = 0
    for g, s in enumerate(sizes):
        np.testing.assert_allclose(ref[g], lv[start:start + s].T @ dv[start:start + s], rtol=1e-12, atol=1e-12)
        start += s
    assert (ref[1] == 0).all()
    np.testing.assert_allclose(ref.sum(axis=0), lv.T @ dv, rtol=1e-12, atol=1e-12)


def test_I5_group_offset_selects_slice_and_shards_sum_to_full():
    lhs, w, sizes, _ = _case()
    full, _ = oracle.gmm(lhs, w, sizes)
    offs = oracle.group_offsets(sizes, lhs.shape[0])
    acc = np.zeros_like(full)
    for go, L in [(0, 2), (2, 1), (3, 2)]:
        part, _ = oracle.gmm(lhs, w[go:go + L], sizes, group_offset=go)
        lo, hi = offs[go], offs[go + L]
        np.testing.assert_array_equal(part[lo:hi], full[lo:hi])
        assert (part[:lo] == 0).all() and (part[hi:] == 0).all()
        acc += part
    np.testing.assert_array_equal(acc, full)


def test_I6_integer_inputs_exact_and_each_row_uses_its_expert():
    rng = np.random.default_rng(13)
    m, k, n, G = 37, 256, 9, 4
    sizes = np.array([11, 0, 20, 6], np.int32)
    lhs_i = rng.integers(-8, 9, (m, k))
    base = rng.integers(-8, 9, (n, k))
    w_i = np.stack([(g + 1) * base for g in range(G)])
    ref, _ = oracle.gmm(bf16_bits(lhs_i), bf16_bits(w_i), sizes)
    start = 0
    for g, s in enumerate(sizes):
        for r in range(start, start + s):
            exact = [int(np.dot(lhs_i[r].astype(object), w_i[g, c].astype(object))) for c in range(n)]
            assert ref[r].tolist() == [float(v) for v in exact]
        start += s
    assert (ref[start:] == 0).all()


def test_I7_one_group_is_dense_and_unit_scale_is_no_scale():
    rng = np.random.default_rng(14)
    m, k, n = 19, 64, 7
    lhs, w = rand_bf16(rng, (m, k)), rand_bf16(rng, (1, n, k))
    ref, _ = oracle.gmm(lhs, w, np.array([m]))
    np.testing.assert_allclose(ref, bf16_values(lhs) @ bf16_values(w)[0].T, rtol=1e-12, atol=1e-12)
    ones = np.ones((1, 4, 1, n), np.float32)
    ref1, _ = oracle.gmm(lhs, w, np.array([m]), rhs_scale=ones)
    np.testing.assert_allclose(ref1, ref, rtol=1e-14, atol=1e-14)
    pow2 = np.full((1, 4, 1, n), 0.25, np.float32)
    ref4, _ = oracle.gmm(lhs, w, np.array([m]), rhs_scale=pow2)
    np.testing.assert_array_equal(ref4, ref1 * 0.25)


def test_I7_mag_is_result_on_absolute_inputs():
    rng = np.random.default_rng(15)
    m, k, n, G, nb = 25, 64, 11, 3, 2
    sizes = np.array([8, 9, 8], np.int32)
    lhs, w = rand_bf16(rng, (m, k)), rand_bf16(rng, (G, n, k))
    scale = rng.uniform(-1, 1, (G, nb, 1, n)).astype(np.float32)
    bias = rand_bf16(rng, (G, 1, n))
    _, mag = oracle.gmm(lhs, w, sizes, rhs_scale=scale, rhs_bias=bias)
    absb = lambda b: bf16_bits(np.abs(bf16_values(b)))
    ref_abs, _ = oracle.gmm(absb(lhs), absb(w), sizes, rhs_scale=np.abs(scale), rhs_bias=absb(bias))
    np.testing.assert_allclose(mag, ref_abs, rtol=1e-12, atol=0)


def test_sampled_rows_and_k_rows_match_full_runs():
    lhs, w, sizes, rng = _case()
    full, fmag = oracle.gmm(lhs, w, sizes)
    rows = np.array([0, 5, 9, 10, 22, 23, 40, 47])
    part, pmag = oracle.gmm(lhs, w, sizes, rows=rows)
    np.testing.assert_array_equal(part, full[rows])
    np.testing.assert_array_equal(pmag, fmag[rows])
    dout = rand_bf16(rng, (lhs.shape[0], 6))
    t_full, _ = oracle.tgmm(lhs, dout, sizes)
    kr = np.array([1, 7, 31])
    t_part, _ = oracle.tgmm(lhs, dout, sizes, k_rows=kr)
    np.testing.assert_array_equal(t_part, t_full[:, kr])


def test_negative_sizes_count_as_zero_and_offsets_cap_at_m():
    offs = oracle.group_offsets(np.array([3, -2, 5, 100], np.int32), 10)
    assert offs.tolist() == [0, 3, 3, 8, 10]
    lhs, w, _, _ = _case(G=4, sizes=(0, 0, 0, 0))
    ref_neg, _ = oracle.gmm(lhs, w, np.array([5, -7, 30, 40], np.int32))
    ref_pos, _ = oracle.gmm(lhs, w, np.array([5, 0, 30, 13], np.int32))
    np.testing.assert_array_equal(ref_neg, ref_pos)


def test_rejects_bad_arguments():
    lhs, w, sizes, _ = _case()
    with pytest.raises(ValueError):
        oracle.gmm(lhs, w, sizes, group_offset=3)  # 3 + 5 local groups > 5 total
    with pytest.raises(ValueError):
        oracle.gmm(lhs, w, sizes, rhs_scale=np.ones((5, 3, 1, 16), np.float32))  # k=32 not divisible by 3


# ------------------------------------------------------------------ W8A8 pieces
def test_e8m0_scale_codes():
    codes = np.array([0, 1, 126, 127, 128, 200, 254, 255], np.uint8)
    got = oracle.decode(codes, oracle.E8M0)
    expect = [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 73, 2.0 ** 127, 0.0]
    np.testing.assert_array_equal(got, expect)


def test_lhs_scale_and_e8m0_rhs_scale_against_brute_force():
    rng = np.random.default_rng(13)
    m, k, n, G, nb, nlb = 12, 256, 8, 2, 2, 2
    sizes = [5, 7]
    codes = rng.integers(0, 256, (m, k)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
    lhs_v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    a_scale = rng.uniform(0.001, 0.01, (m, nlb)).astype(np.float32)
    w = rand_bf16(rng, (G, n, k), 0.5)
    e8 = rng.integers(120, 135, (G, nb, 1, n)).astype(np.uint8)
    e8[0, 0, 0, 3] = 255  # decodes to 0
    s_v = np.where(e8 == 255, 0.0, 2.0 ** (e8.astype(np.float64) - 127))
    ref, _ = oracle.gmm(codes, w, np.array(sizes), rhs_scale=e8, lhs_scale=a_scale, lhs_dtype=oracle.E4M3)
    scaled_lhs = lhs_v * np.repeat(a_scale.astype(np.float64), k // nlb, axis=1)
    exp = brute_force_gmm(scaled_lhs, bf16_values(w), sizes, True, scale=s_v)
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-12)


def _bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.uint16).numpy()


def test_quantize_ties_to_even_and_saturation():
    # amax 448 makes the scale exactly 1, so x / scale = x: 1.0625 lies between 1 and 1.125 (even: 1.0),
    # 1.1875 between 1.125 and 1.25 (even: 1.25), 248 between 240 and 256 (even: 256)
    x = _bf16_bits([[448.0, 1.0625, 1.1875, -1.0625, 248.0, 0.0, -448.0, 3.0]])
    q, s = oracle.quantize_e4m3(x, group=8)
    assert s.tolist() == [[1.0]]
    assert q.tolist() == [[0x7E, 0x38, 0x3A, 0xB8, 0x78, 0x00, 0xFE, 0x44]]


def test_quantize_matches_torch_rounding_and_error_bound():
    rng = np.random.default_rng(14)
    m, k = 16, 512
    x = (rng.standard_normal((m, k)) * np.exp2(rng.integers(-6, 7, (m, 1)))).astype(np.float32)
    x[3, 128:256] = 0.0                                  # an all-zero group
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.uint16).numpy()
    q, s = oracle.quantize_e4m3(bits, group=128)
    xv = bf16_values(bits)
    assert s[3, 1] == 1.0 and (q[3, 128:256] == 0).all()
    # the scale is amax / 448 in fp32; the largest element of each group maps to +-448
    amax = np.abs(xv).reshape(m, 4, 128).max(axis=2).astype(np.float32)
    np.testing.assert_array_equal(s[amax > 0], (amax / np.float32(448.0))[amax > 0])
    y = (xv.astype(np.float32) / np.repeat(s, 128, axis=1)).astype(np.float32)
    ok = np.abs(y) <= 448.0
    lib = torch.from_numpy(y[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q[ok], lib)
    qv = oracle.decode(q).astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1)
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, np.repeat(s.astype(np.float64), 128, axis=1) * 2.0 ** -10)
    assert (np.abs(qv - xv) <= bound * (1 + 1e-9)).all()


def test_quantize_nan_group():
    x = _bf16_bits([[1.0, float("nan"), 2.0, 3.0, 1.0, 2.0, 3.0, 4.0]])
    q, s = oracle.quantize_e4m3(x, group=4)
    assert np.isnan(s[0, 0]) and s[0, 1] == np.float32(4.0) / np.float32(448.0)
    assert (q[0, :4] & 0x7F == 0x7F).all()


# ------------------------------------------------------------------ microscaling block scales
def test_mxfp8_block_scales_against_brute_force():
    # e4m3 weights with one E8M0 scale per 32 consecutive k of each weight row (MXFP8)
    rng = np.random.default_rng(21)
    m, k, n, G = 14, 128, 6, 2
    sizes = [6, 8]
    lhs = rand_bf16(rng, (m, k))
    codes = rng.integers(0, 256, (G, n, k)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x40
    e8 = rng.integers(118, 136, (G, n, k // 32)).astype(np.uint8)
    e8[0, 1, 2] = 255   # a zero block
    e8[1, 4, 0] = 0     # 2^-127
    w_v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s_v = np.where(e8 == 255, 0.0, 2.0 ** (e8.astype(np.float64) - 127))
    ref, _ = oracle.gmm(lhs, codes, np.array(sizes), rhs_dtype=oracle.E4M3, rhs_block_scale=e8)
    exp = brute_force_gmm(bf16_values(lhs), w_v * np.repeat(s_v, 32, axis=2), sizes, True)
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-300)


def test_nvfp4_block_scales_with_tensor_scale_against_brute_force():
    # e2m1 weights (packed, low nibble first) with one e4m3 scale per 16 k and an fp32 scale per
    # expert and column (NVFP4's second level, here the per-block rhs_scale with one block)
    rng = np.random.default_rng(22)
    m, k, n, G = 10, 64, 5, 2
    sizes = [4, 6]
    lhs = rand_bf16(rng, (m, k))
    packed = rng.integers(0, 256, (G, n, k // 2)).astype(np.uint8)
    s8 = rng.integers(0x20, 0x60, (G, n, k // 16)).astype(np.uint8)  # positive finite e4m3 codes
    tensor_scale = rng.uniform(0.5, 2.0, (G, 1, 1, n)).astype(np.float32)
    w_v = unpack_nibbles(packed, E2M1_TABLE)
    s_v = torch.from_numpy(s8.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref, _ = oracle.gmm(lhs, packed, np.array(sizes), rhs_dtype=oracle.E2M1, rhs_block_scale=s8,
                        rhs_block_scale_dtype=oracle.E4M3, rhs_scale=tensor_scale)
    exp = brute_force_gmm(bf16_values(lhs), w_v * np.repeat(s_v, 16, axis=2), sizes, True,
                          scale=tensor_scale.astype(np.float64))
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-300)


def test_one_block_per_row_equals_the_per_column_scale():
    # a block scale whose block is the whole row is the per-(expert, column) scale with one quant block
    rng = np.random.default_rng(23)
    m, k, n, G = 9, 64, 7, 3
    sizes = [2, 4, 3]
    lhs = rand_bf16(rng, (m, k))
    w = rand_bf16(rng, (G, n, k))
    s = rng.uniform(0.25, 4.0, (G, n, 1)).astype(np.float32)
    a, _ = oracle.gmm(lhs, w, np.array(sizes), rhs_block_scale=s)
    b, _ = oracle.gmm(lhs, w, np.array(sizes), rhs_scale=s.reshape(G, n).reshape(G, 1, 1, n))
    np.testing.assert_allclose(a, b, rtol=1e-14, atol=0)
