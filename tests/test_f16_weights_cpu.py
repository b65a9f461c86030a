"""The fp16-weight kernel's code-to-fp16 arithmetic (gemm_f16w.cu), restated with numpy's
float16 and checked, for every code, against the oracle's format decoders:

- int8: the code with its sign bit flipped, under a 0x64 byte, is the fp16 number 1024 + 128 + v;
  one fp16 subtraction of 1152 gives v.
- int4 / uint4: a code in the low nibble of a half under 0x6400 is 1024 + c (signed codes biased
  by 8 first), less 1032 or 1024; in the second nibble it is 1024 + 16 c, and one fused
  multiply-add by 1/16 and -72 or -64 gives the value.  Eight codes of a word come out in the
  order (0, 4), (1, 5), (2, 6), (3, 7).
- NVFP4: an e2m1 code's sign and magnitude bits at fp16 bits 15 and 11..9 are 2^-14 times its
  value; times 2^14 and then times its block's e4m3 scale, both fp16 multiplications are exact
  for every code and every finite scale (the products have at most 6 significant bits, lie
  within 6 * 448 and on fp16's grid).
- MXFP8: every e4m3fn code is an fp16 value (the two NaN codes are NaN), and the kernel's fold of
  one 16-column accumulator per 32-k block, each scaled by its E8M0 byte of the step's 4-byte
  word (byte q for block q), reproduces the definition: a host statement of that fold against
  the oracle.
"""

import numpy as np
import pytest

import oracle


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16)


def f16_bits(x):
    return np.asarray(x, np.float16).view(np.uint16)


def fma16(a, b, c):
    """One fused multiply-add rounded once to fp16 (the products and sums here are exact in
    float64)."""
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(np.float16)


def test_int8_codes_to_fp16():
    codes = np.arange(256, dtype=np.uint32)
    half = f16(0x6400 | (codes ^ 0x80))
    got = (half - np.float16(1152)).astype(np.float64)
    want = oracle.decode(codes.astype(np.uint8).view(np.int8).reshape(1, -1), oracle.INT8).ravel()
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("signed", [True, False], ids=["int4", "uint4"])
def test_four_bit_codes_to_fp16_in_both_nibbles(signed):
    c = np.arange(16, dtype=np.uint32)
    u = c ^ 8 if signed else c
    low = (f16(0x6400 | u) - np.float16(1032 if signed else 1024)).astype(np.float64)
    high = fma16(f16(0x6400 | (u << 4)), np.float16(1.0 / 16), np.float16(-72 if signed else -64)).astype(np.float64)
    # the oracle's decoder: two codes per byte, the even k in the low nibble
    packed = (c | (c << 4)).astype(np.uint8).reshape(1, -1)
    want = oracle.decode(packed, oracle.INT4 if signed else oracle.UINT4).reshape(16, 2)
    np.testing.assert_array_equal(low, want[:, 0])
    np.testing.assert_array_equal(high, want[:, 1])


def _nib8(w, signed):
    """The kernel's nib8_to_f16 on one 32-bit word: four fp16 pairs (lo, hi)."""
    u = w ^ 0x88888888 if signed else w
    sub, add = (1032, -72) if signed else (1024, -64)
    u8 = u >> 8
    out = []
    for v, second in ((u, False), (u, True), (u8, False), (u8, True)):
        mask = 0x00F000F0 if second else 0x000F000F
        halves = (v & mask) | 0x64006400
        lo, hi = f16(halves & 0xFFFF), f16(halves >> 16)
        if second:
            out.append((fma16(lo, np.float16(1.0 / 16), np.float16(add)), fma16(hi, np.float16(1.0 / 16), np.float16(add))))
        else:
            out.append((lo - np.float16(sub), hi - np.float16(sub)))
    return [(float(a), float(b)) for a, b in out]


@pytest.mark.parametrize("signed", [True, False], ids=["int4", "uint4"])
def test_four_bit_word_order(signed):
    rng = np.random.Generator(np.random.PCG64(5))
    for _ in range(64):
        nib = rng.integers(0, 16, size=8)
        w = int(sum(int(n) << (4 * i) for i, n in enumerate(nib)))
        packed = np.array([[nib[0] | nib[1] << 4, nib[2] | nib[3] << 4, nib[4] | nib[5] << 4, nib[6] | nib[7] << 4]],
                          np.uint8)
        vals = oracle.decode(packed, oracle.INT4 if signed else oracle.UINT4).ravel()  # k order
        assert _nib8(w, signed) == [(vals[i], vals[i + 4]) for i in range(4)]


def _e2m1_half(c):
    return f16(((c & 7) << 9) | ((c & 8) << 12))


def test_e2m1_codes_to_fp16():
    c = np.arange(16, dtype=np.uint32)
    got = (_e2m1_half(c) * np.float16(2.0 ** 14)).astype(np.float64)
    packed = (c | (c << 4)).astype(np.uint8).reshape(1, -1)
    want = oracle.decode(packed, oracle.E2M1).reshape(16, 2)[:, 0]
    np.testing.assert_array_equal(got, want)


def test_e2m1_word_order():
    # the kernel's e2m1x8_to_f16: word i of the output holds codes i and i + 4
    rng = np.random.Generator(np.random.PCG64(6))
    for _ in range(64):
        nib = rng.integers(0, 16, size=8)
        w = int(sum(int(n) << (4 * i) for i, n in enumerate(nib)))
        for i in range(4):
            v = w >> (4 * i)
            bits = ((v & 0x00070007) << 9) | ((v & 0x00080008) << 12)
            assert (bits & 0xFFFF) == int(f16_bits(_e2m1_half(np.uint32(nib[i]))))
            assert (bits >> 16) == int(f16_bits(_e2m1_half(np.uint32(nib[i + 4]))))


def test_nvfp4_code_times_scale_is_exact_in_fp16():
    codes = np.arange(16, dtype=np.uint32)
    packed = (codes | (codes << 4)).astype(np.uint8).reshape(1, -1)
    w = oracle.decode(packed, oracle.E2M1).reshape(16, 2)[:, 0]
    scales_all = oracle.decode(np.arange(256, dtype=np.uint8).reshape(1, -1), oracle.E4M3).ravel()
    finite = np.isfinite(scales_all)
    scales = scales_all[finite]
    # every e4m3 value is an fp16 value (cvt.rn.f16x2.e4m3x2 is exact)
    np.testing.assert_array_equal(scales.astype(np.float16).astype(np.float64), scales)
    # the kernel's order: the code's half times 2^14, then times the scale
    step1 = (_e2m1_half(codes) * np.float16(2.0 ** 14))
    got = (step1[:, None] * scales.astype(np.float16)[None, :]).astype(np.float64)
    want = w[:, None] * scales[None, :]
    np.testing.assert_array_equal(got, want)
    assert np.abs(want).max() <= 6 * 448


def test_e4m3_codes_to_fp16_exact():
    codes = np.arange(256, dtype=np.uint8).reshape(1, -1)
    v = oracle.decode(codes, oracle.E4M3).ravel()
    nan = np.isnan(v)
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]
    np.testing.assert_array_equal(v[~nan].astype(np.float16).astype(np.float64), v[~nan])


def _e8m0(b):
    return 0.0 if b == 255 else 2.0 ** (int(b) - 127)


def test_mxfp8_block_fold_matches_oracle():
    """The kernel's arithmetic for one (row, weight row), restated: per 128-wide step the row is
    stored as fp16 x / sc (sc = 2^(E - 141), E the exponent field of the step's largest |x|, at
    least 15); each 32-k block q sums the exact products (x / sc) w into fp32 (D_q); the epilogue
    reads the step's E8M0 word e4 and adds u_q * (sc * D_q), u_q = s_w * 2^(e_q - 127) with e_q
    = byte q of e4, the two halves of the word in order."""
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(11))
    m, k, n = 3, 256, 5
    x = torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).to(torch.bfloat16)
    x[1] = x[1] * 2.0 ** 20
    xb = x.view(torch.uint16).numpy()
    xv = x.float().numpy().astype(np.float64)
    codes = rng.integers(0, 256, size=(1, n, k), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN weights
    w = oracle.decode(codes.reshape(n, k), oracle.E4M3).reshape(n, k)
    e = rng.integers(118, 137, size=(1, n, k // 32), dtype=np.uint8)
    e[0, 1, 0], e[0, 2, 5] = 255, 0
    ref, mag = oracle.gmm(xb, codes, np.array([m], np.int32), rhs_dtype=oracle.E4M3, rhs_block_scale=e,
                          rhs_block_scale_dtype=oracle.E8M0)
    got = np.zeros((m, n))
    for r in range(m):
        for c in range(n):
            acc = np.float32(0.0)
            for ks in range(k // 128):
                seg = slice(128 * ks, 128 * ks + 128)
                big = int(np.abs(xb[r, seg].astype(np.int64) & 0x7FFF).max()) >> 7
                sc = 2.0 ** (max(big, 15) - 141)
                h = (xv[r, seg] / sc).astype(np.float16).astype(np.float64)
                assert np.array_equal(h * sc, xv[r, seg])  # the split holds these rows exactly
                d = [np.float32(np.sum(h[32 * q:32 * q + 32] * w[c, 128 * ks + 32 * q:128 * ks + 32 * q + 32]))
                     for q in range(4)]
                e4 = int.from_bytes(bytes(e[0, c, 4 * ks:4 * ks + 4]), "little")
                for half in range(2):
                    u0 = np.float32(_e8m0((e4 >> (16 * half)) & 255))
                    u1 = np.float32(_e8m0((e4 >> (16 * half + 8)) & 255))
                    s = np.float32(sc)
                    acc = np.float32(acc + u0 * (s * d[2 * half]))
                    acc = np.float32(acc + u1 * (s * d[2 * half + 1]))
            got[r, c] = acc
    bound = 4 * 2.0 ** -24 * (k // 32 + 8) * mag
    assert np.all(np.abs(got - ref) <= bound + 1e-300), np.max(np.abs(got - ref) / np.maximum(mag, 1e-300))
    # a wrong byte-to-block mapping (the halves swapped) does not pass
    swapped = e.copy()
    swapped[0, :, 0::4], swapped[0, :, 2::4] = e[0, :, 2::4], e[0, :, 0::4]
    ref_sw, _ = oracle.gmm(xb, codes, np.array([m], np.int32), rhs_dtype=oracle.E4M3, rhs_block_scale=swapped,
                           rhs_block_scale_dtype=oracle.E8M0)
    assert not np.all(np.abs(got - ref_sw) <= bound)
