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
