"""The exact two-term e4m3 split of bf16 activation rows, written out on the host for the
tests: the fp8 kernels' statement (the split pass and the in-kernel token split) in numpy, with
fp32 arithmetic where the kernels use fp32 and e4m3fn rounding to the nearest value, ties to
the even code, saturating at 448.  e4m3 values come from the oracle's decoder.  Steps holding
an infinity or a NaN are not covered (the kernels give their rows a NaN scale)."""

import numpy as np

import oracle


def e4m3_rne(y):
    """float32 -> e4m3fn codes: nearest value, ties to the even code, saturating at 448."""
    vals = oracle.decode(np.arange(0x7F, dtype=np.uint8))  # codes 0..126, increasing
    a = np.abs(y.astype(np.float64))
    idx = np.clip(np.searchsorted(vals, a), 1, 126)
    lo, hi = vals[idx - 1], vals[idx]
    up = (hi - a < a - lo) | ((hi - a == a - lo) & (idx % 2 == 0))
    code = np.where(a >= vals[126], 126, np.where(up, idx, idx - 1))
    return (code | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def split_statement(x_bits, step):
    """The two-term split written out on the host: per row and k step, e = the biased exponent
    of the step's largest |x| clamped to [8, 254], y = x * 2^(134 - e) in fp32,
    h = e4m3(y), l = e4m3(16 (y - h)) in fp32, scale = 2^(e - 134)."""
    m, k = x_bits.shape
    ksteps = -(-k // step)
    xf = (x_bits.astype(np.uint32) << 16).view(np.float32)
    planes = np.zeros((2, m, k), np.uint8)
    scales = np.zeros((m, ksteps), np.float32)
    for s in range(ksteps):
        cols = slice(s * step, min(k, (s + 1) * step))
        amax = ((x_bits[:, cols].astype(np.uint32) << 16) & 0x7FFFFFFF).max(axis=1)
        e = np.clip(amax >> 23, 8, 254).astype(np.uint32)
        inv = ((261 - e) << 23).astype(np.uint32).view(np.float32)
        y = xf[:, cols] * inv[:, None]
        h = e4m3_rne(y)
        vh = oracle.decode(h).astype(np.float32)
        planes[0][:, cols] = h
        planes[1][:, cols] = e4m3_rne((y - vh) * np.float32(16))
        scales[:, s] = ((e - 7) << 23).astype(np.uint32).view(np.float32)
    return planes, scales
