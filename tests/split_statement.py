"""The two-level e4m3 split of bf16 activation rows, written out on the host for the tests: the
fp8 kernels' statement (the split pass and the in-kernel token split) in numpy, with fp32
arithmetic where the kernels use fp32 and e4m3fn rounding to the nearest value, ties to the
even code, saturating at 448.  e4m3 values come from the oracle's decoder.

Per row and k step, with M1 the largest |x| (fp32 bits, sign cleared) and e1 its exponent field
clamped to [8, 254]:
    s1 = 2^(e1 - 134),  y = x * 2^(134 - e1),  h = e4m3(y),  l = e4m3(16 (y - h)),
    r = x - s1 (h + l / 16)                                   (exact in fp32)
and the same again on r with its own largest magnitude M2 (s2 = 0 and h2 = l2 = 0 codes when
r is zero over the whole step):
    s2 = 2^(e2 - 134),  h2 = e4m3(r 2^(134 - e2)),  l2 = e4m3(16 (r 2^(134 - e2) - h2)),
    r2 = r - s2 (h2 + l2 / 16).
The step is marked (s2's sign bit set) when r2 != 0 somewhere in it or it holds an infinity or a
NaN; s1 is then NaN for a non-finite step, which has no second level (s2 = -0)."""

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
    code = np.where(np.isnan(y), 0x7F, code)
    return (code | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def _exponent(amax_bits):
    return np.clip(amax_bits >> 23, 8, 254).astype(np.uint32)


def _scale(e):
    return ((e - 7) << 23).astype(np.uint32).view(np.float32)


def _inv_scale(e):
    return ((261 - e) << 23).astype(np.uint32).view(np.float32)


def _level(v, e):
    """One split level of the fp32 values v [rows, cols] with exponent fields e [rows]:
    (h codes, l codes, the rest v - s (h + l / 16))."""
    with np.errstate(invalid="ignore", over="ignore"):
        y = v * _inv_scale(e)[:, None]
        h = e4m3_rne(y)
        vh = oracle.decode(h).astype(np.float32)
        l = e4m3_rne((y - vh) * np.float32(16))
        vl = oracle.decode(l).astype(np.float32)
        rest = v - _scale(e)[:, None] * (vh + vl * np.float32(0.0625))
    return h, l, rest


def split_statement(x_bits, step):
    """Returns planes uint8 [4, m, k] (h, l, h2, l2) and scales float32 [m, k steps, 2] (s1, s2)."""
    m, k = x_bits.shape
    ksteps = -(-k // step)
    xf = (x_bits.astype(np.uint32) << 16).view(np.float32)
    planes = np.zeros((4, m, k), np.uint8)
    scales = np.zeros((m, ksteps, 2), np.float32)
    for s in range(ksteps):
        cols = slice(s * step, min(k, (s + 1) * step))
        x = xf[:, cols]
        amax = (x.view(np.uint32) & 0x7FFFFFFF).max(axis=1)
        e1 = _exponent(amax)
        h, l, r = _level(x, e1)
        nonfinite = amax >= 0x7F800000
        rmax = np.where(nonfinite, 0, (r.view(np.uint32) & 0x7FFFFFFF).max(axis=1))
        e2 = _exponent(rmax)
        h2, l2, r2 = _level(r, e2)
        live = rmax != 0
        h2[~live] = 0
        l2[~live] = 0
        s2 = np.where(live, _scale(e2), np.float32(0))
        rest = live & ((r2.view(np.uint32) & 0x7FFFFFFF) != 0).any(axis=1)
        marked = rest | nonfinite
        planes[0][:, cols], planes[1][:, cols], planes[2][:, cols], planes[3][:, cols] = h, l, h2, l2
        scales[:, s, 0] = np.where(nonfinite, np.float32(np.nan), _scale(e1))
        scales[:, s, 1] = (s2.view(np.uint32) | np.where(marked, 0x80000000, 0).astype(np.uint32)).view(np.float32)
    return planes, scales


def reconstruct(planes, scales, step):
    """s1 (h + l / 16) + s2 (h2 + l2 / 16) per value (fp64), and the per-row, per-step marks."""
    m, k = planes.shape[1:]
    v = [oracle.decode(planes[i]) for i in range(4)]
    s1 = np.repeat(scales[:, :, 0], step, axis=1)[:, :k].astype(np.float64)
    s2 = np.abs(np.repeat(scales[:, :, 1], step, axis=1)[:, :k].astype(np.float64))
    marked = np.signbit(scales[:, :, 1])
    return s1 * (v[0] + v[1] / 16) + s2 * (v[2] + v[3] / 16), marked


F16_ORDER = np.array([0, 4, 1, 5, 2, 6, 3, 7])  # k of each stored position within 8 k (4-bit weights)


def split_statement_f16(x_bits, perm):
    """The fp16 split of the integer-weight kernel (act_split_f16): per row and 128-wide step, with
    e the exponent field of the largest |x| (at least 15), sc = 2^(e - 141) and the fp16 values
    rne_f16(x / sc); a step is marked (second scale word -0) when some x is not sc times its fp16
    value, or it holds an infinity or a NaN.  Returns plane uint16 [m, k] (fp16 bits; each 8 k in
    the order F16_ORDER when perm) and scales float32 [m, k / 128, 2] (sc, +-0)."""
    m, k = x_bits.shape
    ksteps = k // 128
    xf = (x_bits.astype(np.uint32) << 16).view(np.float32)
    plane = np.zeros((m, k), np.uint16)
    scales = np.zeros((m, ksteps, 2), np.float32)
    for s in range(ksteps):
        cols = slice(128 * s, 128 * (s + 1))
        x = xf[:, cols]
        amax = (x.view(np.uint32) & 0x7FFFFFFF).max(axis=1)
        e = np.maximum(amax >> 23, 15).astype(np.uint32)
        sc = ((e - 14) << 23).astype(np.uint32).view(np.float32)
        inv = ((268 - e) << 23).astype(np.uint32).view(np.float32)
        with np.errstate(invalid="ignore", over="ignore"):
            h = (x * inv[:, None]).astype(np.float16)
            exact = h.astype(np.float32) * sc[:, None] == x
        marked = ~exact.all(axis=1) | (amax >= 0x7F800000)
        plane[:, cols] = h.view(np.uint16)
        scales[:, s, 0] = sc
        scales[:, s, 1] = np.where(marked, np.float32(-0.0), np.float32(0.0))
    if perm:
        plane = plane.reshape(m, k // 8, 8)[:, :, F16_ORDER].reshape(m, k)
    return plane, scales
