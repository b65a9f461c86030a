"""bf16 activations against 8- and 4-bit weights: every element of the result must meet the
bound |gpu - ref| <= 1e-3 * mag + 2^-8 * |ref| for every finite input, however widely the
magnitudes inside one k step of a row are spread, and non-finite activations must give what
the definition gives (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230",
gmm.py _accum: the bf16 activations meet the weights in a dot_general with an fp32 result,
so every product is exact and only the fp32 sums round; x * inf is +-inf, 0 * inf is NaN).

The hard rows put a large value on weights that are zero and small values on live weights, so
that mag (the sum of |x w s|) is made of the small values alone while the large one sets the
row's scale.  Both ways of splitting the rows run: the split pass (options act_split="pass") and
the split inside the kernel (act_split="kernel")."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import ORACLE_FORMAT, bits, check_close, use_options

pytestmark = pytest.mark.gpu
DEV = "cuda"
FORMATS = ["e4m3", "e5m2", "e2m1", "int8", "int4", "uint4"]


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


@pytest.fixture(params=["pass", "kernel"])
def split(request, monkeypatch):
    use_options(monkeypatch, act_split=request.param)
    return request.param


def _step(fmt):
    return 128 if fmt == "int8" else 256


def _bf16(values):
    """float64 values -> bf16 tensor on the device (each value must be a bf16 value)."""
    t = torch.tensor(np.asarray(values, np.float64), dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), "test values must be exact bf16 values"
    return b.to(DEV)


def _zero_weights_at(rhs, fmt, kmask):
    """rhs with every weight at the k positions of `kmask` ([k] bool) set to zero."""
    if fmt in W.PACKED:
        codes = rhs.cpu().numpy().copy()
        lo, hi = codes & 0x0F, codes >> 4
        lo[..., kmask[0::2]] = 0
        hi[..., kmask[1::2]] = 0
        return torch.from_numpy((lo | (hi << 4)).astype(np.uint8)).to(DEV)
    w = rhs.clone()
    w.view(torch.uint8)[..., torch.from_numpy(kmask).to(DEV)] = 0
    return w


def _run(lhs, rhs, fmt, sizes, scale, bias=None, group_offset=0, out_dtype=torch.float32):
    kw = {"rhs_format": fmt} if fmt in W.PACKED else {}
    out = G.gmm(lhs, rhs, torch.tensor(sizes, dtype=torch.int32, device=DEV), rhs_scale=scale, rhs_bias=bias,
                group_offset=group_offset, out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, group_offset=group_offset,
                          rhs_scale=None if scale is None else bits(scale),
                          rhs_bias=None if bias is None else bits(bias), rhs_dtype=ORACLE_FORMAT[fmt])
    return out, ref, mag


def _hard_rows(k, step):
    """Rows whose steps each hold a large value at their first position (where the weights are
    zero) and small ones elsewhere:
      0  1.0 and 3 * 2^-22 (a small value 2^-22 of the large one, rounded by a 2^13 split range)
      1  1.0 and bf16 subnormals (3 * 2^-133 and -5 * 2^-133)
      2  2^100 and +-5 * 2^-30
      3  -448 and values 2^-20 (1 + j / 128) of alternating sign
      4  three magnitudes: 1.0, 2^-30 (1 + j / 64) and 2^-60 (1 + j / 32) in turn
      5  2^-120 and 3 * 2^-133 (the whole step below 2^-119)
      6  3 * 2^-22 everywhere, no large value
      7  zero"""
    j = np.arange(k)
    first = (j % step) == 0
    rows = np.zeros((8, k))
    rows[0] = np.where(first, 1.0, 3 * 2.0 ** -22)
    rows[1] = np.where(first, 1.0, np.where(j % 2 == 0, 3.0, -5.0) * 2.0 ** -133)
    rows[2] = np.where(first, 2.0 ** 100, np.where(j % 3 == 0, -5.0, 5.0) * 2.0 ** -30)
    rows[3] = np.where(first, -448.0, np.where(j % 2 == 0, 1.0, -1.0) * (1 + (j % 128) / 128) * 2.0 ** -20)
    third = np.where(j % 2 == 0, (1 + (j % 64) / 64) * 2.0 ** -30, (1 + (j % 32) / 32) * 2.0 ** -60)
    rows[4] = np.where(first, 1.0, third)
    rows[5] = np.where(first, 2.0 ** -120, 3 * 2.0 ** -133)
    rows[6] = 3 * 2.0 ** -22
    return rows, first


@pytest.mark.parametrize("fmt", FORMATS)
def test_small_values_beside_a_large_value_on_zero_weights(fmt, split):
    m, k, n = 8, 512, 136  # n: one full 128-wide tile and a tail of 8
    step = _step(fmt)
    rows, first = _hard_rows(k, step)
    lhs = _bf16(rows)
    rhs = _zero_weights_at(W.weights(fmt, (1, n, k), 301, DEV), fmt, first)
    # scales in [1, 2): the subnormal rows' results stay above 2^-130, where fp32 (the
    # accumulator and the f32 output) still holds them to 2^-19 of their size
    scale = W.uniform((1, 2, 1, n), 1.0, 2.0, 302, DEV)
    out, ref, mag = _run(lhs, rhs, fmt, np.array([m], np.int32), scale)
    check_close(out, ref, mag, f"{fmt} split={split}: small values beside a large one on zero weights")


@pytest.mark.parametrize("fmt", ["e4m3", "int8", "int4"])
def test_three_magnitudes_in_ragged_groups(fmt, split):
    """Random rows made of three magnitude clusters 2^25 apart, the largest (the first value of
    every step) on zero weights for half of the columns, over ragged groups (chunks of 1 to 16 rows, a group across two
    chunks), a group_offset slice and a bf16 output."""
    sizes = np.array([5, 0, 23, 1, 9, 14], np.int32)
    m, k, n = int(sizes.sum()) + 3, 768, 264
    step = _step(fmt)
    g = np.random.Generator(np.random.PCG64(303))
    cluster = g.integers(1, 3, (m, k))
    cluster[:, ::step] = 0  # every step holds a large value, at its first position only
    mant = g.uniform(1, 2, (m, k)) * np.where(g.random((m, k)) < 0.5, -1, 1)
    x = mant * 2.0 ** (-25.0 * cluster)
    lhs = torch.tensor(x).to(torch.bfloat16).to(DEV)
    big = np.zeros(k, bool)
    big[::step] = True
    L = 4
    rhs = W.weights(fmt, (L, n, k), 304, DEV)
    dead = _zero_weights_at(rhs, fmt, big)
    # columns [0, 132) see the large values only through zero weights
    rhs[:, :132] = dead[:, :132]
    top = W.FORMAT_MAX[fmt]
    scale = W.uniform((L, 3, 1, n), 0.5 / top, 2.0 / top, 305, DEV)
    out, ref, mag = _run(lhs, rhs, fmt, sizes, scale, group_offset=2, out_dtype=torch.bfloat16)
    check_close(out, ref, mag, f"{fmt} split={split}: three magnitudes")


@pytest.mark.parametrize("fmt", ["e4m3", "int8", "e2m1"])
def test_infinite_activations(fmt, split):
    """x * w summed with an infinite x: +-inf where the weight is non-zero, NaN where it is
    zero (0 * inf) and where +inf and -inf meet; a NaN activation makes its row NaN."""
    m, k, n = 6, 512, 128
    step = _step(fmt)
    x = W.normal((m, k), 1.0, 306, "cpu").double().numpy()
    x[0, 5] = np.inf
    x[1, 5] = -np.inf
    x[2, 5], x[2, 300] = np.inf, -np.inf
    x[3, 9] = np.nan
    x[4, 0] = np.inf  # the large value of its step is infinite; the others finite
    lhs = torch.tensor(x).to(torch.bfloat16).to(DEV)
    rhs = W.weights(fmt, (1, n, k), 307, DEV)
    # weights at k = 5 and 300 are zero for every third column
    kmask = np.zeros(k, bool)
    kmask[[5, 300]] = True
    dead = _zero_weights_at(rhs, fmt, kmask)
    rhs[:, ::3] = dead[:, ::3]
    top = W.FORMAT_MAX[fmt]
    scale = W.uniform((1, 2, 1, n), 0.5 / top, 2.0 / top, 308, DEV)
    bias = W.normal((1, 1, n), 1.0, 309, DEV)
    out, ref, mag = _run(lhs, rhs, fmt, np.array([m], np.int32), scale, bias=bias)
    assert np.isinf(ref[0]).any() and np.isnan(ref[0]).any()  # the case covers both outcomes
    check_close(out, ref, mag, f"{fmt} split={split}: infinite activations")
    assert torch.isfinite(out[5]).all()


def test_fp8_decode_workload_with_wide_rows(split):
    """The decode workload's shapes (256 rows, 64 experts of [2048, 4096] e4m3, 32 quant
    blocks, bias) with every 16th activation row replaced by a hard row (sampled rows are
    checked against the oracle; the other rows must be unchanged by the replacement)."""
    d = W.fp8_decode(DEV)
    sizes = d["group_sizes"]
    hard, first = _hard_rows(4096, 256)
    lhs = d["lhs"].clone()
    for i, r in enumerate(range(0, 256, 16)):
        lhs[r] = _bf16(hard[i % 7])
    gs = torch.tensor(sizes, dtype=torch.int32, device=DEV)
    out = G.gmm(lhs, d["rhs"], gs, rhs_scale=d["rhs_scale"])
    plain = G.gmm(d["lhs"], d["rhs"], gs, rhs_scale=d["rhs_scale"])
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    rows = np.unique(np.concatenate([np.arange(0, 256, 16), np.arange(5, 256, 37)]))
    ref, mag = oracle.gmm(bits(lhs), bits(d["rhs"]), sizes, rhs_scale=bits(d["rhs_scale"]), rows=rows)
    check_close(out[torch.from_numpy(rows).to(DEV)], ref, mag, f"decode workload, hard rows, split={split}")
    keep = [r for r in range(256) if r % 16 != 0]
    assert torch.equal(out[keep], plain[keep])


def test_infinite_e5m2_weights(split):
    """Reading on infinite e5m2 weights: the split's terms can be zero (0 * inf = NaN), so a
    column that meets an infinite weight comes out +-inf or NaN where the definition gives
    +-inf; every other column is within the bound."""
    m, k, n = 12, 512, 128
    lhs = W.normal((m, k), 1.0, 310, DEV)
    codes = W.weights("e5m2", (1, n, k), 311, DEV).view(torch.uint8).clone()
    touched = [3, 40, 77, 100]
    for j, c in enumerate(touched):
        codes[0, c, 17 * (j + 1)] = 0x7C if j % 2 == 0 else 0xFC  # +inf, -inf
    rhs = codes.view(torch.float8_e5m2)
    scale = W.uniform((1, 2, 1, n), 1.0, 2.0, 312, DEV)
    out, ref, mag = _run(lhs, rhs, "e5m2", np.array([m], np.int32), scale)
    assert np.isinf(ref[:, touched]).all()
    o = out.cpu()
    assert not torch.isfinite(o[:, touched]).any()
    rest = [c for c in range(n) if c not in touched]
    check_close(o[:, rest], ref[:, rest], mag[:, rest], f"e5m2 split={split}: columns without infinities")
