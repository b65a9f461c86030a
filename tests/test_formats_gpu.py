"""GPU parity for the weight formats of common.py's supported list beyond bf16 and e4m3fn:
e5m2, int8, int4, uint4 and e2m1 (the 4-bit ones packed two per byte, even k in the low
nibble), on the fp8 tensor-core kernel, against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, oracle_gmm

pytestmark = pytest.mark.gpu
DEV = "cuda"
FORMATS = ["e5m2", "int8", "int4", "uint4", "e2m1"]


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _gs(sizes):
    return torch.tensor(np.asarray(sizes, np.int32), dtype=torch.int32, device=DEV)


def _fmt_kw(fmt):
    return {"rhs_format": fmt} if fmt in W.PACKED else {}


def _case(fmt, m, k, n, sizes, nb, *, out_dtype=torch.bfloat16, group_offset=0, local=None, seed=0,
          with_scale=True, bias_dtype=torch.bfloat16):
    sizes = np.asarray(sizes, np.int32)
    L = local if local is not None else sizes.size - group_offset
    lhs = W.normal((m, k), 1.0, seed + 1, DEV)
    rhs = W.weights(fmt, (L, n, k), seed + 2, DEV)
    top = W.FORMAT_MAX[fmt]
    scale = W.uniform((L, nb, 1, n), 0.5 / top, 2.0 / top, seed + 3, DEV) if with_scale else None
    bias = None if bias_dtype is None else W.normal((L, 1, n), 1.0, seed + 4, DEV, dtype=bias_dtype)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, rhs_bias=bias, group_offset=group_offset,
                out_dtype=out_dtype, **_fmt_kw(fmt))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(lhs, rhs, sizes, group_offset=group_offset, rhs_scale=scale, rhs_bias=bias,
                          rhs_format=fmt)
    finite = np.isfinite(ref)
    if not finite.all():  # e5m2 infinities and NaN: non-finite wherever the oracle is
        g = out.cpu().to(torch.float64).numpy()
        assert (np.isfinite(g) == finite).all()
        ref, mag = np.where(finite, ref, 0.0), np.where(finite, mag, 0.0)
        out = torch.from_numpy(np.where(finite, g, 0.0))
    check_close(out, ref, mag, f"{fmt} m={m} k={k} n={n} nb={nb} sizes={sizes.tolist()}")
    return out


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16out", "f32out"])
def test_ragged_decode_shapes(fmt, out_dtype):
    # groups of 0..40 rows (chunks of 8, 16 and 32 rows, some spanning two chunks), n with an
    # 8-wide tail, k = 640 (an odd number of 128-wide sub-tiles), quant blocks of 128
    sizes = [3, 0, 17, 1, 40, 0, 8, 16, 5, 33]
    _case(fmt, int(np.sum(sizes)) + 9, 640, 392, sizes, 5, out_dtype=out_dtype, seed=3)


@pytest.mark.parametrize("fmt", FORMATS)
def test_group_offset_and_f32_bias_no_scale(fmt):
    sizes = [3, 0, 17, 1, 40, 0, 8, 16, 5, 33]
    _case(fmt, 140, 256, 256, sizes, 1, group_offset=4, local=5, with_scale=False, bias_dtype=torch.float32, seed=5)


@pytest.mark.parametrize("fmt", FORMATS)
def test_every_code_comes_out_exactly(fmt):
    # out[r, c] = sum_k onehot(r)[k] * W[c, k] = W[c, r]: one exact product per output
    m = k = 256
    n = 128
    if fmt in W.PACKED:
        # row c: bytes (c + j) % 256 -> every nibble pair in every position
        codes = ((np.arange(n)[:, None] + np.arange(k // 2)[None, :]) % 256).astype(np.uint8)
        rhs = torch.from_numpy(codes[None]).to(DEV)
    elif fmt == "int8":
        codes = ((np.arange(n)[:, None] + np.arange(k)[None, :]) % 256).astype(np.uint8).view(np.int8)
        rhs = torch.from_numpy(codes[None].copy()).to(DEV)
    else:  # e5m2 finite codes (infinities and NaN are covered by the next test)
        finite = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], np.uint8)
        codes = finite[(np.arange(n)[:, None] + np.arange(k)[None, :]) % finite.size]
        rhs = torch.from_numpy(codes[None]).view(torch.float8_e5m2).to(DEV)
    lhs = torch.eye(m, k, dtype=torch.bfloat16, device=DEV)
    out = G.gmm(lhs, rhs, _gs([m]), out_dtype=torch.float32, **_fmt_kw(fmt))
    expect = oracle.decode(codes, {"e5m2": oracle.E5M2, "int8": oracle.INT8, "int4": oracle.INT4,
                                   "uint4": oracle.UINT4, "e2m1": oracle.E2M1}[fmt]).T
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), expect)
    assert G.read_device_errors() == 0


def test_e5m2_infinities_and_nan():
    # A non-finite weight makes every output that uses it non-finite on this path.  The
    # definition gives +-inf for an infinite weight; here the activation is split into two
    # e4m3 terms, and the l term times the infinity is NaN when l is 0 or of the other sign,
    # so such an output is +-inf or NaN depending on the row.
    m, k, n = 16, 128, 128
    codes = np.full((1, n, k), 0x3C, np.uint8)  # 1.0
    codes[0, 5, 7] = 0x7C    # +inf
    codes[0, 9, 100] = 0x7F  # NaN
    lhs = W.normal((m, k), 1.0, 3, DEV).abs()
    out = G.gmm(lhs, torch.from_numpy(codes).view(torch.float8_e5m2).to(DEV), _gs([m]),
                out_dtype=torch.float32).cpu()
    assert (~torch.isfinite(out[:, 5])).all()
    assert not (out[:, 5] == float("-inf")).any()
    assert torch.isnan(out[:, 9]).all()
    others = [c for c in range(n) if c not in (5, 9)]
    assert torch.isfinite(out[:, others]).all()


@pytest.mark.parametrize("fmt", ["int8", "int4", "e2m1"])
def test_integer_weights_exact(fmt):
    # integer-valued lhs and power-of-two scales: every sum is exact in fp32
    m, k, n = 48, 256, 128
    sizes = np.array([10, 0, 21, 17], np.int32)
    lhs = W.integer_valued((m, k), -4, 4, 5, DEV)
    rhs = W.weights(fmt, (4, n, k), 6, DEV)
    scale = torch.tensor([0.5, 2.0], device=DEV).repeat(4, 1).reshape(4, 2, 1, 1).expand(4, 2, 1, n).contiguous()
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, out_dtype=torch.float32, **_fmt_kw(fmt))
    ref, _ = oracle_gmm(lhs, rhs, sizes, rhs_scale=scale, rhs_format=fmt)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_decode_workload_full(fmt):
    """The decode workload's shapes (256 rows, 64 experts of [2048, 4096], 32 k-blocks) with
    weights in another format, every output element checked."""
    d = W.fp8_decode(DEV, fmt=fmt)
    sizes = d["group_sizes"]
    out = G.gmm(d["lhs"], d["rhs"], _gs(sizes), rhs_scale=d["rhs_scale"], rhs_bias=d["rhs_bias"], **_fmt_kw(fmt))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(d["lhs"], d["rhs"], sizes, rhs_scale=d["rhs_scale"], rhs_bias=d["rhs_bias"],
                          rhs_format=fmt)
    check_close(out, ref, mag, f"decode workload, {fmt} weights")
