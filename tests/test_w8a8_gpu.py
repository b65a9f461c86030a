"""The W8A8 path (page "gemm_quant.rs": per-token-group e4m3 activations with f32 scales per 128
columns, e4m3 weights with per-block scales): the quantiser's codes and scales must equal the
oracle's bit for bit (NaN codes compared without their sign), and the W8A8 grouped matmul must
match the oracle evaluated on the same codes and scales."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_quant(x, group):
    q, sc = G.quantize_e4m3(x, group=group)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_e4m3(_bits(x), group)
    gq = q.view(torch.uint8).cpu().numpy()
    gs = sc.cpu().numpy()
    nan_q = (rq & 0x7F) == 0x7F
    assert np.array_equal((gq & 0x7F) == 0x7F, nan_q), "NaN codes differ"
    assert np.array_equal(gq[~nan_q], rq[~nan_q]), f"codes differ at {np.argwhere((gq != rq) & ~nan_q)[:5]}"
    nan_s = np.isnan(rs)
    assert np.array_equal(np.isnan(gs), nan_s)
    assert np.array_equal(gs[~nan_s].view(np.uint32), rs[~nan_s].view(np.uint32)), "scales differ"


@pytest.mark.parametrize("group", [64, 128, 256])
@pytest.mark.parametrize("m,k", [(1, 256), (37, 512), (300, 2048)])
def test_quantiser_matches_oracle_bit_for_bit(group, m, k):
    x = W.normal((m, k), 1.0, 100 + m, DEV)
    _check_quant(x, group)


def test_quantiser_wide_range_zero_and_nan_groups():
    m, k = 8, 1024
    x = W.normal((m, k), 1.0, 7, DEV)
    # rows spanning many binades, a zero group, a group with a single tiny value, NaN, inf
    x[0] *= torch.logspace(-30, 30, k, base=2.0, device=DEV).to(torch.bfloat16)
    x[1, :128] = 0
    x[2, 128:256] = 0
    x[2, 200] = 1e-30
    x[3, 5] = float("nan")
    x[4, 300] = float("inf")
    x[5, 600] = -float("inf")
    x[6] = x[6] * 1e20
    x[7] = x[7] * 1e-20
    _check_quant(x, 128)


def test_quantiser_ties_round_to_even():
    # amax 448 gives scale 1, so the codes are the e4m3 rounding of the bf16 values themselves;
    # values half-way between e4m3 neighbours must go to the even code
    m, k = 2, 128
    vals = torch.tensor([448.0, 1.0 + 1 / 16, 1.0 + 3 / 16, 2.0 + 1 / 8, -(1.0 + 1 / 16), 17.0, 19.0, 0.0],
                        dtype=torch.float32)
    x = vals.repeat(k // vals.numel()).reshape(1, k).repeat(m, 1).to(torch.bfloat16).to(DEV)
    _check_quant(x, 128)
    q, sc = G.quantize_e4m3(x, group=128)
    assert sc[0, 0].item() == 1.0
    dec = q.float().cpu()[0, :8].tolist()
    assert dec == [448.0, 1.0, 1.25, 2.0, -1.0, 16.0, 20.0, 0.0]


def test_quantiser_rejects_bad_arguments():
    x = W.normal((4, 256), 1.0, 1, DEV)
    with pytest.raises(G.GmmError) as e:
        G.quantize_e4m3(x, group=96)
    assert e.value.status == 3  # GMM_ERR_SHAPE
    with pytest.raises(G.GmmError):
        G.quantize_e4m3(W.normal((4, 200), 1.0, 1, DEV), group=128)
    with pytest.raises(G.GmmError):
        G.quantize_e4m3(x.float(), group=128)


# ------------------------------------------------------------------ W8A8 grouped matmul
from parity import ORACLE_FORMAT, check_close  # noqa: E402

FORMATS = ["e4m3", "e5m2", "int8", "int4", "uint4", "e2m1"]


def _quantised(m, k, seed, group=128):
    """Activations quantised by the oracle on the CPU: (codes uint8, scales f32, and both on the device)."""
    x = W.normal((m, k), 1.0, seed)
    q_np, s_np = oracle.quantize_e4m3(_bits(x), group)
    q = torch.from_numpy(q_np).view(torch.float8_e4m3fn).to(DEV)
    return q_np, s_np, q, torch.from_numpy(s_np).to(DEV)


def _weights(fmt, L, n, k, nb, seed, e8m0=False):
    rhs = W.weights(fmt, (L, n, k), seed, DEV)
    if e8m0:
        scale = torch.randint(118, 133, (L, nb, 1, n), generator=torch.Generator().manual_seed(seed + 1),
                              dtype=torch.uint8)
        scale[0, 0, 0, :3] = torch.tensor([0, 255, 127], dtype=torch.uint8)
        scale = scale.to(DEV)
    else:
        top = W.FORMAT_MAX[fmt]
        scale = W.uniform((L, nb, 1, n), 0.5 / top, 2.0 / top, seed + 1, DEV)
    bias = W.normal((L, 1, n), 1.0, seed + 2, DEV)
    kw = {"rhs_format": fmt} if fmt in W.PACKED else {}
    return rhs, scale, bias, kw


def _oracle(lhs_np, rhs, sizes, scale, bias, fmt, lhs_scale=None, lhs_dtype=None, **kw):
    sc = scale.cpu().numpy() if scale.dtype == torch.uint8 else _stored(scale)
    return oracle.gmm(lhs_np, _stored(rhs), sizes, rhs_scale=sc, rhs_bias=_stored(bias), lhs_dtype=lhs_dtype,
                      rhs_dtype=ORACLE_FORMAT[fmt], lhs_scale=lhs_scale, **kw)


def _stored(t):
    return W.stored_bits(t)


SIZES = np.array([0, 37, 1, 64, 50, 9], np.int32)  # sum 161 of 200 rows: a tail of rows in no group


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", FORMATS)
def test_w8a8_matches_oracle(fmt, out_dtype):
    m, k, n, L = 200, 512, 384, 6
    q_np, s_np, q, sc = _quantised(m, k, 11)
    rhs, scale, bias, kw = _weights(fmt, L, n, k, 4, 12)
    gs = torch.tensor(SIZES, device=DEV)
    out = G.gmm(q, rhs, gs, rhs_scale=scale, rhs_bias=bias, lhs_scale=sc, out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle(q_np, rhs, SIZES, scale, bias, fmt, lhs_scale=s_np, lhs_dtype=oracle.E4M3)
    check_close(out, ref, mag, f"W8A8 {fmt}")


@pytest.mark.parametrize("fmt", ["e4m3", "int8", "e2m1"])
@pytest.mark.parametrize("lhs_kind", ["bf16", "e4m3"])
def test_e8m0_weight_scales(fmt, lhs_kind):
    m, k, n, L = 200, 768, 256, 6
    rhs, scale, bias, kw = _weights(fmt, L, n, k, 3, 21, e8m0=True)
    gs = torch.tensor(SIZES, device=DEV)
    if lhs_kind == "e4m3":
        q_np, s_np, q, sc = _quantised(m, k, 22)
        out = G.gmm(q, rhs, gs, rhs_scale=scale, rhs_bias=bias, lhs_scale=sc, out_dtype=torch.float32, **kw)
        ref, mag = _oracle(q_np, rhs, SIZES, scale, bias, fmt, lhs_scale=s_np, lhs_dtype=oracle.E4M3)
    else:
        x = W.normal((m, k), 1.0, 22, DEV)
        out = G.gmm(x, rhs, gs, rhs_scale=scale, rhs_bias=bias, out_dtype=torch.float32, **kw)
        ref, mag = _oracle(_stored(x), rhs, SIZES, scale, bias, fmt)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    check_close(out, ref, mag, f"E8M0 scales, {lhs_kind} activations, {fmt} weights")
    # the byte 255 zeroes block 0 of column 1 in group 0's slice: its rows equal the oracle's there too
    assert scale[0, 0, 0, 1].item() == 255


def test_w8a8_without_lhs_scale_and_with_wide_lhs_blocks():
    m, k, n, L = 200, 1024, 256, 6
    rhs, scale, bias, kw = _weights("e4m3", L, n, k, 2, 31)
    gs = torch.tensor(SIZES, device=DEV)
    q_np, s_np, q, sc = _quantised(m, k, 32, group=256)  # lhs blocks 256 wide
    out = G.gmm(q, rhs, gs, rhs_scale=scale, rhs_bias=bias, lhs_scale=sc, out_dtype=torch.float32)
    ref, mag = _oracle(q_np, rhs, SIZES, scale, bias, "e4m3", lhs_scale=s_np, lhs_dtype=oracle.E4M3)
    check_close(out, ref, mag, "lhs blocks of 256")
    out = G.gmm(q, rhs, gs, rhs_scale=scale, rhs_bias=bias, out_dtype=torch.float32)  # lhs scale 1
    ref, mag = _oracle(q_np, rhs, SIZES, scale, bias, "e4m3", lhs_dtype=oracle.E4M3)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    check_close(out, ref, mag, "no lhs scale")


@pytest.mark.parametrize("device_offset", [False, True])
def test_w8a8_group_offset_and_kept_rows(device_offset):
    m, k, n, G_, L, go = 200, 512, 256, 6, 3, 2
    q_np, s_np, q, sc = _quantised(m, k, 41)
    rhs, scale, bias, kw = _weights("int4", L, n, k, 4, 42)
    gs = torch.tensor(SIZES, device=DEV)
    offset = torch.tensor([go], dtype=torch.int32, device=DEV) if device_offset else go
    out = G.gmm(q, rhs, gs, rhs_scale=scale, rhs_bias=bias, lhs_scale=sc, group_offset=offset,
                out_dtype=torch.float32, **kw)
    ref, mag = _oracle(q_np, rhs, SIZES, scale, bias, "int4", lhs_scale=s_np, lhs_dtype=oracle.E4M3, group_offset=go)
    check_close(out, ref, mag, "W8A8 with group_offset")
    before = W.normal((m, n), 3.0, 43, DEV, dtype=torch.float32) + 100.0
    kept = before.clone()
    G.gmm_into(q, rhs, gs, kept, rhs_scale=scale, rhs_bias=bias, lhs_scale=sc, group_offset=offset, **kw)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    offs = np.concatenate([[0], np.cumsum(SIZES)])
    lo, hi = offs[go], offs[go + L]
    assert torch.equal(kept[lo:hi], out[lo:hi])
    assert torch.equal(kept[:lo], before[:lo]) and torch.equal(kept[hi:], before[hi:])


def test_quantise_then_gmm_equals_the_oracle_pipeline():
    m, k, n, L = 200, 512, 384, 6
    x = W.normal((m, k), 1.0, 51)
    x[7, 100] = float("nan")  # row 7 (group 1) quantises to a NaN scale: its outputs are NaN
    rhs, scale, bias, kw = _weights("e4m3", L, n, k, 4, 52)
    gs = torch.tensor(SIZES, device=DEV)
    q, sc = G.quantize_e4m3(x.to(DEV))
    out = G.gmm(q, rhs, gs, rhs_scale=scale, rhs_bias=bias, lhs_scale=sc, out_dtype=torch.float32)
    torch.cuda.synchronize()
    q_np, s_np = oracle.quantize_e4m3(_bits(x), 128)
    ref, mag = _oracle(q_np, rhs, SIZES, scale, bias, "e4m3", lhs_scale=s_np, lhs_dtype=oracle.E4M3)
    assert torch.isnan(out[7]).all()
    keep = np.ones(m, bool)
    keep[7] = False
    check_close(out[torch.from_numpy(keep).to(DEV)], ref[keep], mag[keep], "quantise + W8A8 gmm")


def test_w8a8_decode_workload_sampled_rows():
    wl = W.fp8_decode(DEV)
    sizes = wl["group_sizes"]
    m, k = wl["lhs"].shape
    q, sc = G.quantize_e4m3(wl["lhs"])
    out = G.gmm(q, wl["rhs"], torch.tensor(sizes, device=DEV), rhs_scale=wl["rhs_scale"],
                rhs_bias=wl["rhs_bias"], lhs_scale=sc)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    q_np, s_np = oracle.quantize_e4m3(_bits(wl["lhs"]), 128)
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_np)
    rows = np.random.default_rng(5).choice(m, 24, replace=False)
    ref, mag = oracle.gmm(q_np, _stored(wl["rhs"]), sizes, rhs_scale=_stored(wl["rhs_scale"]),
                          rhs_bias=_stored(wl["rhs_bias"]), rows=rows, lhs_dtype=oracle.E4M3, rhs_dtype=oracle.E4M3,
                          lhs_scale=s_np)
    check_close(out[torch.from_numpy(rows).to(DEV)], ref, mag, "W8A8 decode workload")
