"""Microscaling weight block scales on the GPU: MXFP8 (float8_e4m3fn weights with one E8M0
scale per 32 consecutive k of a weight row) against the oracle evaluated on the same stored
bytes, with the per-block fp32 scale, bias, ragged groups, group_offset and both output dtypes,
on the fp16-weight kernel (the default) and on the decoding kernel (e4m3_kernel="decode", and
scales that are not 4-byte aligned); then NVFP4."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, use_options

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _mx_scales(shape, seed, specials=True):
    g = torch.Generator().manual_seed(seed)
    e = torch.randint(118, 137, shape, generator=g, dtype=torch.uint8)
    if specials:
        e[0, 1, 0] = 255   # a zero block
        e[0, 2, 1] = 0     # 2^-127
    return e


def _oracle(lhs, rhs, sizes, mx, go=0, rhs_scale=None, bias=None, rows=None):
    return oracle.gmm(W.stored_bits(lhs), W.stored_bits(rhs), sizes, group_offset=go,
                      rhs_scale=None if rhs_scale is None else W.stored_bits(rhs_scale),
                      rhs_bias=None if bias is None else W.stored_bits(bias), rows=rows,
                      rhs_dtype=oracle.E4M3, rhs_block_scale=mx.cpu().numpy(), rhs_block_scale_dtype=oracle.E8M0)


SIZES = np.array([0, 37, 1, 64, 50, 9], np.int32)


@pytest.mark.parametrize("kernel", ["auto", "decode"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_scale", [False, True])
def test_mxfp8_matches_oracle(with_scale, out_dtype, kernel, monkeypatch):
    if kernel == "decode":
        use_options(monkeypatch, e4m3_kernel="decode")
    m, k, n, L = 200, 512, 384, 6
    lhs = W.normal((m, k), 1.0, 61, DEV)
    rhs = W.weights("e4m3", (L, n, k), 62, DEV)
    mx = _mx_scales((L, n, k // 32), 63).to(DEV)
    scale = W.uniform((L, 2, 1, n), 0.5, 2.0, 64, DEV) if with_scale else None
    bias = W.normal((L, 1, n), 1.0, 65, DEV)
    out = G.gmm(lhs, rhs, torch.tensor(SIZES, device=DEV), rhs_scale=scale, rhs_bias=bias, rhs_block_scale=mx,
                out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle(lhs, rhs, SIZES, mx, rhs_scale=scale, bias=bias)
    check_close(out, ref, mag, f"MXFP8 (scale {with_scale}, {kernel})")


@pytest.mark.parametrize("device_offset", [False, True])
def test_mxfp8_group_offset_and_kept_rows(device_offset):
    m, k, n, L, go = 200, 256, 256, 3, 2
    lhs = W.normal((m, k), 1.0, 71, DEV)
    rhs = W.weights("e4m3", (L, n, k), 72, DEV)
    mx = _mx_scales((L, n, k // 32), 73).to(DEV)
    gs = torch.tensor(SIZES, device=DEV)
    offset = torch.tensor([go], dtype=torch.int32, device=DEV) if device_offset else go
    out = G.gmm(lhs, rhs, gs, rhs_block_scale=mx, group_offset=offset, out_dtype=torch.float32)
    ref, mag = _oracle(lhs, rhs, SIZES, mx, go=go)
    check_close(out, ref, mag, "MXFP8 with group_offset")
    before = W.normal((m, n), 3.0, 74, DEV, dtype=torch.float32) + 100.0
    kept = before.clone()
    G.gmm_into(lhs, rhs, gs, kept, rhs_block_scale=mx, group_offset=offset)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    offs = np.concatenate([[0], np.cumsum(SIZES)])
    lo, hi = offs[go], offs[go + L]
    assert torch.equal(kept[lo:hi], out[lo:hi])
    assert torch.equal(kept[:lo], before[:lo]) and torch.equal(kept[hi:], before[hi:])


def test_unit_block_scales_equal_the_plain_decoding_kernel(monkeypatch):
    # E8M0 127 is 1: on the decoding kernel the result is the one without block scales, bit for bit
    m, k, n, L = 120, 384, 256, 4
    lhs = W.normal((m, k), 1.0, 81, DEV)
    rhs = W.weights("e4m3", (L, n, k), 82, DEV)
    sizes = torch.tensor([30, 0, 50, 40], dtype=torch.int32, device=DEV)
    ones = torch.full((L, n, k // 32), 127, dtype=torch.uint8, device=DEV)
    use_options(monkeypatch, e4m3_kernel="decode")
    with_mx = G.gmm(lhs, rhs, sizes, rhs_block_scale=ones, out_dtype=torch.float32)
    plain = G.gmm(lhs, rhs, sizes, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(with_mx, plain)


def test_mxfp8_marked_rows_are_summed_again_with_their_block_scales():
    # activation steps the fp16 split cannot hold mark their rows, which are summed again from
    # the stored values with the E8M0 scales; a zero block (E8M0 255) and 2^-127 included
    m, k, n, L = 24, 512, 256, 2
    x = W.normal((m, k), 1.0, 141).float()
    x[3, ::128] = 1.0
    x[3, 1::128] = 1.5 * 2.0 ** -40
    x[5] = x[5] * torch.pow(2.0, torch.linspace(-40, 10, k))
    x[7, ::128] = 3e4
    x[7, 5::128] = 2.0 ** -30
    lhs = x.to(torch.bfloat16).to(DEV)
    rhs = W.weights("e4m3", (L, n, k), 142, DEV)
    mx = _mx_scales((L, n, k // 32), 143).to(DEV)
    sizes = np.array([10, 14], np.int32)
    out = G.gmm(lhs, rhs, torch.tensor(sizes, device=DEV), rhs_block_scale=mx, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle(lhs, rhs, sizes, mx)
    check_close(out, ref, mag, "MXFP8 with marked rows")


def test_mxfp8_scales_off_four_byte_alignment_take_the_decoding_kernel():
    m, k, n, L = 64, 256, 128, 2
    lhs = W.normal((m, k), 1.0, 151, DEV)
    rhs = W.weights("e4m3", (L, n, k), 152, DEV)
    mx = _mx_scales((L, n, k // 32), 153)
    store = torch.empty(mx.numel() + 1, dtype=torch.uint8, device=DEV)
    store[1:] = mx.reshape(-1).to(DEV)
    shifted = store[1:].view(L, n, k // 32)  # one byte past an aligned allocation
    sizes = np.array([40, 24], np.int32)
    out = G.gmm(lhs, rhs, torch.tensor(sizes, device=DEV), rhs_block_scale=shifted, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle(lhs, rhs, sizes, mx)
    check_close(out, ref, mag, "MXFP8, scales at an odd address")


def test_mxfp8_decode_workload_sampled_rows():
    wl = W.fp8_decode(DEV)
    sizes = wl["group_sizes"]
    m, k = wl["lhs"].shape
    L, n = wl["rhs"].shape[0], wl["rhs"].shape[1]
    mx = _mx_scales((L, n, k // 32), 91, specials=False).to(DEV)
    out = G.gmm(wl["lhs"], wl["rhs"], torch.tensor(sizes, device=DEV), rhs_block_scale=mx,
                rhs_scale=wl["rhs_scale"], rhs_bias=wl["rhs_bias"])
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    rows = np.random.default_rng(6).choice(m, 20, replace=False)
    ref, mag = _oracle(wl["lhs"], wl["rhs"], sizes, mx, rhs_scale=wl["rhs_scale"], bias=wl["rhs_bias"], rows=rows)
    check_close(out[torch.from_numpy(rows).to(DEV)], ref, mag, "MXFP8 decode workload")


# ------------------------------------------------------------------ NVFP4
def _nvfp4_scales(shape, seed):
    # positive e4m3 block scales spanning 2^-4 .. 2^4, one NaN-free code set
    return W.uniform(shape, 0.0625, 16.0, seed, DEV).to(torch.float8_e4m3fn)


def _oracle_fp4(lhs, rhs, sizes, bs, go=0, rhs_scale=None, bias=None, rows=None):
    return oracle.gmm(W.stored_bits(lhs), W.stored_bits(rhs), sizes, group_offset=go,
                      rhs_scale=None if rhs_scale is None else W.stored_bits(rhs_scale),
                      rhs_bias=None if bias is None else W.stored_bits(bias), rows=rows, rhs_dtype=oracle.E2M1,
                      rhs_block_scale=W.stored_bits(bs), rhs_block_scale_dtype=oracle.E4M3)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_scale", [False, True])
def test_nvfp4_matches_oracle(with_scale, out_dtype):
    m, k, n, L = 200, 512, 384, 6
    lhs = W.normal((m, k), 1.0, 101, DEV)
    rhs = W.weights("e2m1", (L, n, k), 102, DEV)
    bs = _nvfp4_scales((L, n, k // 16), 103)
    tensor_scale = W.uniform((L, 1, 1, n), 0.5, 2.0, 104, DEV) if with_scale else None
    bias = W.normal((L, 1, n), 1.0, 105, DEV)
    out = G.gmm(lhs, rhs, torch.tensor(SIZES, device=DEV), rhs_scale=tensor_scale, rhs_bias=bias,
                rhs_block_scale=bs, rhs_format="e2m1", out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle_fp4(lhs, rhs, SIZES, bs, rhs_scale=tensor_scale, bias=bias)
    check_close(out, ref, mag, f"NVFP4 (tensor scale {with_scale})")


def test_nvfp4_every_code_and_group_offset():
    # every e2m1 code in both nibbles of every weight row, exact integer-valued activations
    m, k, n, L, go = 64, 256, 128, 2, 1
    lhs = W.integer_valued((m, k), -4, 4, 111, DEV)
    codes = torch.arange(256, dtype=torch.int32, device=DEV).remainder(256).to(torch.uint8)
    rhs = codes.repeat(L * n * (k // 2) // 256).reshape(L, n, k // 2)
    bs = _nvfp4_scales((L, n, k // 16), 112)
    sizes = np.array([10, 30, 24], np.int32)
    out = G.gmm(lhs, rhs, torch.tensor(sizes, device=DEV), rhs_block_scale=bs, rhs_format="e2m1",
                group_offset=go, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle_fp4(lhs, rhs, sizes, bs, go=go)
    check_close(out, ref, mag, "NVFP4 every code")


def test_nvfp4_marked_rows_are_summed_again_with_their_block_scales():
    # activations whose 128-wide steps the fp16 split cannot hold (values below fp16's grid
    # under a large one, a NaN-free wide spread): those rows are marked and summed again from
    # the stored values, block scales included
    m, k, n, L = 24, 512, 256, 2
    x = W.normal((m, k), 1.0, 131).float()
    x[3, ::128] = 1.0
    x[3, 1::128] = 1.5 * 2.0 ** -40                               # below fp16's grid: marked
    x[5] = x[5] * torch.pow(2.0, torch.linspace(-40, 10, k))      # many binades per step
    x[7, ::128] = 3e4
    x[7, 5::128] = 2.0 ** -30
    lhs = x.to(torch.bfloat16).to(DEV)
    rhs = W.weights("e2m1", (L, n, k), 132, DEV)
    bs = _nvfp4_scales((L, n, k // 16), 133)
    sizes = np.array([10, 14], np.int32)
    out = G.gmm(lhs, rhs, torch.tensor(sizes, device=DEV), rhs_block_scale=bs, rhs_format="e2m1",
                out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = _oracle_fp4(lhs, rhs, sizes, bs)
    check_close(out, ref, mag, "NVFP4 with marked rows")


def test_nvfp4_decode_workload_sampled_rows():
    wl = W.fp8_decode(DEV, fmt="e2m1")
    sizes = wl["group_sizes"]
    m, k = wl["lhs"].shape
    L, n = wl["rhs"].shape[0], wl["rhs"].shape[1]
    bs = _nvfp4_scales((L, n, k // 16), 121)
    out = G.gmm(wl["lhs"], wl["rhs"], torch.tensor(sizes, device=DEV), rhs_block_scale=bs, rhs_format="e2m1",
                rhs_bias=wl["rhs_bias"])
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    rows = np.random.default_rng(7).choice(m, 20, replace=False)
    ref, mag = _oracle_fp4(wl["lhs"], wl["rhs"], sizes, bs, bias=wl["rhs_bias"], rows=rows)
    check_close(out[torch.from_numpy(rows).to(DEV)], ref, mag, "NVFP4 decode workload")
