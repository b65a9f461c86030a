"""Shapes of the 8- and 4-bit weight kernel at the edges of its schedule: fewer items than CTAs,
one item per CTA over a long k (64 or 128 steps), item counts just above the CTA count, ragged
chunks with quant blocks wider than a step (a step's weight scales from one block, or from two
when a step straddles a block boundary), and e4m3 activations in 32-row chunks.  Each result is
checked against the fp64 oracle, and the split pass against the in-kernel split (same bits where
both run the e4m3 kernel; int8 runs on the fp16-MMA kernel after the pass)."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import ORACLE_FORMAT, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _problem(fmt, sizes, k, n, nb, seed):
    sizes = np.asarray(sizes, np.int32)
    m = int(sizes.sum())
    lhs = W.normal((m, k), 1.0, seed, DEV)
    rhs = W.weights(fmt, (sizes.size, n, k), seed + 1, DEV)
    top = W.FORMAT_MAX[fmt]
    scale = W.uniform((sizes.size, nb, 1, n), 0.5 / top, 2.0 / top, seed + 2, DEV)
    bias = W.normal((sizes.size, 1, n), 1.0, seed + 3, DEV)
    kw = {"rhs_format": fmt} if fmt in W.PACKED else {}
    return sizes, lhs, rhs, scale, bias, kw


def _check(out, sizes, lhs, rhs, scale, bias, fmt, what):
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, rhs_scale=bits(scale), rhs_bias=bits(bias),
                          rhs_dtype=ORACLE_FORMAT[fmt])
    check_close(out, ref, mag, what)


@pytest.mark.parametrize("fmt", ["e4m3", "int8", "e2m1"])
@pytest.mark.parametrize("sizes,k,n,nb", [
    ([3], 256, 128, 2),                 # one item of one or two steps
    ([9, 0, 7], 16384, 128, 16),        # two items of 64 (128) steps, blocks of 1024 k
    ([16] * 80, 1024, 256, 4),          # 160 items of 4 (8) steps: just above the CTA count
    ([5, 40, 1, 0, 77, 16], 1536, 384, 3),  # ragged chunks, 6 (12) steps, blocks of 512 k
    ([7, 20], 1152, 256, 3),            # blocks of 384 k: a 256-wide step straddles two
])
def test_edge_shapes_match_the_oracle(fmt, sizes, k, n, nb):
    sizes, lhs, rhs, scale, bias, kw = _problem(fmt, sizes, k, n, nb, 200)
    gs = torch.tensor(sizes, device=DEV)
    call = lambda: G.gmm(lhs, rhs, gs, rhs_scale=scale, rhs_bias=bias, out_dtype=torch.float32, **kw)
    with G.options(act_split="pass"):
        pre = call()
    with G.options(act_split="kernel"):
        inside = call()
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    _check(pre, sizes, lhs, rhs, scale, bias, fmt, f"{fmt} sizes={sizes.tolist()} k={k}")
    if fmt == "int8":
        # the split pass feeds int8 to the fp16-MMA kernel, the in-kernel split to the e4m3 one
        _check(inside, sizes, lhs, rhs, scale, bias, fmt, f"{fmt} sizes={sizes.tolist()} k={k}, split inside")
    else:
        assert torch.equal(pre, inside)


def test_e4m3_activations_in_32_row_chunks():
    # W8A8: e4m3 rows with per-token-group scales, 32-row chunks
    sizes = np.array([40, 3, 0, 25], np.int32)
    m, k, n = int(sizes.sum()), 2048, 256
    x = W.normal((m, k), 1.0, 400, DEV)
    q, a_scale = G.quantize_e4m3(x)
    rhs = W.weights("e4m3", (4, n, k), 401, DEV)
    scale = W.uniform((4, 4, 1, n), 0.5 / 448, 2.0 / 448, 402, DEV)
    out = G.gmm(q, rhs, torch.tensor(sizes, device=DEV), rhs_scale=scale, lhs_scale=a_scale,
                out_dtype=torch.float32)
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)  # the error flags alone
    minimal = G.gmm(q, rhs, torch.tensor(sizes, device=DEV), rhs_scale=scale, lhs_scale=a_scale,
                    out_dtype=torch.float32, workspace=small)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0 and G.read_device_errors(workspace=small) == 0
    assert torch.equal(out, minimal)
    ref, mag = oracle.gmm(bits(q), bits(rhs), sizes, rhs_scale=bits(scale), lhs_scale=bits(a_scale),
                          lhs_dtype=oracle.E4M3, rhs_dtype=oracle.E4M3)
    check_close(out, ref, mag, "W8A8, 32-row chunks")


@pytest.mark.parametrize("n", [384, 392])
def test_e8m0_weight_scales(n):
    # E8M0 scale rows of n bytes: copied in bulk when n % 16 == 0, else loaded by the warp
    sizes = np.array([9, 0, 30], np.int32)
    m, k = int(sizes.sum()), 1024
    lhs = W.normal((m, k), 1.0, 500, DEV)
    rhs = W.weights("e4m3", (3, n, k), 501, DEV)
    e8 = torch.randint(118, 126, (3, 8, 1, n), dtype=torch.uint8, device=DEV,
                       generator=torch.Generator(device=DEV).manual_seed(502))
    bias = W.normal((3, 1, n), 1.0, 503, DEV)
    gs = torch.tensor(sizes, device=DEV)
    call = lambda: G.gmm(lhs, rhs, gs, rhs_scale=e8, rhs_bias=bias, out_dtype=torch.float32)
    with G.options(act_split="pass"):
        pre = call()
    with G.options(act_split="kernel"):
        inside = call()
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    assert torch.equal(pre, inside)
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, rhs_scale=bits(e8), rhs_bias=bits(bias),
                          rhs_dtype=oracle.E4M3)
    check_close(pre, ref, mag, f"E8M0 scales, n={n}")
