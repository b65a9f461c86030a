"""GPU parity for the two calls that work on one shard's slice of the experts.

gmm_into (page "tpu-inference ...", gmm.py: existing_out, aliased to the output):
rows of the local groups must equal the oracle's result for that slice, and every
other row must keep, bit for bit, what the caller put in the buffer.  Two shards
with disjoint slices writing into one buffer must give the full grouped matmul.

tgmm_local (gmm.py make_group_metadata: start_group / num_nonzero_groups, with
empty groups visited): out[l] must equal the oracle's tgmm for group
group_offset + l, whose rows come from the prefix sum over all groups."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, oracle_gmm, oracle_tgmm, use_options

pytestmark = pytest.mark.gpu
DEV = "cuda"
KERNELS = ["single", "pair", "swap", "swap_pair"]


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _gs(sizes):
    return torch.tensor(np.asarray(sizes, np.int32), dtype=torch.int32, device=DEV)


def _local_rows(sizes, go, L, m):
    offs = np.concatenate([[0], np.cumsum(np.maximum(sizes, 0))])
    lo, hi = min(int(offs[go]), m), min(int(offs[go + L]), m)
    mask = np.zeros(m, bool)
    mask[lo:hi] = True
    return mask


def _seeded_out(m, n, dtype, seed):
    # A recognisable fill (no zeros, so an unwanted zeroing pass shows).
    return W.normal((m, n), 3.0, seed, DEV, dtype=dtype) + 100.0


def _check_into(out, before, ref, mag, mask, what):
    keep = ~mask
    assert torch.equal(out[torch.from_numpy(keep).to(DEV)], before[torch.from_numpy(keep).to(DEV)]), \
        f"{what}: rows outside the local groups changed"
    check_close(out[torch.from_numpy(mask).to(DEV)], ref[mask], mag[mask], what)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("transpose_rhs", [True, False], ids=["NT", "NN"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16out", "f32out"])
def test_gmm_into_keeps_rows_outside_the_slice(kernel, transpose_rhs, out_dtype, monkeypatch):
    use_options(monkeypatch, bf16_kernel=kernel)
    # 7 groups, slice [2, 5) holds an empty group and a one-row group; sum 603 < m = 650.
    m, k, n = 650, 136, 264
    sizes = np.array([100, 37, 0, 1, 250, 120, 95], np.int32)
    go, L = 2, 3
    lhs = W.normal((m, k), 1.0, 11, DEV)
    shape = (L, n, k) if transpose_rhs else (L, k, n)
    rhs = W.normal(shape, 0.05, 12, DEV)
    bias = W.normal((L, 1, n), 1.0, 13, DEV)
    out = _seeded_out(m, n, out_dtype, 14)
    before = out.clone()
    res = G.gmm_into(lhs, rhs, _gs(sizes), out, rhs_bias=bias, transpose_rhs=transpose_rhs, group_offset=go)
    torch.cuda.synchronize()
    assert res.data_ptr() == out.data_ptr()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(lhs, rhs, sizes, transpose_rhs=transpose_rhs, group_offset=go, rhs_bias=bias)
    _check_into(out, before, ref, mag, _local_rows(sizes, go, L, m), f"gmm_into {kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_two_shards_into_one_buffer_make_the_full_product(kernel, monkeypatch):
    use_options(monkeypatch, bf16_kernel=kernel)
    m, k, n = 520, 128, 256
    sizes = np.array([90, 0, 130, 64, 1, 200], np.int32)  # sum 485 < m
    rhs_all = W.normal((6, n, k), 0.05, 22, DEV)
    lhs = W.normal((m, k), 1.0, 21, DEV)
    out = torch.zeros((m, n), dtype=torch.float32, device=DEV)
    for go, L in ((0, 3), (3, 3)):
        G.gmm_into(lhs, rhs_all[go:go + L].contiguous(), _gs(sizes), out, group_offset=go)
    torch.cuda.synchronize()
    ref, mag = oracle_gmm(lhs, rhs_all, sizes)
    check_close(out, ref, mag, f"two shards via gmm_into {kernel}")


@pytest.mark.parametrize("e4m3", [True, False], ids=["e4m3", "bf16w"])
def test_gmm_into_block_scaled_path(e4m3):
    m, k, n, nb = 70, 256, 264, 2
    sizes = np.array([5, 9, 0, 17, 3, 30], np.int32)  # sum 64 < m
    go, L = 1, 4
    lhs = W.normal((m, k), 1.0, 31, DEV)
    rhs = W.e4m3_normal((L, n, k), 32, DEV) if e4m3 else W.normal((L, n, k), 0.05, 32, DEV)
    scale = W.uniform((L, nb, 1, n), 0.5 / 448, 2.0 / 448, 33, DEV)
    bias = W.normal((L, 1, n), 1.0, 34, DEV, dtype=torch.float32)
    out = _seeded_out(m, n, torch.bfloat16, 35)
    before = out.clone()
    G.gmm_into(lhs, rhs, _gs(sizes), out, rhs_scale=scale, rhs_bias=bias, group_offset=go)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(lhs, rhs, sizes, group_offset=go, rhs_scale=scale, rhs_bias=bias)
    _check_into(out, before, ref, mag, _local_rows(sizes, go, L, m), "gmm_into scaled")


def test_gmm_into_matches_gmm_on_local_rows():
    # Same kernels, same rounding: the local rows agree bit for bit with gmm().
    m, k, n = 300, 192, 256
    sizes = np.array([40, 80, 60, 70], np.int32)
    lhs = W.normal((m, k), 1.0, 41, DEV)
    rhs = W.normal((2, n, k), 0.05, 42, DEV)
    full = G.gmm(lhs, rhs, _gs(sizes), group_offset=1)
    out = _seeded_out(m, n, torch.bfloat16, 43)
    G.gmm_into(lhs, rhs, _gs(sizes), out, group_offset=1)
    torch.cuda.synchronize()
    rows = torch.from_numpy(_local_rows(sizes, 1, 2, m)).to(DEV)
    assert torch.equal(out[rows], full[rows])
    assert (full[~rows] == 0).all()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32out", "bf16out"])
@pytest.mark.parametrize("go,L", [(0, 3), (2, 4), (5, 1), (0, 7)])
def test_tgmm_local_is_the_slice_of_tgmm(go, L, out_dtype):
    # Groups with 0, 1 and ragged row counts; sum 541 < m = 560; k and n with tails.
    m, k, n = 560, 200, 264
    sizes = np.array([130, 0, 1, 200, 64, 0, 146], np.int32)
    lhs = W.normal((m, k), 1.0, 51, DEV)
    dout = W.normal((m, n), 1.0, 52, DEV)
    out = G.tgmm_local(lhs, dout, _gs(sizes), group_offset=go, num_local_groups=L, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (L, k, n)
    assert G.read_device_errors() == 0
    ref, mag = oracle_tgmm(lhs, dout, sizes)
    check_close(out, ref[go:go + L], mag[go:go + L], f"tgmm_local go={go} L={L}")


def test_tgmm_local_shards_concatenate_to_tgmm():
    m, k, n = 1100, 128, 256
    sizes = np.array([300, 0, 250, 1, 400, 149], np.int32)
    lhs = W.normal((m, k), 1.0, 61, DEV)
    dout = W.normal((m, n), 1.0, 62, DEV)
    full = G.tgmm(lhs, dout, _gs(sizes))
    parts = [G.tgmm_local(lhs, dout, _gs(sizes), group_offset=go, num_local_groups=L) for go, L in ((0, 2), (2, 4))]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts), full)
