"""Full-size parity at the workloads' real shapes, in the launch configuration bench.py
times.  The oracle checks every element of the tiny workload and a seeded sample of up to
256 rows per group (plus each group's first and last row) of the large ones; tgmm is
checked on 256 seeded k-rows of every group's [k, n] block."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, oracle_gmm, oracle_tgmm

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _gs(sizes):
    return torch.tensor(np.asarray(sizes, np.int32), dtype=torch.int32, device=DEV)


def _sampled_check(out, lhs, rhs, sizes, what, transpose_rhs=True, seed=0):
    offs = oracle.group_offsets(sizes, lhs.shape[0])
    rows = W.sample_rows(seed, offs, 256)
    tail = np.arange(int(offs[-1]), lhs.shape[0])[:64]  # rows past sum(group_sizes), if any
    rows = np.concatenate([rows, tail]).astype(np.int64)
    ref, mag = oracle_gmm(lhs, rhs, sizes, transpose_rhs=transpose_rhs, rows=rows)
    check_close(out[torch.from_numpy(rows).to(out.device)], ref, mag, what)


def test_tiny_full_compare():
    d = W.tiny(DEV)
    out = G.gmm(d["lhs"], d["rhs"], _gs(d["group_sizes"]), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (d["group_sizes"] == 0).sum() == 1
    ref, mag = oracle_gmm(d["lhs"], d["rhs"], d["group_sizes"])
    check_close(out, ref, mag, "tiny")


def test_mixtral_up_sampled():
    d = W.mixtral_up(DEV)
    out = G.gmm(d["lhs"], d["rhs"], _gs(d["group_sizes"]))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    _sampled_check(out, d["lhs"], d["rhs"], d["group_sizes"], "mixtral_up", seed=1)


@pytest.fixture(scope="module")
def moe():
    return W.moe128(DEV)


def test_moe128_routing_shape(moe):
    sizes = moe["group_sizes"]
    assert sizes.sum() == 32768 and (sizes == 0).sum() == 10


def test_moe128_wi_nt_sampled(moe):
    out = G.gmm(moe["lhs"], moe["wi"], _gs(moe["group_sizes"]))
    torch.cuda.synchronize()
    _sampled_check(out, moe["lhs"], moe["wi"], moe["group_sizes"], "wi NT", seed=2)


def test_moe128_wo_nt_sampled(moe):
    # wo read as [G, n=2048, k=1024] on its own 1024-wide input
    out = G.gmm(moe["lhs_wo"], moe["wo"], _gs(moe["group_sizes"]))
    torch.cuda.synchronize()
    _sampled_check(out, moe["lhs_wo"], moe["wo"], moe["group_sizes"], "wo NT", seed=3)


def test_moe128_wo_nn_sampled(moe):
    # wo read as [G, k=2048, n=1024] on the shared 2048-wide input
    out = G.gmm(moe["lhs"], moe["wo"], _gs(moe["group_sizes"]), transpose_rhs=False)
    torch.cuda.synchronize()
    _sampled_check(out, moe["lhs"], moe["wo"], moe["group_sizes"], "wo NN", transpose_rhs=False, seed=4)


def test_moe128_dlhs_nt_matches_nn_on_transposed_weight(moe):
    gs = _gs(moe["group_sizes"])
    nt = G.gmm(moe["dout"], moe["wi"], gs)
    wt = moe["wi"].transpose(1, 2).contiguous()
    nn = G.gmm(moe["dout"], wt, gs, transpose_rhs=False)
    torch.cuda.synchronize()
    del wt
    assert torch.equal(nt, nn)
    _sampled_check(nt, moe["dout"], moe["wi"], moe["group_sizes"], "dlhs NT", seed=5)


def test_moe128_tgmm_sampled(moe):
    dw = G.tgmm(moe["lhs"], moe["dout"], _gs(moe["group_sizes"]))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    rng = np.random.Generator(np.random.PCG64(6))
    k_rows = np.sort(rng.choice(2048, 256, replace=False)).astype(np.int64)
    ref, mag = oracle_tgmm(moe["lhs"], moe["dout"], moe["group_sizes"], k_rows=k_rows)
    check_close(dw[:, torch.from_numpy(k_rows).to(DEV)], ref, mag, "tgmm")
    empty = np.flatnonzero(moe["group_sizes"] == 0)
    assert (dw[torch.from_numpy(empty).to(DEV)] == 0).all()
