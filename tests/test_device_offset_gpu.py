"""gmm with group_offset held in device memory (page "tpu-inference ...", gmm.py: group_offset
is a ()-shaped int32 device array): the kernels read it when they run, so the result must equal
the host-offset call bit for bit on every kernel, an out-of-range value must be flagged with
nothing written, and one captured CUDA graph must serve several offsets."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, oracle_gmm, use_options

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16_KERNELS = ["single", "pair", "swap", "swap_pair"]


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _gs(sizes):
    return torch.tensor(np.asarray(sizes, np.int32), dtype=torch.int32, device=DEV)


def _dev_offset(go):
    return torch.tensor([go], dtype=torch.int32, device=DEV)


SIZES = [60, 0, 130, 7, 200, 33, 90]  # 7 groups, sum 520


@pytest.mark.parametrize("kernel", BF16_KERNELS)
@pytest.mark.parametrize("go,L", [(0, 3), (2, 4), (4, 3)])
def test_bf16_device_offset_equals_host_offset(kernel, go, L, monkeypatch):
    use_options(monkeypatch, bf16_kernel=kernel)
    m, k, n = 560, 192, 264
    lhs = W.normal((m, k), 1.0, 1, DEV)
    rhs = W.normal((L, n, k), 0.05, 2, DEV)
    bias = W.normal((L, 1, n), 1.0, 3, DEV)
    host = G.gmm(lhs, rhs, _gs(SIZES), rhs_bias=bias, group_offset=go, out_dtype=torch.float32)
    dev = G.gmm(lhs, rhs, _gs(SIZES), rhs_bias=bias, group_offset=_dev_offset(go), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    assert torch.equal(host, dev)
    ref, mag = oracle_gmm(lhs, rhs, np.asarray(SIZES, np.int32), group_offset=go, rhs_bias=bias)
    check_close(dev, ref, mag, f"device offset {go} ({kernel})")


@pytest.mark.parametrize("fmt", ["e4m3", "int4"])
def test_fp8_device_offset_equals_host_offset(fmt):
    m, k, n, L, go = 140, 256, 256, 4, 3
    sizes = [3, 0, 17, 1, 40, 0, 8, 16, 5, 33]
    lhs = W.normal((m, k), 1.0, 4, DEV)
    rhs = W.weights(fmt, (L, n, k), 5, DEV)
    scale = W.uniform((L, 2, 1, n), 0.5 / 448, 2.0 / 448, 6, DEV)
    kw = {"rhs_format": fmt} if fmt in W.PACKED else {}
    host = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, group_offset=go, **kw)
    dev = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, group_offset=_dev_offset(go), **kw)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    assert torch.equal(host, dev)


def test_device_offset_with_kept_rows():
    m, k, n, L, go = 560, 128, 256, 3, 2
    lhs = W.normal((m, k), 1.0, 7, DEV)
    rhs = W.normal((L, n, k), 0.05, 8, DEV)
    out = W.normal((m, n), 3.0, 9, DEV) + 100.0
    before = out.clone()
    expect = G.gmm_into(lhs, rhs, _gs(SIZES), before.clone(), group_offset=go)
    G.gmm_into(lhs, rhs, _gs(SIZES), out, group_offset=_dev_offset(go))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    assert torch.equal(out, expect)


@pytest.mark.parametrize("kernel", BF16_KERNELS + ["fp8"])
@pytest.mark.parametrize("bad", [-1, 5])
def test_out_of_range_device_offset_is_flagged_and_writes_nothing(kernel, bad, monkeypatch):
    # 7 groups, 3 local: valid offsets are 0..4
    m, k, n, L = 560, 256, 256, 3
    lhs = W.normal((m, k), 1.0, 10, DEV)
    if kernel == "fp8":
        rhs = W.weights("e4m3", (L, n, k), 11, DEV)
    else:
        use_options(monkeypatch, bf16_kernel=kernel)
        rhs = W.normal((L, n, k), 0.05, 11, DEV)
    out = torch.full((m, n), 7.0, dtype=torch.bfloat16, device=DEV)
    G.gmm(lhs, rhs, _gs(SIZES), group_offset=_dev_offset(bad), out=out)
    torch.cuda.synchronize()
    assert G.read_device_errors() == G.DEVERR_GROUP_OFFSET
    assert (out == 7.0).all()


def test_one_cuda_graph_serves_several_offsets():
    m, k, n, L = 560, 256, 512, 3
    lhs = W.normal((m, k), 1.0, 12, DEV)
    rhs = W.normal((L, n, k), 0.05, 13, DEV)
    gs = _gs(SIZES)
    offset = _dev_offset(0)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # library, the stream's workspace and kernel attributes set up
        G.gmm(lhs, rhs, gs, group_offset=offset, out=out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        G.gmm(lhs, rhs, gs, group_offset=offset, out=out)
    for go in (0, 4, 2):
        offset.fill_(go)
        graph.replay()
        torch.cuda.synchronize()
        assert G.read_device_errors(stream=s) == 0
        assert torch.equal(out, G.gmm(lhs, rhs, gs, group_offset=go)), f"replay with offset {go}"
