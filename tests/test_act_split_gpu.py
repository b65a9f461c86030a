"""bf16 activations with 8- and 4-bit weights: the two-level e4m3 split of each
activation row, made once per row by a pass into the workspace (the default with a full
workspace) or inside the fp8 kernel for every weight tile (options act_split="kernel", or a
workspace of the minimum size).  Both feed the same operand rows and scales to the same MMAs
and fold, so their outputs must be the same bits.  They must also match the fp64 oracle,
with groups whose rows span two chunks, a ragged last k step, an n tail, a group_offset
slice, rows with infinities and NaN, and activations too large for the scratch."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import ORACLE_FORMAT, bits, check_close, use_options
from split_statement import split_statement, split_statement_f16

pytestmark = pytest.mark.gpu
DEV = "cuda"
FORMATS = ["e4m3", "e5m2", "e2m1", "int8", "int4", "uint4"]
# Groups of 0..40 rows: chunks of 8, 16 and 32 rows, two groups spanning two chunks.
SIZES = np.array([3, 0, 17, 1, 40, 0, 8, 16, 5, 33], np.int32)


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _inputs(fmt, m, k, n, L, nb, seed):
    lhs = W.normal((m, k), 1.0, seed, DEV)
    rhs = W.weights(fmt, (L, n, k), seed + 1, DEV)
    top = W.FORMAT_MAX[fmt]
    scale = W.uniform((L, nb, 1, n), 0.5 / top, 2.0 / top, seed + 2, DEV) if nb else None
    bias = W.normal((L, 1, n), 1.0, seed + 3, DEV)
    return lhs, rhs, scale, bias, ({"rhs_format": fmt} if fmt in W.PACKED else {})


def _both(monkeypatch, call):
    """The call's output with the split pass and with the in-kernel split."""
    use_options(monkeypatch, act_split="pass")
    pre = call()
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    use_options(monkeypatch, act_split="kernel")
    inside = call()
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    use_options(monkeypatch, act_split="auto")
    return pre, inside


# With bf16 activations the split pass feeds these formats to the fp16-MMA kernel (an fp16
# split, gemm_f16w.cu), the split inside the kernel to the e4m3 kernel: two exact methods whose
# fp32 sums may round differently, so both are held to the oracle instead of to each other.
F16_FORMATS = {"int8", "int4"}


def _modes_agree(fmt, pre, inside, ref, mag, what):
    if fmt in F16_FORMATS:
        check_close(inside, ref, mag, f"{what}, split inside the kernel")
    else:
        _same_bits(pre, inside)


def _same_bits(a, b):
    ia = a.view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.view(torch.int16 if b.element_size() == 2 else torch.int32)
    nan = torch.isnan(a)
    assert torch.equal(nan, torch.isnan(b)), "NaN positions differ"
    assert torch.equal(ia[~nan], ib[~nan]), f"{int((ia != ib).sum())} elements differ"


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16out", "f32out"])
@pytest.mark.parametrize("fmt", FORMATS)
def test_pass_equals_kernel_split_and_oracle(fmt, out_dtype, monkeypatch):
    # k = 640: two 256-wide steps and a 128-wide one; n = 392 ends 8 columns into a tile
    m, k, n, nb = int(SIZES.sum()) + 9, 640, 392, 5
    lhs, rhs, scale, bias, kw = _inputs(fmt, m, k, n, SIZES.size, nb, 80)
    gs = torch.tensor(SIZES, device=DEV)
    pre, inside = _both(monkeypatch, lambda: G.gmm(lhs, rhs, gs, rhs_scale=scale, rhs_bias=bias,
                                                   out_dtype=out_dtype, **kw))
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), SIZES, rhs_scale=bits(scale), rhs_bias=bits(bias),
                          rhs_dtype=ORACLE_FORMAT[fmt])
    check_close(pre, ref, mag, f"{fmt} split pass")
    _modes_agree(fmt, pre, inside, ref, mag, fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_group_offset_slice_without_scale(fmt, monkeypatch):
    sizes = np.array([5, 12, 0, 33, 7, 1, 20], np.int32)
    go, L = 2, 4
    m, k, n = int(sizes.sum()), 1024, 256
    lhs, rhs, _, bias, kw = _inputs(fmt, m, k, n, L, 0, 90)
    gs = torch.tensor(sizes, device=DEV)
    pre, inside = _both(monkeypatch, lambda: G.gmm(lhs, rhs, gs, rhs_bias=bias, group_offset=go,
                                                   out_dtype=torch.float32, **kw))
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, group_offset=go, rhs_bias=bits(bias),
                          rhs_dtype=ORACLE_FORMAT[fmt])
    check_close(pre, ref, mag, f"{fmt} go={go}")
    _modes_agree(fmt, pre, inside, ref, mag, f"{fmt} go={go}")


def test_wide_range_infinities_and_nan(monkeypatch):
    # rows whose steps span many binades (marked for the exact path), a row with an infinity
    # and a row with a NaN: both modes give the definition's infinities and NaNs
    sizes = np.array([6, 10], np.int32)
    m, k, n = 16, 512, 128
    x = W.normal((m, k), 1.0, 100)
    ramp = torch.pow(2.0, torch.linspace(-30, 20, k)).to(torch.bfloat16)
    x[1] = x[1] * ramp
    x[3, 17] = float("inf")
    x[12, 300] = float("nan")
    lhs = x.to(DEV)
    rhs = W.weights("e4m3", (2, n, k), 101, DEV)
    scale = W.uniform((2, 4, 1, n), 0.5 / 448, 2.0 / 448, 102, DEV)
    gs = torch.tensor(sizes, device=DEV)
    pre, inside = _both(monkeypatch, lambda: G.gmm(lhs, rhs, gs, rhs_scale=scale, out_dtype=torch.float32))
    _same_bits(pre, inside)
    assert torch.isnan(pre[12]).all() and torch.isinf(pre[3]).any()
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, rhs_scale=bits(scale), rhs_dtype=oracle.E4M3)
    check_close(pre, ref, mag, "wide range")


def test_minimum_workspace_splits_inside(monkeypatch):
    m, k, n = int(SIZES.sum()), 768, 256
    lhs, rhs, scale, bias, _ = _inputs("e4m3", m, k, n, SIZES.size, 3, 110)
    gs = torch.tensor(SIZES, device=DEV)
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)  # the error flags only
    full = G.gmm(lhs, rhs, gs, rhs_scale=scale, rhs_bias=bias, out_dtype=torch.float32)
    minimal = G.gmm(lhs, rhs, gs, rhs_scale=scale, rhs_bias=bias, out_dtype=torch.float32, workspace=small)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0 and G.read_device_errors(workspace=small) == 0
    _same_bits(full, minimal)
    use_options(monkeypatch, act_split="pass")
    with pytest.raises(G.GmmError):
        G.gmm(lhs, rhs, gs, rhs_scale=scale, workspace=small)


def test_activations_beyond_the_scratch_split_inside(monkeypatch):
    # 4 m k = 37.7 MB does not fit the 16 MiB scratch: auto falls back to the in-kernel split
    m, k, n = 2304, 4096, 128
    sizes = np.array([1000, 0, 1304], np.int32)
    lhs, rhs, scale, _, _ = _inputs("e4m3", m, k, n, 3, 32, 120)
    gs = torch.tensor(sizes, device=DEV)
    auto = G.gmm(lhs, rhs, gs, rhs_scale=scale, out_dtype=torch.float32)
    use_options(monkeypatch, act_split="kernel")
    inside = G.gmm(lhs, rhs, gs, rhs_scale=scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    _same_bits(auto, inside)
    use_options(monkeypatch, act_split="pass")
    with pytest.raises(G.GmmError):
        G.gmm(lhs, rhs, gs, rhs_scale=scale)
    rows = np.array([0, 999, 1000, 2303])
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, rhs_scale=bits(scale), rhs_dtype=oracle.E4M3, rows=rows)
    check_close(auto[torch.from_numpy(rows).to(DEV)], ref, mag, "beyond the scratch")


@pytest.mark.parametrize("go", [0, 32])
def test_decode_workload_both_modes(go, monkeypatch):
    fd = W.fp8_decode(torch.device(DEV))
    gs = torch.tensor(fd["group_sizes"], dtype=torch.int32, device=DEV)
    pre, inside = _both(monkeypatch, lambda: G.gmm(fd["lhs"], fd["rhs"][go:], gs, rhs_scale=fd["rhs_scale"][go:],
                                                   rhs_bias=fd["rhs_bias"][go:], group_offset=go))
    _same_bits(pre, inside)


@pytest.mark.parametrize("fmt,m,k", [("e4m3", 1, 128), ("int8", 1, 128), ("e2m1", 3, 384), ("int4", 9, 256),
                                     ("uint4", 40, 128)])
def test_smallest_shapes(fmt, m, k, monkeypatch):
    # one row; a single 128-wide step (half of a 256-wide one); int8's 128-wide steps
    sizes = np.array([m], np.int32)
    lhs, rhs, scale, bias, kw = _inputs(fmt, m, k, 128, 1, 1, 140)
    gs = torch.tensor(sizes, device=DEV)
    pre, inside = _both(monkeypatch, lambda: G.gmm(lhs, rhs, gs, rhs_scale=scale, rhs_bias=bias,
                                                   out_dtype=torch.float32, **kw))
    ref, mag = oracle.gmm(bits(lhs), bits(rhs), sizes, rhs_scale=bits(scale), rhs_bias=bits(bias),
                          rhs_dtype=ORACLE_FORMAT[fmt])
    check_close(pre, ref, mag, f"{fmt} m={m} k={k}")
    _modes_agree(fmt, pre, inside, ref, mag, f"{fmt} m={m} k={k}")


@pytest.mark.parametrize("m,fits", [(2032, True), (2040, False)])
def test_scratch_boundary(m, fits, monkeypatch):
    # k = 2048: the split rows take 4 m k bytes, then 256-aligned step scales (m * 8 * 2 * 4):
    # 2032 rows fill the 16 MiB scratch but for its last 1 KB, 2040 rows do not fit
    k, n = 2048, 128
    sizes = np.array([m // 2, 0, m - m // 2], np.int32)
    lhs, rhs, scale, _, _ = _inputs("e4m3", m, k, n, 3, 16, 150)
    gs = torch.tensor(sizes, device=DEV)
    use_options(monkeypatch, act_split="pass")
    if not fits:
        with pytest.raises(G.GmmError):
            G.gmm(lhs, rhs, gs, rhs_scale=scale)
        return
    pre = G.gmm(lhs, rhs, gs, rhs_scale=scale, out_dtype=torch.float32)
    use_options(monkeypatch, act_split="kernel")
    inside = G.gmm(lhs, rhs, gs, rhs_scale=scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    _same_bits(pre, inside)


def test_two_streams_at_once_keep_their_own_split_rows():
    # calls on two streams may overlap; each stream's default workspace holds its own split rows
    sizes = np.array([30, 0, 41, 57], np.int32)
    m, k, n = int(sizes.sum()), 2048, 512
    a = _inputs("e4m3", m, k, n, 4, 4, 160)
    b = _inputs("e4m3", m, k, n, 4, 4, 170)
    gs = torch.tensor(sizes, device=DEV)
    call = lambda t: G.gmm(t[0], t[1], gs, rhs_scale=t[2], rhs_bias=t[3], out_dtype=torch.float32)
    ref_a, ref_b = call(a), call(b)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(4):
        with torch.cuda.stream(s1):
            oa = call(a)
        with torch.cuda.stream(s2):
            ob = call(b)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    assert G.read_device_errors(stream=s1) == 0 and G.read_device_errors(stream=s2) == 0
    for oa, ob in outs:
        _same_bits(oa, ref_a)
        _same_bits(ob, ref_b)


@pytest.mark.parametrize("fmt", ["e4m3", "int4"])
def test_captured_graph_replays_with_new_activations(fmt):
    # the split pass and the matmul (its programmatic dependent) captured in one CUDA graph,
    # replayed with new activations and group sizes copied into the captured buffers
    sizes1 = np.array([7, 0, 19, 33, 4], np.int32)
    sizes2 = np.array([0, 30, 1, 8, 24], np.int32)
    m, k, n = 63, 1024, 384
    lhs, rhs, scale, bias, kw = _inputs(fmt, m, k, n, 5, 4, 180)
    lhs1, lhs2 = lhs.clone(), W.normal((m, k), 1.0, 185, DEV)
    gs = torch.tensor(sizes1, device=DEV)
    out = torch.empty((m, n), dtype=torch.float32, device=DEV)
    call = lambda: G.gmm(lhs, rhs, gs, rhs_scale=scale, rhs_bias=bias, out=out, **kw)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # the stream's workspace and the kernels' attributes set up
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for x, sizes in ((lhs2, sizes2), (lhs1, sizes1)):
        ref = G.gmm(x, rhs, torch.tensor(sizes, device=DEV), rhs_scale=scale, rhs_bias=bias,
                    out_dtype=torch.float32, **kw)
        lhs.copy_(x)
        gs.copy_(torch.from_numpy(sizes))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert G.read_device_errors(stream=s) == 0
        _same_bits(out, ref)


def _hard_split_rows(m, k):
    x = W.normal((m, k), 1.0, 190).float()
    x[1] = 0.0                                                   # a zero row: e clamps
    x[2] = -0.0                                                  # negative zeros
    x[3] = x[3] * 1e-30                                          # tiny values
    x[4] = x[4] * torch.pow(2.0, torch.linspace(-30, 20, k))     # many binades per step
    x[5, :8] = torch.tensor([128.0, 1.0625, 1.1875, -1.0625, 3.0, 0.0078125, -0.0, 2.0 ** -20])  # ties
    x[6] = x[6] * 3e4                                            # large values
    x[7, 1:] = 3 * 2.0 ** -22                                    # one large value, small ones
    x[7, 0] = x[7, 128] = x[7, 256] = x[7, 384] = x[7, 512] = 1.0
    x[8] = torch.where(torch.arange(k) % 2 == 0, 1.5 * 2.0 ** -30, 1.25 * 2.0 ** -60)  # marked steps
    x[8, ::128] = 1.0
    x[9, ::128] = 1.0                                            # fp16 subnormals: held to 2^-24 sc
    x[9, 1::128] = 2.0 ** -33
    x[10, ::128] = 1.0                                           # below fp16's grid: marked
    x[10, 1::128] = 1.5 * 2.0 ** -40
    return x.to(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("fmt,step", [("e4m3", 256)])
def test_split_rows_equal_a_host_statement_of_the_split(fmt, step):
    # the pass's h / l / h2 / l2 planes and (s1, s2) step scales, read back from the workspace,
    # bit for bit
    m, k, n = 37, 640, 128
    x = W.normal((m, k), 1.0, 190).float()
    x[1] = 0.0                                                   # a zero row: e clamps to 8
    x[2] = -0.0                                                  # negative zeros
    x[3] = x[3] * 1e-30                                          # tiny values
    x[4] = x[4] * torch.pow(2.0, torch.linspace(-30, 20, k))     # many binades per step
    x[5, :8] = torch.tensor([128.0, 1.0625, 1.1875, -1.0625, 3.0, 0.0078125, -0.0, 2.0 ** -20])  # ties
    x[6] = x[6] * 3e4                                            # large values
    x[7, 1:] = 3 * 2.0 ** -22                                    # one large value, small ones
    x[7, 0] = x[7, 128] = x[7, 256] = x[7, 384] = x[7, 512] = 1.0
    x[8] = torch.where(torch.arange(k) % 2 == 0, 1.5 * 2.0 ** -30, 1.25 * 2.0 ** -60)  # marked steps
    x[8, ::128] = 1.0
    lhs = x.to(torch.bfloat16).to(DEV)
    rhs = W.weights(fmt, (1, n, k), 191, DEV)
    G.gmm(lhs, rhs, torch.tensor([m], dtype=torch.int32, device=DEV), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ws = G.workspace_for(torch.device(DEV))
    ksteps = -(-k // step)
    planes = ws[256:256 + 4 * m * k].cpu().numpy().reshape(4, m, k)
    at = (256 + 4 * m * k + 255) // 256 * 256
    scales = ws[at:at + 8 * m * ksteps].cpu().numpy().view(np.float32).reshape(m, ksteps, 2)
    want_planes, want_scales = split_statement(bits(lhs), step)
    assert np.signbit(want_scales[8, :, 1]).all() and not np.signbit(want_scales[7, :, 1]).any()
    bad = np.argwhere(planes != want_planes)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"
    assert np.array_equal(scales.view(np.uint32), want_scales.view(np.uint32))


def test_unknown_setting_is_rejected(monkeypatch):
    lhs, rhs, scale, _, _ = _inputs("e4m3", 16, 256, 128, 1, 1, 130)
    use_options(monkeypatch, act_split=5)
    with pytest.raises(G.GmmError):
        G.gmm(lhs, rhs, torch.tensor([16], dtype=torch.int32, device=DEV), rhs_scale=scale)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_fp16_split_rows_equal_a_host_statement(fmt):
    # the integer formats' split pass: fp16 values (each 8 k reordered for 4-bit weights) and
    # (scale, mark) per 128-wide step, read back from the workspace, bit for bit
    m, k, n = 37, 640, 128
    lhs = _hard_split_rows(m, k)
    rhs = W.weights(fmt, (1, n, k), 191, DEV)
    kw = {"rhs_format": fmt} if fmt in W.PACKED else {}
    G.gmm(lhs, rhs, torch.tensor([m], dtype=torch.int32, device=DEV), out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ws = G.workspace_for(torch.device(DEV))
    ksteps = k // 128
    plane = ws[256:256 + 2 * m * k].cpu().numpy().view(np.uint16).reshape(m, k)
    at = (256 + 2 * m * k + 255) // 256 * 256
    scales = ws[at:at + 8 * m * ksteps].cpu().numpy().view(np.float32).reshape(m, ksteps, 2)
    want_plane, want_scales = split_statement_f16(bits(lhs), fmt != "int8")
    assert np.signbit(want_scales[10, :, 1]).all() and not np.signbit(want_scales[9, :, 1]).any()
    assert np.signbit(want_scales[8, :, 1]).all() and not np.signbit(want_scales[7, :, 1]).any()
    bad = np.argwhere(plane != want_plane)
    assert bad.size == 0, f"{len(bad)} values differ, first at {bad[:3].tolist()}"
    assert np.array_equal(scales.view(np.uint32), want_scales.view(np.uint32))
