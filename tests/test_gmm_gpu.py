"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Small cases compare every output element and span several 128x256 tiles with
ragged m, k and n tails, empty groups, sum(group_sizes) < m, many groups,
group_offset slices, bias, both weight layouts and both output dtypes.  Integer
inputs check indexing bit for bit (each row must use exactly its group's
expert)."""

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


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _gs(sizes):
    return torch.tensor(sizes, dtype=torch.int32, device=DEV)


def _gmm_case(m, k, n, sizes, *, transpose_rhs=True, out_dtype=torch.bfloat16, group_offset=0, local=None,
              bias_dtype=None, seed=0, wstd=0.05):
    sizes = np.asarray(sizes, np.int32)
    L = local if local is not None else sizes.size - group_offset
    lhs = W.normal((m, k), 1.0, seed + 1, DEV)
    shape = (L, n, k) if transpose_rhs else (L, k, n)
    rhs = W.normal(shape, wstd, seed + 2, DEV)
    bias = None if bias_dtype is None else W.normal((L, 1, n), 1.0, seed + 3, DEV, dtype=bias_dtype)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_bias=bias, transpose_rhs=transpose_rhs, group_offset=group_offset,
                out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(lhs, rhs, sizes, transpose_rhs=transpose_rhs, group_offset=group_offset, rhs_bias=bias)
    check_close(out, ref, mag, f"gmm m={m} k={k} n={n} sizes={sizes.tolist()}")
    return out


LAYOUTS = [pytest.param(True, id="NT"), pytest.param(False, id="NN")]
ODT = [pytest.param(torch.bfloat16, id="bf16out"), pytest.param(torch.float32, id="f32out")]
KERNELS = ["single", "pair", "swap", "swap_pair"]


@pytest.fixture(params=KERNELS)
def kernel(request, monkeypatch):
    """Runs the test once per bf16 forward kernel (options.bf16_kernel)."""
    use_options(monkeypatch, bf16_kernel=request.param)
    return request.param


@pytest.mark.parametrize("transpose_rhs", LAYOUTS)
@pytest.mark.parametrize("out_dtype", ODT)
def test_ragged_tiles_and_tails(transpose_rhs, out_dtype, kernel):
    # 5 groups (one empty, one of a single row), sum 588 < m = 700; k = 200 is
    # 3 full 64-wide steps plus 8; n = 520 is two 256-wide tiles plus 8.
    _gmm_case(700, 200, 520, [130, 0, 257, 1, 200], transpose_rhs=transpose_rhs, out_dtype=out_dtype)


@pytest.mark.parametrize("transpose_rhs", LAYOUTS)
def test_small_m_single_tile(transpose_rhs, kernel):
    _gmm_case(50, 64, 256, [20, 30], transpose_rhs=transpose_rhs, out_dtype=torch.float32)


@pytest.mark.parametrize("transpose_rhs", LAYOUTS)
def test_one_group_is_dense(transpose_rhs, kernel):
    _gmm_case(384, 512, 768, [384], transpose_rhs=transpose_rhs)


def test_all_groups_empty_gives_zeros(kernel):
    out = _gmm_case(300, 128, 256, [0, 0, 0])
    assert (out == 0).all()


def test_many_groups_multi_chunk_scan(kernel):
    rng = np.random.default_rng(3)
    sizes = rng.integers(0, 9, 300).astype(np.int32)
    sizes[rng.choice(300, 60, replace=False)] = 0
    _gmm_case(int(sizes.sum()) + 17, 128, 256, sizes, seed=5)


@pytest.mark.parametrize("go,local", [(0, 3), (2, 3), (3, 3), (5, 1)])
def test_group_offset_slices(go, local, kernel):
    _gmm_case(900, 192, 264, [150, 0, 333, 100, 7, 200], group_offset=go, local=local, seed=go)


@pytest.mark.parametrize("bias_dtype", [torch.bfloat16, torch.float32])
def test_bias(bias_dtype, kernel):
    _gmm_case(400, 128, 264, [100, 0, 250], bias_dtype=bias_dtype, out_dtype=torch.float32)


@pytest.mark.parametrize("transpose_rhs", LAYOUTS)
def test_integer_inputs_bit_exact(transpose_rhs, kernel):
    # Each group's expert is (g+1) * base: a row multiplied by the wrong expert
    # is off by an integer factor, and every sum is exact in fp32.
    m, k, n = 520, 256, 264
    sizes = np.array([129, 0, 127, 200, 1], np.int32)
    lhs = W.integer_valued((m, k), -8, 8, 11, DEV)
    base = W.integer_valued((n, k), -8, 8, 12, DEV, dtype=torch.float32)
    w_nk = torch.stack([(g + 1) * base for g in range(sizes.size)]).to(torch.bfloat16)
    rhs = w_nk if transpose_rhs else w_nk.transpose(1, 2).contiguous()
    out = G.gmm(lhs, rhs, _gs(sizes), transpose_rhs=transpose_rhs, out_dtype=torch.float32)
    ref, _ = oracle_gmm(lhs, rhs, sizes, transpose_rhs=transpose_rhs)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_nt_matches_nn_on_transposed_weight():
    m, k, n = 640, 320, 512
    sizes = np.array([100, 300, 0, 240], np.int32)
    lhs = W.normal((m, k), 1.0, 21, DEV)
    w = W.normal((4, n, k), 0.05, 22, DEV)
    nt = G.gmm(lhs, w, _gs(sizes), transpose_rhs=True, out_dtype=torch.float32)
    nn = G.gmm(lhs, w.transpose(1, 2).contiguous(), _gs(sizes), transpose_rhs=False, out_dtype=torch.float32)
    ref, mag = oracle_gmm(lhs, w, sizes)
    check_close(nt, ref, mag, "NT")
    check_close(nn, ref, mag, "NN")
    # both layouts feed the same products to the tensor core in the same k order
    assert torch.equal(nt, nn)


def test_device_error_flags_and_clamping(kernel):
    m, k, n = 256, 64, 256
    lhs = W.normal((m, k), 1.0, 31, DEV)
    rhs = W.normal((3, n, k), 0.05, 32, DEV)
    G.read_device_errors()
    sizes = np.array([100, -5, 400], np.int32)  # negative, and the sum runs past m
    out = G.gmm(lhs, rhs, _gs(sizes), out_dtype=torch.float32)
    flags = G.read_device_errors()
    assert flags == G.DEVERR_NEGATIVE_GROUP_SIZE | G.DEVERR_GROUP_SIZES_EXCEED_M
    ref, mag = oracle_gmm(lhs, rhs, sizes)
    check_close(out, ref, mag, "clamped sizes")
    assert G.read_device_errors() == 0  # flags were cleared by the read


def test_stream_ordering_on_side_stream():
    s = torch.cuda.Stream()
    m, k, n = 512, 128, 256
    sizes = np.array([200, 312], np.int32)
    lhs = W.normal((m, k), 1.0, 41, DEV)
    rhs = W.normal((2, n, k), 0.05, 42, DEV)
    gs = _gs(sizes)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = G.gmm(lhs, rhs, gs, out_dtype=torch.float32)
    s.synchronize()
    ref, mag = oracle_gmm(lhs, rhs, sizes)
    check_close(out, ref, mag, "side stream")


# ------------------------------------------------------------------------ tgmm
@pytest.fixture(params=["pair", "single"])
def tgmm_kernel(request, monkeypatch):
    """Runs the test on the one-SM tgmm kernel (default) and the SM-pair kernel (options.tgmm_kernel)."""
    use_options(monkeypatch, tgmm_kernel=request.param)
    return request.param


def _tgmm_case(m, k, n, sizes, out_dtype=torch.float32, seed=0):
    sizes = np.asarray(sizes, np.int32)
    lhs = W.normal((m, k), 1.0, seed + 1, DEV)
    dout = W.normal((m, n), 1.0, seed + 2, DEV)
    out = G.tgmm(lhs, dout, _gs(sizes), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_tgmm(lhs, dout, sizes)
    check_close(out, ref, mag, f"tgmm m={m} k={k} n={n} sizes={sizes.tolist()}")
    return out


@pytest.mark.parametrize("out_dtype", ODT)
def test_tgmm_ragged(out_dtype, tgmm_kernel):
    # group rows 100 (tail 36), 0, 333, 64 (exactly one chunk), 3; rows 500..599 unused
    _tgmm_case(600, 200, 264, [100, 0, 333, 64, 3], out_dtype=out_dtype)


def test_tgmm_group_edges_straddle_chunks(tgmm_kernel):
    _tgmm_case(1000, 128, 256, [65, 63, 1, 128, 129, 0, 614], seed=7)


def test_tgmm_all_empty_is_zero(tgmm_kernel):
    out = _tgmm_case(64, 128, 256, [0, 0])
    assert (out == 0).all()


def test_tgmm_sums_to_dense_when_groups_cover_all_rows(tgmm_kernel):
    m, k, n = 384, 128, 256
    sizes = np.array([100, 84, 200], np.int32)
    lhs = W.normal((m, k), 1.0, 51, DEV)
    dout = W.normal((m, n), 1.0, 52, DEV)
    out = G.tgmm(lhs, dout, _gs(sizes))
    dense = lhs.double().T @ dout.double()
    assert torch.allclose(out.double().sum(0), dense, rtol=1e-4, atol=1e-3)


def test_tgmm_pair_matches_single_sm_kernel(monkeypatch):
    # k = 392 (one full 256-wide pair tile, then 136: the second CTA holds 8 columns), n = 136
    sizes = np.array([130, 0, 1, 257, 64, 48], np.int32)
    lhs = W.normal((520, 392), 1.0, 61, DEV)
    dout = W.normal((520, 136), 1.0, 62, DEV)
    outs = {}
    for kern in ("pair", "single"):
        use_options(monkeypatch, tgmm_kernel=kern)
        outs[kern] = G.tgmm(lhs, dout, _gs(sizes))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_tgmm(lhs, dout, sizes)
    for kern, out in outs.items():
        check_close(out, ref, mag, f"tgmm {kern}")


# ------------------------------------------------ SM-pair kernel (>= 192 rows per group on average)
@pytest.mark.parametrize("transpose_rhs", LAYOUTS)
@pytest.mark.parametrize("out_dtype", ODT)
def test_pair_ragged_tiles_and_tails(transpose_rhs, out_dtype, monkeypatch):
    use_options(monkeypatch, bf16_kernel="pair")
    # 256-row pair tiles over groups of 300, 0, 513, 1, 400 rows (sum 1214 < m = 1500);
    # k = 200 and n = 520 leave tails in both dimensions.
    _gmm_case(1500, 200, 520, [300, 0, 513, 1, 400], transpose_rhs=transpose_rhs, out_dtype=out_dtype, seed=3)


@pytest.mark.parametrize("go,local", [(0, 3), (2, 3), (5, 1)])
def test_pair_group_offset_slices(go, local, monkeypatch):
    use_options(monkeypatch, bf16_kernel="pair")
    _gmm_case(1800, 192, 264, [250, 0, 333, 700, 7, 300], group_offset=go, local=local, seed=10 + go)


def test_pair_bias_and_single_group(monkeypatch):
    use_options(monkeypatch, bf16_kernel="pair")
    _gmm_case(1024, 256, 520, [1024], bias_dtype=torch.bfloat16, out_dtype=torch.float32, seed=17)


@pytest.mark.parametrize("transpose_rhs", LAYOUTS)
def test_pair_integer_inputs_bit_exact(transpose_rhs, monkeypatch):
    use_options(monkeypatch, bf16_kernel="pair")
    m, k, n = 1100, 256, 264
    sizes = np.array([257, 0, 255, 400, 1], np.int32)
    lhs = W.integer_valued((m, k), -8, 8, 13, DEV)
    base = W.integer_valued((n, k), -8, 8, 14, DEV, dtype=torch.float32)
    w_nk = torch.stack([(g + 1) * base for g in range(sizes.size)]).to(torch.bfloat16)
    rhs = w_nk if transpose_rhs else w_nk.transpose(1, 2).contiguous()
    out = G.gmm(lhs, rhs, _gs(sizes), transpose_rhs=transpose_rhs, out_dtype=torch.float32)
    ref, _ = oracle_gmm(lhs, rhs, sizes, transpose_rhs=transpose_rhs)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_three_kernels_agree_on_the_same_problem(monkeypatch):
    # The same rows and experts through each bf16 forward kernel: every result is
    # inside the bound, and the pair and single-SM kernels (same tile orientation,
    # same k order) agree bit for bit.
    m, k, n = 1536, 320, 512
    sizes = np.array([200, 340, 0, 300, 150, 0, 400, 146], np.int32)
    lhs = W.normal((m, k), 1.0, 21, DEV)
    w = W.normal((8, n, k), 0.05, 22, DEV)
    ref, mag = oracle_gmm(lhs, w, sizes)
    outs = {}
    for kern in KERNELS:
        use_options(monkeypatch, bf16_kernel=kern)
        outs[kern] = G.gmm(lhs, w, _gs(sizes), out_dtype=torch.float32)
        check_close(outs[kern], ref, mag, kern)
    assert torch.equal(outs["pair"], outs["single"])


def test_unknown_kernel_choice_is_rejected(monkeypatch):
    use_options(monkeypatch, bf16_kernel=9)
    lhs = W.normal((64, 64), 1.0, 1, DEV)
    w = W.normal((1, 64, 64), 0.05, 2, DEV)
    with pytest.raises(G.GmmError):
        G.gmm(lhs, w, _gs([64]))


# ------------------------------------------------------------------ the largest group count
def _max_groups_sizes(seed):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(0, 4, 1024).astype(np.int32)   # GMM_MAX_GROUPS groups, many empty
    return sizes


def test_max_groups_forward(kernel):
    sizes = _max_groups_sizes(31)
    _gmm_case(int(sizes.sum()) + 5, 128, 128, sizes, seed=31)


def test_max_groups_tgmm(tgmm_kernel):
    sizes = _max_groups_sizes(32)
    m = int(sizes.sum()) + 3
    lhs = W.normal((m, 128), 1.0, 33, DEV)
    dout = W.normal((m, 128), 1.0, 34, DEV)
    dw = G.tgmm(lhs, dout, _gs(sizes))
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_tgmm(lhs, dout, sizes)
    check_close(dw, ref, mag, "tgmm with 1024 groups")


def test_max_groups_fp8_weights():
    sizes = _max_groups_sizes(35)
    m = int(sizes.sum()) + 2
    lhs = W.normal((m, 128), 1.0, 36, DEV)
    rhs = W.weights("e4m3", (1024, 128, 128), 37, DEV)
    scale = W.uniform((1024, 1, 1, 128), 0.5 / 448, 2.0 / 448, 38, DEV)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(lhs, rhs, sizes, rhs_scale=scale)
    check_close(out, ref, mag, "fp8 weights with 1024 groups")
