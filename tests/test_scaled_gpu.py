"""GPU parity for the block-scaled path (e4m3 or bf16 weights with per-(group, k-block, n)
fp32 scale and bias) against the fp64 oracle, including every e4m3fn code decoded by the
kernel itself."""

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


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


@pytest.fixture(autouse=True, params=["tensor", "decode"])
def e4m3_kernel(request, monkeypatch):
    """Every test runs on both e4m3 kernels: the e4m3 tensor-core kernel (default) and the
    kernel that decodes the weights to bf16 (options.e4m3_kernel = "decode")."""
    use_options(monkeypatch, e4m3_kernel=request.param)
    return request.param


def _gs(sizes):
    return torch.tensor(np.asarray(sizes, np.int32), dtype=torch.int32, device=DEV)


def _codes_to_e4m3(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(DEV)


def test_every_finite_e4m3_code_decodes_exactly():
    # out[r, c] = sum_k onehot(r)[k] * W[c, k] = dec(W[c, r]): a single exact product.
    m = k = 256
    n = 256
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    codes = finite[(np.arange(n)[:, None] + np.arange(k)[None, :]) % finite.size]
    rhs = _codes_to_e4m3(codes[None])
    lhs = torch.eye(m, k, dtype=torch.bfloat16, device=DEV)
    out = G.gmm(lhs, rhs, _gs([m]), out_dtype=torch.float32)
    expect = oracle.decode(codes).T  # [k=r, n=c]
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), expect)
    assert G.read_device_errors() == 0


def test_nan_codes_propagate():
    m, k, n = 16, 128, 128
    codes = np.full((1, n, k), 0x38, np.uint8)  # 1.0
    codes[0, 5, 7] = 0x7F
    codes[0, 9, 100] = 0xFF
    lhs = W.normal((m, k), 1.0, 3, DEV)
    out = G.gmm(lhs, _codes_to_e4m3(codes), _gs([m]), out_dtype=torch.float32).cpu()
    assert torch.isnan(out[:, 5]).all() and torch.isnan(out[:, 9]).all()
    others = [c for c in range(n) if c not in (5, 9)]
    assert torch.isfinite(out[:, others]).all()


def _scaled_case(m, k, n, sizes, nb, *, e4m3=True, out_dtype=torch.bfloat16, group_offset=0, local=None,
                 bias_dtype=torch.bfloat16, with_scale=True, seed=0):
    sizes = np.asarray(sizes, np.int32)
    L = local if local is not None else sizes.size - group_offset
    lhs = W.normal((m, k), 1.0, seed + 1, DEV)
    rhs = W.e4m3_normal((L, n, k), seed + 2, DEV) if e4m3 else W.normal((L, n, k), 0.05, seed + 2, DEV)
    scale = W.uniform((L, nb, 1, n), 0.5 / 448, 2.0 / 448, seed + 3, DEV) if with_scale else None
    bias = None if bias_dtype is None else W.normal((L, 1, n), 1.0, seed + 4, DEV, dtype=bias_dtype)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, rhs_bias=bias, group_offset=group_offset,
                out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(lhs, rhs, sizes, group_offset=group_offset, rhs_scale=scale, rhs_bias=bias)
    check_close(out, ref, mag, f"scaled m={m} k={k} n={n} nb={nb} sizes={sizes.tolist()}")
    return out


@pytest.mark.parametrize("nb", [1, 2, 4])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_decode_shapes_ragged(nb, out_dtype):
    # groups of 0..40 rows (several span 2-3 token chunks of 16), n with a 8-wide tail
    sizes = [3, 0, 17, 1, 40, 0, 8, 16, 5, 33]
    _scaled_case(int(np.sum(sizes)) + 9, 512, 392, sizes, nb, out_dtype=out_dtype, seed=nb)


@pytest.mark.parametrize("go,local", [(0, 4), (4, 6), (9, 1)])
def test_group_offset(go, local):
    sizes = [3, 0, 17, 1, 40, 0, 8, 16, 5, 33]
    _scaled_case(140, 256, 256, sizes, 2, group_offset=go, local=local, seed=go)


def test_no_scale_e4m3_and_f32_bias():
    _scaled_case(60, 384, 256, [20, 0, 30], 1, with_scale=False, bias_dtype=torch.float32)


def test_no_bias():
    _scaled_case(60, 256, 256, [20, 7, 30], 2, bias_dtype=None)


def test_bf16_weights_with_scale():
    _scaled_case(90, 512, 264, [12, 0, 50, 20], 4, e4m3=False, out_dtype=torch.float32)


def test_integer_exact_e4m3():
    # small integers are exact in e4m3 and bf16; power-of-two scales keep every sum exact
    m, k, n = 48, 256, 128
    sizes = np.array([10, 0, 21, 17], np.int32)
    lhs = W.integer_valued((m, k), -4, 4, 5, DEV)
    base = W.integer_valued((n, k), -4, 4, 6, DEV, dtype=torch.float32)
    rhs = torch.stack([(g + 1) * base for g in range(4)]).to(torch.float8_e4m3fn)
    scale = torch.tensor([0.5, 2.0], device=DEV).repeat(4, 1).reshape(4, 2, 1, 1).expand(4, 2, 1, n).contiguous()
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, out_dtype=torch.float32)
    ref, _ = oracle_gmm(lhs, rhs, sizes, rhs_scale=scale)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("go", [0, 32])
def test_fp8_decode_workload_full(go):
    """The FP8 decode workload at full size (256 rows, 64 experts of [2048, 4096] e4m3, 32
    k-blocks of 128), every output element checked; the second call slices experts 32-63."""
    d = W.fp8_decode(DEV)
    sizes = d["group_sizes"]
    rhs, scale, bias = d["rhs"][go:], d["rhs_scale"][go:], d["rhs_bias"][go:]
    out = G.gmm(d["lhs"], rhs, _gs(sizes), rhs_scale=scale, rhs_bias=bias, group_offset=go)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    ref, mag = oracle_gmm(d["lhs"], rhs, sizes, group_offset=go, rhs_scale=scale, rhs_bias=bias)
    check_close(out, ref, mag, f"fp8 decode go={go}")
    if go:
        offs = oracle.group_offsets(sizes, 256)
        assert (out[: offs[go]] == 0).all()


def test_activation_split_is_exact_for_eight_bit_values():
    # lhs: every bf16 significand (8 bits) times 2^e, e in [-2, 2]; weights: +-2^j, j in [-1, 1];
    # two quant blocks with scales 2^{-1,0,1}.  Every product is a multiple of 2^-10 below 2^4,
    # so each block's sum (< 2^11) and the scaled total (multiples of 2^-11 below 2^13) are exact
    # in fp32 whatever the order: the result must equal the oracle bit for bit, i.e. the e4m3
    # kernel's h + l / 16 split of the activations loses nothing.
    m, k, n = 40, 256, 256
    sizes = np.array([9, 31], np.int32)
    g = torch.Generator().manual_seed(71)
    mant = 1.0 + torch.randint(0, 128, (m, k), generator=g).double() / 128.0
    ex = torch.randint(-2, 3, (m, k), generator=g).double()
    sign = torch.where(torch.rand((m, k), generator=g) < 0.5, -1.0, 1.0).double()
    lhs = (sign * mant * torch.pow(2.0, ex)).to(torch.bfloat16).to(DEV)
    wj = torch.randint(-1, 2, (2, n, k), generator=g).double()
    ws = torch.where(torch.rand((2, n, k), generator=g) < 0.5, -1.0, 1.0).double()
    rhs = (ws * torch.pow(2.0, wj)).float().to(torch.float8_e4m3fn).to(DEV)
    scale = torch.pow(2.0, torch.randint(-1, 2, (2, 2, 1, n), generator=g).float()).to(DEV)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, out_dtype=torch.float32)
    ref, _ = oracle_gmm(lhs, rhs, sizes, rhs_scale=scale)
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_wide_dynamic_range_activations():
    # Within one 128-wide k step values span 2^-40 .. 2^8 (many below 2^-14 of the step's
    # largest); whole rows scaled by 2^100 and 2^-100.
    m, k, n = 24, 384, 256
    sizes = np.array([24], np.int32)
    g = torch.Generator().manual_seed(72)
    x = torch.randn((m, k), generator=g).double() * torch.pow(2.0, torch.randint(-40, 9, (m, k), generator=g).double())
    x[3] *= 2.0 ** 100
    x[7] *= 2.0 ** -100
    lhs = x.to(torch.bfloat16).to(DEV)
    rhs = W.e4m3_normal((1, n, k), 73, DEV)
    scale = W.uniform((1, 3, 1, n), 0.5 / 448, 2.0 / 448, 74, DEV)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_scale=scale, out_dtype=torch.float32)
    ref, mag = oracle_gmm(lhs, rhs, sizes, rhs_scale=scale)
    check_close(out, ref, mag, "wide dynamic range")


def test_zero_rows_give_the_bias_and_nan_propagates():
    m, k, n = 20, 256, 256
    sizes = np.array([20], np.int32)
    lhs = W.normal((m, k), 1.0, 81, DEV)
    lhs[4] = 0
    lhs[9, 130] = float("nan")
    rhs = W.e4m3_normal((1, n, k), 82, DEV)
    bias = W.normal((1, 1, n), 1.0, 83, DEV, dtype=torch.float32)
    out = G.gmm(lhs, rhs, _gs(sizes), rhs_bias=bias, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out[4], bias[0, 0])
    assert torch.isnan(out[9]).all()
    keep = [r for r in range(m) if r != 9]
    assert torch.isfinite(out[keep]).all()
