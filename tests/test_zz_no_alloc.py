"""gmm_noalloc: the grouped matmul for callers that cannot allocate device memory (their
device memory belongs to another component's allocator, or cudaMalloc is not allowed on
their path).  It runs the gmm kernels with a scratch array compiled into the library in
place of a caller-supplied workspace.

Called here through the C ABI (ctypes), three times in a row on different inputs; each result
must match the fp64 oracle within the bound the other parity tests use,
|gpu - ref| <= 1e-3 * mag + 2^-8 * |ref|, and agree with gmm() (which uses its own workspace)
within the same bound.  The third call has activation rows whose split marks them, so the
fp8 kernel's last CTA recomputes them through the counters kept in the library's array.  This
file is collected last so that a run stopping at the first failure has run every other test."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import REL_MAG, REL_REF, check_close, oracle_gmm

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _noalloc(lhs, rhs, gs, out, *, scale=None, bias=None, group_offset=0):
    lib = G.load_library()
    rc = lib.gmm_noalloc(lhs.data_ptr(), G._code(lhs), lhs.shape[0], lhs.shape[1], rhs.data_ptr(), G._code(rhs),
                         rhs.shape[0], rhs.shape[1], 1, gs.data_ptr(), gs.shape[0], group_offset,
                         None if scale is None else scale.data_ptr(), 0 if scale is None else scale.shape[1],
                         None if bias is None else bias.data_ptr(), 0 if bias is None else G._code(bias),
                         out.data_ptr(), G._code(out), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, G.GmmError("gmm_noalloc", rc)
    return out


def _agree(a, b, mag):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.all(np.abs(a - b) <= REL_MAG * mag + REL_REF * np.abs(b))


def test_noalloc_matches_gmm_on_two_calls_in_a_row():
    # call 1: bf16 weights, ragged groups with an empty one
    sizes1 = np.array([130, 0, 257, 1, 200], np.int32)
    lhs1 = W.normal((700, 256), 1.0, 61, DEV)
    rhs1 = W.normal((5, 520, 256), 0.05, 62, DEV)
    gs1 = torch.tensor(sizes1, device=DEV)
    # call 2: e4m3 weights with block scales and bias, a group_offset slice
    sizes2 = np.array([3, 0, 17, 9, 30], np.int32)
    lhs2 = W.normal((64, 512), 1.0, 63, DEV)
    rhs2 = W.e4m3_normal((3, 256, 512), 64, DEV)
    scale2 = W.uniform((3, 4, 1, 256), 0.5 / 448, 2.0 / 448, 65, DEV)
    bias2 = W.normal((3, 1, 256), 1.0, 66, DEV)
    gs2 = torch.tensor(sizes2, device=DEV)

    # call 3: e4m3 weights, rows holding three magnitudes 2^22 apart (1.0, 3 * 2^-22, 2^-44):
    # the two split levels hold only two, so the rows are marked and summed again
    sizes3 = np.array([20, 44], np.int32)
    lhs3 = W.normal((64, 512), 1.0, 67, DEV)
    lhs3[::5] = 3 * 2.0 ** -22
    lhs3[::5, ::64] = 1.0
    lhs3[::5, 1::64] = 2.0 ** -44
    rhs3 = W.e4m3_normal((2, 256, 512), 68, DEV)
    scale3 = W.uniform((2, 2, 1, 256), 0.5 / 448, 2.0 / 448, 69, DEV)
    gs3 = torch.tensor(sizes3, device=DEV)

    out1 = _noalloc(lhs1, rhs1, gs1, torch.full((700, 520), float("nan"), dtype=torch.bfloat16, device=DEV))
    out2 = _noalloc(lhs2, rhs2, gs2, torch.full((64, 256), float("nan"), dtype=torch.bfloat16, device=DEV),
                    scale=scale2, bias=bias2, group_offset=2)
    out3 = _noalloc(lhs3, rhs3, gs3, torch.full((64, 256), float("nan"), dtype=torch.bfloat16, device=DEV),
                    scale=scale3)
    torch.cuda.synchronize()

    ref1 = G.gmm(lhs1, rhs1, gs1)
    ref2 = G.gmm(lhs2, rhs2, gs2, rhs_scale=scale2, rhs_bias=bias2, group_offset=2)
    ref3 = G.gmm(lhs3, rhs3, gs3, rhs_scale=scale3)
    torch.cuda.synchronize()
    oref1, mag1 = oracle_gmm(lhs1, rhs1, sizes1)
    oref2, mag2 = oracle_gmm(lhs2, rhs2, sizes2, group_offset=2, rhs_scale=scale2, rhs_bias=bias2)
    oref3, mag3 = oracle_gmm(lhs3, rhs3, sizes3, rhs_scale=scale3)
    check_close(out1, oref1, mag1, "noalloc bf16 weights")
    check_close(out2, oref2, mag2, "noalloc e4m3 weights, scales, bias, offset")
    check_close(out3, oref3, mag3, "noalloc e4m3 weights, marked rows")
    _agree(out1, ref1, mag1)
    _agree(out2, ref2, mag2)
    _agree(out3, ref3, mag3)
