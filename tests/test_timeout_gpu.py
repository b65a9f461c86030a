"""The bounded pipeline waits, made to run out on purpose without a fault.  A test switch of the
per-call options (test_drop_stage) makes one producer of a kernel leave a stage unissued: in the
one-SM kernel CTA 0 skips the copies of that stage; in the SM-pair kernels the second CTA of the
first pair stops issuing.  With a short wait bound (wait_limit_cycles) the consumer's wait for
that stage gives up: the call returns, the device report says GMM_ERR_TIMEOUT (and reading it
clears it), every copy and MMA in flight has been waited for and the tensor memory freed, so the
next ordinary call on the same workspace and stream runs on every SM and matches the oracle."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, oracle_gmm, oracle_tgmm

pytestmark = pytest.mark.gpu
DEV = "cuda"
ERR_TIMEOUT = 11  # GMM_ERR_TIMEOUT
SHORT_WAIT = 2_000_000  # clock cycles, about a millisecond
SIZES = np.array([300, 0, 500, 224], np.int32)  # sum 1024


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


def _workspace():
    return torch.zeros(G.load_library().gmm_workspace_bytes(), dtype=torch.uint8, device=DEV)


def _gmm_problem(seed):
    lhs = W.normal((int(SIZES.sum()), 512), 1.0, seed, DEV)
    rhs = W.normal((SIZES.size, 768, 512), 0.05, seed + 1, DEV)
    return lhs, rhs, torch.tensor(SIZES, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("kernel,drop", [("single", 2), ("single", 8), ("pair", 1), ("pair", 3),
                                         ("swap_pair", 2)])
def test_gmm_wait_runs_out_and_the_next_call_is_exact(kernel, drop):
    lhs, rhs, gs = _gmm_problem(seed=10 + drop)
    ws = _workspace()
    G.gmm(lhs, rhs, gs, out_dtype=torch.float32, workspace=ws,
          options={"bf16_kernel": kernel, "wait_limit_cycles": SHORT_WAIT, "test_drop_stage": drop})
    assert G.get_device_error(workspace=ws) == ERR_TIMEOUT
    assert G.read_device_errors(workspace=ws) == 0  # the read cleared the report
    # the same kernel, every SM, default bound: TMEM was freed and nothing is left in flight
    for _ in range(2):
        out = G.gmm(lhs, rhs, gs, out_dtype=torch.float32, workspace=ws, options={"bf16_kernel": kernel})
        assert G.read_device_errors(workspace=ws) == 0
    ref, mag = oracle_gmm(lhs, rhs, SIZES)
    check_close(out, ref, mag, f"{kernel} after a timed-out call")


def test_a_short_bound_alone_does_not_time_out():
    lhs, rhs, gs = _gmm_problem(seed=30)
    ws = _workspace()
    out = G.gmm(lhs, rhs, gs, out_dtype=torch.float32, workspace=ws,
                options={"bf16_kernel": "single", "wait_limit_cycles": SHORT_WAIT})
    assert G.get_device_error(workspace=ws) == 0
    ref, mag = oracle_gmm(lhs, rhs, SIZES)
    check_close(out, ref, mag, "single with a short wait bound")


def test_a_stage_past_the_end_is_no_drop():
    lhs, rhs, gs = _gmm_problem(seed=31)
    ws = _workspace()
    out = G.gmm(lhs, rhs, gs, out_dtype=torch.float32, workspace=ws,
                options={"bf16_kernel": "pair", "wait_limit_cycles": SHORT_WAIT, "test_drop_stage": 1 << 30})
    assert G.get_device_error(workspace=ws) == 0
    ref, mag = oracle_gmm(lhs, rhs, SIZES)
    check_close(out, ref, mag, "pair with an unreachable dropped stage")


@pytest.mark.parametrize("drop", [1, 4])
def test_tgmm_pair_wait_runs_out_and_the_next_call_is_exact(drop):
    m, k, n = int(SIZES.sum()), 256, 512
    lhs = W.normal((m, k), 1.0, 40 + drop, DEV)
    dout = W.normal((m, n), 1.0, 50 + drop, DEV)
    gs = torch.tensor(SIZES, dtype=torch.int32, device=DEV)
    ws = _workspace()
    G.tgmm(lhs, dout, gs, workspace=ws,
           options={"tgmm_kernel": "pair", "wait_limit_cycles": SHORT_WAIT, "test_drop_stage": drop})
    assert G.get_device_error(workspace=ws) == ERR_TIMEOUT
    out = G.tgmm(lhs, dout, gs, workspace=ws, options={"tgmm_kernel": "pair"})
    assert G.read_device_errors(workspace=ws) == 0
    ref, mag = oracle_tgmm(lhs, dout, SIZES)
    check_close(out, ref, mag, "tgmm pair after a timed-out call")


def test_timeout_options_are_checked():
    lhs, rhs, gs = _gmm_problem(seed=60)
    for bad in ({"wait_limit_cycles": -1}, {"test_drop_stage": -2}):
        with pytest.raises(G.GmmError) as e:
            G.gmm(lhs, rhs, gs, options=bad)
        assert e.value.status == 3
