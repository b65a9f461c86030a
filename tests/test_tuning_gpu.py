"""The tiling table on the GPU: gmm_tune times every bf16 kernel choice and records the fastest;
gmm then runs that choice (its output equals the forced kernel's bit for bit); a table entry
replaces the built-in rule; a per-call bf16_kernel option still overrides both."""

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B
from moe_grouped_matrix_gb300 import workloads as W
from parity import check_close, oracle_gmm

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = {G.KERNEL_PAIR: "pair", G.KERNEL_SWAP_PAIR: "swap_pair", G.KERNEL_SWAP: "swap", G.KERNEL_SINGLE: "single"}


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()
    G.load_library()
    oracle.build()


@pytest.fixture(autouse=True)
def clean_table():
    G.tuning_clear()
    yield
    G.tuning_clear()


def _problem(seed=0):
    m, k, n = 2300, 512, 1024
    sizes = np.array([300, 0, 700, 250, 450, 600], np.int32)
    lhs = W.normal((m, k), 1.0, seed + 1, DEV)
    rhs = W.normal((6, n, k), 0.05, seed + 2, DEV)
    return lhs, rhs, sizes, torch.tensor(sizes, dtype=torch.int32, device=DEV)


def _forced(lhs, rhs, gs, name):
    return G.gmm(lhs, rhs, gs, out_dtype=torch.float32, options={"bf16_kernel": name})


def test_tune_records_the_fastest_choice_and_gmm_uses_it(monkeypatch):
    lhs, rhs, sizes, gs = _problem()
    kernel, raster, ms = G.tune(lhs, rhs, gs, out_dtype=torch.float32, iterations=3)
    assert kernel in NAMES and ms > 0
    rows = G.tuning_rows_log2(lhs.shape[0], sizes.size)
    assert G.tuning_get(rows, lhs.shape[1], rhs.shape[1], sizes.size, True, torch.float32) == (kernel, raster)
    out = G.gmm(lhs, rhs, gs, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert G.read_device_errors() == 0
    assert torch.equal(out, _forced(lhs, rhs, gs, NAMES[kernel]))
    ref, mag = oracle_gmm(lhs, rhs, sizes)
    check_close(out, ref, mag, f"tuned choice {NAMES[kernel]} raster {raster}")


@pytest.mark.parametrize("kernel", list(NAMES))
def test_table_entry_replaces_the_rule(kernel, monkeypatch):
    lhs, rhs, sizes, gs = _problem(seed=3)
    rows = G.tuning_rows_log2(lhs.shape[0], sizes.size)
    G.tuning_set(rows, lhs.shape[1], rhs.shape[1], sizes.size, True, torch.float32, kernel, 16)
    out = G.gmm(lhs, rhs, gs, out_dtype=torch.float32)
    assert torch.equal(out, _forced(lhs, rhs, gs, NAMES[kernel]))
    # a per-call choice wins over the entry
    other = G.KERNEL_SINGLE if kernel != G.KERNEL_SINGLE else G.KERNEL_SWAP
    with G.options(bf16_kernel=NAMES[other]):
        with_option = G.gmm(lhs, rhs, gs, out_dtype=torch.float32)
    assert torch.equal(with_option, _forced(lhs, rhs, gs, NAMES[other]))
    ref, mag = oracle_gmm(lhs, rhs, sizes)
    check_close(out, ref, mag, f"table entry {NAMES[kernel]}")


def test_tune_rejects_quantized_weights():
    lhs = W.normal((64, 256), 1.0, 5, DEV)
    rhs = W.weights("e4m3", (1, 256, 256), 6, DEV)
    with pytest.raises(G.GmmError) as e:
        G.tune(lhs, rhs, torch.tensor([64], dtype=torch.int32, device=DEV))
    assert e.value.status == 2
