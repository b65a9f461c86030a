"""The Python binding has no CPU path: every entry point refuses host tensors before any work,
and the library's absence is an error, not a fallback."""

import pytest
import torch

import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def library():
    B.build()


def _host():
    lhs = torch.zeros((4, 128), dtype=torch.bfloat16)
    rhs = torch.zeros((2, 64, 128), dtype=torch.bfloat16)
    sizes = torch.tensor([2, 2], dtype=torch.int32)
    return lhs, rhs, sizes


@pytest.mark.parametrize("call", [
    lambda l, r, s: G.gmm(l, r, s),
    lambda l, r, s: G.gmm_into(l, r, s, torch.zeros((4, 64), dtype=torch.bfloat16)),
    lambda l, r, s: G.gmm(l, r, s, rhs_block_scale=torch.zeros((2, 64, 4), dtype=torch.uint8)),
    lambda l, r, s: G.tgmm(l, torch.zeros((4, 64), dtype=torch.bfloat16), s),
    lambda l, r, s: G.tgmm_local(l, torch.zeros((4, 64), dtype=torch.bfloat16), s, 0, 1),
    lambda l, r, s: G.quantize_e4m3(l),
], ids=["gmm", "gmm_into", "gmm_ex", "tgmm", "tgmm_local", "quantize_e4m3"])
def test_host_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA tensor"):
        call(*_host())


def test_a_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(G, "LIB_PATH", str(tmp_path / "libgmm.so"))
    monkeypatch.setattr(G, "_lib", None)
    with pytest.raises(ImportError, match="missing"):
        G.load_library()
