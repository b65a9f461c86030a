"""Shared helpers for the GPU parity tests: run the oracle on the same stored bytes
the CUDA library read, and apply the acceptance bound
    |gpu - ref| <= 1e-3 * mag + 2^-8 * |ref|   (element-wise; NaN never accepted)
where ref is the oracle's exact-product fp64 sum and mag the same sum over
absolute values.  The bound covers fp32 accumulation of up to ~4096 products
(relative error well under 1e-3 of mag) plus one bf16 rounding of the result
(at most 2^-9 of |result| for round-to-nearest-even).  Where the definition's
result is not finite (an infinite or NaN input: x * inf is +-inf, 0 * inf and
inf - inf are NaN, IEEE arithmetic in the pages' dot_general) the GPU must give
the same infinity, or a NaN where ref is NaN.  Below the output format's
smallest normal (2^-126 for bf16 and f32) its values are spaced evenly, 2^-133
apart for bf16 and 2^-149 for f32, so no stored value need lie within 2^-8 of
ref there: the bound adds half that spacing, the most one rounding of the result
to the format can cost."""

import numpy as np
import torch

import oracle
import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300.workloads import stored_bits

REL_MAG = 1e-3
REL_REF = 2.0 ** -8


def bits(t):
    return stored_bits(t)


def check_close(gpu: torch.Tensor, ref: np.ndarray, mag: np.ndarray, what: str):
    g = gpu.detach().cpu().to(torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    finite = np.isfinite(ref)
    tiny = 2.0 ** -134 if gpu.dtype == torch.bfloat16 else 2.0 ** -150
    with np.errstate(invalid="ignore"):
        bound = REL_MAG * mag + REL_REF * np.abs(ref) + tiny
        err = np.abs(g - ref)
        ok = np.where(finite, err <= bound, (g == ref) | (np.isnan(ref) & np.isnan(g)))
    bad = ~ok  # NaN in g fails here unless ref is NaN
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = ", ".join(f"{tuple(i)}: gpu={g[tuple(i)]!r} ref={ref[tuple(i)]!r} mag={mag[tuple(i)]!r}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside the bound; {details}")


# Stored-format names of the weights -> the oracle's dtype codes (None: from the array's dtype).
ORACLE_FORMAT = {None: None, "e4m3": oracle.E4M3, "e5m2": oracle.E5M2, "int8": oracle.INT8, "int4": oracle.INT4,
                 "uint4": oracle.UINT4, "e2m1": oracle.E2M1}


def oracle_gmm(lhs, rhs, group_sizes_np, *, transpose_rhs=True, group_offset=0, rhs_scale=None, rhs_bias=None,
               rows=None, rhs_format=None):
    if rhs_format is None and rhs.dtype == torch.float8_e5m2:
        rhs_format = "e5m2"
    return oracle.gmm(bits(lhs), bits(rhs), group_sizes_np, transpose_rhs=transpose_rhs, group_offset=group_offset,
                      rhs_scale=None if rhs_scale is None else bits(rhs_scale),
                      rhs_bias=None if rhs_bias is None else bits(rhs_bias), rows=rows,
                      rhs_dtype=ORACLE_FORMAT[rhs_format])


def oracle_tgmm(lhs, dout, group_sizes_np, k_rows=None):
    return oracle.tgmm(bits(lhs), bits(dout), group_sizes_np, k_rows=k_rows)


def use_options(monkeypatch, **kw):
    """Kernel choices (gmm_options fields, e.g. bf16_kernel="pair", act_split="kernel") for the
    library calls of the rest of the test; undone when the test ends."""
    current = dict(getattr(G._defaults, "kw", {}))
    current.update(kw)
    monkeypatch.setattr(G._defaults, "kw", current, raising=False)
