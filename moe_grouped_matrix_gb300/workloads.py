"""Seeded synthetic inputs for the grouped matmul (MoE-shaped workloads).

This module only draws random numbers and routing counts: it holds none of the
grouped matmul's arithmetic, so the CUDA library and the CPU oracle can both be
fed from it without sharing any of the method.

Workloads (sizes follow the MoE layers the grouped matmul serves; the pages'
own workload is a 128-expert top-8 MoE, page "Megablox: transposed-RHS gmm_v2
kernel for the backward dlhs", Context section):

* ``tiny``        lhs [512,256] ~N(0,1); rhs [8,512,256] ~N(0,1/16) (std 1/sqrt(256)),
                  NT layout; group sizes: multinomial of 512 rows over 7 groups, one
                  seeded group forced empty; fp32 output.
* ``mixtral_up``  8192 tokens, top-2 of 8 experts (softmax of N(0,1) logits) ->
                  16384 rows; lhs [16384,4096] ~N(0,1); rhs [8,28672,4096] ~N(0,0.02),
                  NT; bf16 output.
* ``moe128``      4096 tokens, top-8 of 128 experts; 10 seeded experts never chosen,
                  the other 118 weighted by rank^-1.1 over a seeded permutation and
                  drawn without replacement -> 32768 rows; lhs [32768,2048] ~N(0,1);
                  wi [128,2048,2048], wo [128,2048,1024] ~N(0,0.02); dout ~N(0,0.01).
* ``fp8_decode``  64 tokens, uniform top-4 of 64 experts -> 256 rows; lhs [256,4096]
                  ~N(0,1); rhs e4m3fn [64,2048,4096] from N(0,1) clipped to +-448;
                  rhs_scale [64,32,1,2048] ~U(0.5,2)/448; rhs_bias [64,1,2048] ~N(0,1).

Standard deviations are what the ``N(0, s)`` figures denote.  Tensors are drawn
with ``torch.Generator`` on the device they are requested on, so the same seed
gives different bytes on CPU and GPU; a parity check always feeds both sides the
same stored bytes.
"""

from __future__ import annotations

import numpy as np
import torch


# ---------------------------------------------------------------- group sizes
def group_sizes_multinomial(seed: int, m: int, groups: int) -> np.ndarray:
    """m rows spread uniformly over all groups but one seeded group, which is empty."""
    rng = np.random.Generator(np.random.PCG64(seed))
    empty = int(rng.integers(groups))
    p = np.full(groups, 1.0 / (groups - 1))
    p[empty] = 0.0
    sizes = rng.multinomial(m, p)
    return sizes.astype(np.int32)


def group_sizes_topk_softmax(seed: int, tokens: int, experts: int, topk: int) -> np.ndarray:
    """Counts of a softmax top-k router over N(0,1) logits; ties go to the lower index."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((tokens, experts))
    # softmax is monotone, so the top-k of the probabilities is the top-k of the logits
    order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    return np.bincount(order.reshape(-1), minlength=experts).astype(np.int32)


def group_sizes_zipf(seed: int, tokens: int, experts: int, topk: int, s: float,
                     n_empty: int) -> np.ndarray:
    """Zipf-skewed top-k routing with `n_empty` experts that no token picks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(experts)
    empty = perm[:n_empty]
    live = perm[n_empty:]
    w = np.arange(1, live.size + 1, dtype=np.float64) ** (-s)
    w /= w.sum()
    counts = np.zeros(experts, dtype=np.int64)
    for _ in range(tokens):
        pick = rng.choice(live.size, size=topk, replace=False, p=w)
        counts[live[pick]] += 1
    assert counts[empty].sum() == 0
    return counts.astype(np.int32)


def group_sizes_uniform_topk(seed: int, tokens: int, experts: int, topk: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    counts = np.zeros(experts, dtype=np.int64)
    for _ in range(tokens):
        counts[rng.choice(experts, size=topk, replace=False)] += 1
    return counts.astype(np.int32)


# ---------------------------------------------------------------- tensors
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std) drawn in fp32, then rounded to `dtype` (round-to-nearest-even)."""
    x = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    x = torch.rand(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def e4m3_normal(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) clipped to the e4m3fn range +-448, then cast to float8_e4m3fn."""
    x = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)


def integer_valued(shape, lo: int, hi: int, seed: int, device="cpu", dtype=torch.bfloat16):
    """Uniform integers in [lo, hi] stored in a float dtype (exact in bf16 for |v| <= 256)."""
    x = torch.randint(lo, hi + 1, shape, generator=_gen(seed, device), device=device)
    return x.to(dtype)


# ---------------------------------------------------------------- workloads
def tiny(device="cpu", seed: int = 0):
    gs = group_sizes_multinomial(seed, 512, 8)
    return dict(
        lhs=normal((512, 256), 1.0, seed + 1, device),
        rhs=normal((8, 512, 256), 1.0 / 16.0, seed + 2, device),
        group_sizes=gs, transpose_rhs=True, out_dtype=torch.float32)


def mixtral_up(device="cpu", seed: int = 1):
    gs = group_sizes_topk_softmax(seed, 8192, 8, 2)
    return dict(
        lhs=normal((16384, 4096), 1.0, seed + 1, device),
        rhs=normal((8, 28672, 4096), 0.02, seed + 2, device),
        group_sizes=gs, transpose_rhs=True, out_dtype=torch.bfloat16)


def moe128_group_sizes(seed: int = 2) -> np.ndarray:
    return group_sizes_zipf(seed, 4096, 128, 8, 1.1, 10)


def moe128(device="cpu", seed: int = 2, which=("lhs", "wi", "wo", "lhs_wo", "dout")):
    gs = moe128_group_sizes(seed)
    d = dict(group_sizes=gs)
    if "lhs" in which:
        d["lhs"] = normal((32768, 2048), 1.0, seed + 1, device)
    if "wi" in which:
        d["wi"] = normal((128, 2048, 2048), 0.02, seed + 2, device)
    if "wo" in which:
        d["wo"] = normal((128, 2048, 1024), 0.02, seed + 3, device)
    if "lhs_wo" in which:
        d["lhs_wo"] = normal((32768, 1024), 1.0, seed + 4, device)
    if "dout" in which:
        d["dout"] = normal((32768, 2048), 0.01, seed + 5, device)
    return d


# Largest magnitude of each weight format (the quant scales below are U(0.5, 2) / this).
FORMAT_MAX = {"e4m3": 448.0, "e5m2": 448.0, "int8": 127.0, "int4": 8.0, "uint4": 15.0, "e2m1": 6.0}
PACKED = ("int4", "uint4", "e2m1")


def weights(fmt: str, shape, seed: int, device="cpu") -> torch.Tensor:
    """Weights [G, n, k] in a stored format: e4m3 / e5m2 from N(0,1) (e4m3 clipped to
    +-448), int8 uniform over all 256 codes, the 4-bit formats as uniform random bytes
    (every code equally likely), packed [G, n, k / 2] with the even k in the low nibble."""
    if fmt == "e4m3":
        return e4m3_normal(shape, seed, device)
    if fmt == "e5m2":
        x = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
        return x.to(torch.float8_e5m2)
    if fmt == "int8":
        return torch.randint(-128, 128, shape, generator=_gen(seed, device), device=device).to(torch.int8)
    if fmt in PACKED:
        packed = tuple(shape[:-1]) + (shape[-1] // 2,)
        return torch.randint(0, 256, packed, generator=_gen(seed, device), device=device).to(torch.uint8)
    raise ValueError(fmt)


def fp8_decode(device="cpu", seed: int = 4, fmt: str = "e4m3"):
    """The decode workload; `fmt` other than e4m3 swaps in weights of that format (same
    shapes, scales U(0.5, 2) / the format's largest magnitude)."""
    gs = group_sizes_uniform_topk(seed, 64, 64, 4)
    top = FORMAT_MAX[fmt]
    return dict(
        lhs=normal((256, 4096), 1.0, seed + 1, device),
        rhs=weights(fmt, (64, 2048, 4096), seed + 2, device),
        rhs_scale=uniform((64, 32, 1, 2048), 0.5 / top, 2.0 / top, seed + 3, device),
        rhs_bias=normal((64, 1, 2048), 1.0, seed + 4, device),
        group_sizes=gs, transpose_rhs=True, out_dtype=torch.bfloat16,
        rhs_format=fmt if fmt in PACKED else None)


def sample_rows(seed: int, offsets: np.ndarray, per_group: int) -> np.ndarray:
    """Seeded choice of up to `per_group` rows inside every group (sorted), plus the
    first and last row of each non-empty group so that group edges are always checked."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = []
    for g in range(offsets.size - 1):
        lo, hi = int(offsets[g]), int(offsets[g + 1])
        if hi <= lo:
            continue
        cnt = min(per_group, hi - lo)
        pick = rng.choice(hi - lo, size=cnt, replace=False) + lo
        rows.append(np.unique(np.concatenate([pick, [lo, hi - 1]])))
    return np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)


def stored_bits(t: torch.Tensor) -> np.ndarray:
    """The stored bytes of a CPU tensor as the numpy dtype the oracle reads."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.uint16).numpy()
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.view(torch.uint8).numpy()
    if t.dtype in (torch.float32, torch.int8, torch.uint8):
        return t.numpy()
    raise TypeError(t.dtype)
