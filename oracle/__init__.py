"""Grouped-matmul oracle: TEST INFRASTRUCTURE ONLY.

A ctypes front end for ``oracle.cpp``, the plain fp64 CPU statement of the
grouped matmul (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230",
tpu_inference/kernels/megablox/gmm.py: the ``gmm`` docstring, the ``_accum``
kernel body, ``make_group_metadata`` and ``_zero_uninitialized_memory``).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library and
the CUDA library never imports it.

Inputs are numpy arrays holding the stored bits of each dtype:
``uint16`` for bf16, ``float32``/``uint32`` for f32, ``uint8`` for e4m3fn (the
default for ``uint8``), e5m2 and the 4-bit formats, ``int8`` for int8.  int4,
uint4 and e2m1 are packed two values per byte, the even-indexed value in the low
nibble, so a row of k values is k / 2 bytes; pass their dtype code explicitly.
Outputs are fp64 ``ref`` (the exact-product, fp64-sum result) and ``mag``
(the same sum over absolute values, in which the tolerance is stated).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16, F32, E4M3, E5M2, INT8, INT4, UINT4, E2M1, E8M0 = 0, 1, 2, 3, 4, 5, 6, 7, 8
PACKED = (INT4, UINT4, E2M1)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles oracle.cpp into _liboracle.so with the host C++ compiler."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
            lib.oracle_gmm.argtypes = [P, I, I64, I64, P, I, I32, I64, I, P, I32, I32, P, I32, P, I,
                                       P, I64, P, P, I]
            lib.oracle_gmm.restype = I
            lib.oracle_gmm_ex.argtypes = [P, I, I64, I64, P, I, I32, I64, I, P, I32, I32, P, I, I32, P, I32, P, I,
                                          P, I64, P, P, I]
            lib.oracle_gmm_ex.restype = I
            lib.oracle_gmm_ex2.argtypes = [P, I, I64, I64, P, I, I32, I64, I, P, I32, I32, P, I, I32, P, I32, P, I,
                                           I32, P, I, P, I64, P, P, I]
            lib.oracle_gmm_ex2.restype = I
            lib.oracle_quantize_e4m3.argtypes = [P, I64, I64, I64, P, P]
            lib.oracle_quantize_e4m3.restype = I
            lib.oracle_tgmm.argtypes = [P, I, I64, I64, P, I, I64, P, I32, P, I64, P, P, I]
            lib.oracle_tgmm.restype = I
            lib.oracle_group_offsets.argtypes = [P, I32, I64, P]
            lib.oracle_group_offsets.restype = None
            lib.oracle_decode.argtypes = [P, I, I64, P]
            lib.oracle_decode.restype = I
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray, declared: int | None) -> int:
    if declared is not None:
        return declared
    if a.dtype == np.uint16:
        return BF16
    if a.dtype in (np.float32, np.uint32):
        return F32
    if a.dtype == np.uint8:
        return E4M3
    if a.dtype == np.int8:
        return INT8
    raise TypeError(f"unsupported stored dtype {a.dtype}")


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


def group_offsets(group_sizes: np.ndarray, m: int) -> np.ndarray:
    gs = np.ascontiguousarray(group_sizes, dtype=np.int32)
    out = np.zeros(gs.shape[0] + 1, dtype=np.int64)
    _load().oracle_group_offsets(_ptr(gs), gs.shape[0], m, _ptr(out))
    return out


def gmm(lhs, rhs, group_sizes, *, transpose_rhs=True, group_offset=0, rhs_scale=None,
        rhs_bias=None, rows=None, lhs_dtype=None, rhs_dtype=None, bias_dtype=None, lhs_scale=None,
        rhs_block_scale=None, rhs_block_scale_dtype=None, threads=0):
    """Forward grouped matmul in fp64.  Returns (ref, mag), each [rows, n].

    rhs_scale: f32 [L, nb, 1, n], or uint8 E8M0 codes of that shape.  lhs_scale: None or f32
    [m, num_lhs_blocks] (per-token-group activation scales).  rhs_block_scale: None or
    [L, n, k / block] per-element weight block scales, stored as rhs_block_scale_dtype (E8M0,
    E4M3 or F32; uint8 arrays default to E8M0, float32 to F32)."""
    lhs, rhs, bias = _c(lhs), _c(rhs), _c(rhs_bias)
    gs = np.ascontiguousarray(group_sizes, dtype=np.int32)
    scale_code = F32
    if rhs_scale is not None and np.asarray(rhs_scale).dtype == np.uint8:
        scale = np.ascontiguousarray(rhs_scale)
        scale_code = E8M0
    else:
        scale = None if rhs_scale is None else np.ascontiguousarray(rhs_scale, dtype=np.float32)
    lscale = None if lhs_scale is None else np.ascontiguousarray(lhs_scale, dtype=np.float32)
    m, k = lhs.shape
    L = rhs.shape[0]
    rcode = _dtype_code(rhs, rhs_dtype)
    n = rhs.shape[1] if transpose_rhs else rhs.shape[2] * (2 if rcode in PACKED else 1)
    nb = 0 if scale is None else scale.shape[1]
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    count = m if rows_arr is None else rows_arr.shape[0]
    ref = np.zeros((count, n), dtype=np.float64)
    mag = np.zeros((count, n), dtype=np.float64)
    bscale, bcode, bsize = None, 0, 0
    if rhs_block_scale is not None:
        bscale = np.ascontiguousarray(rhs_block_scale)
        bcode = rhs_block_scale_dtype if rhs_block_scale_dtype is not None else (
            E8M0 if bscale.dtype == np.uint8 else F32)
        bsize = k // bscale.shape[-1]
    rc = _load().oracle_gmm_ex2(
        _ptr(lhs), _dtype_code(lhs, lhs_dtype), m, k, _ptr(rhs), rcode, L, n,
        int(bool(transpose_rhs)), _ptr(gs), gs.shape[0], int(group_offset), _ptr(scale), scale_code, nb,
        _ptr(lscale), 0 if lscale is None else lscale.shape[1], _ptr(bscale), bcode, bsize,
        _ptr(bias), 0 if bias is None else _dtype_code(bias, bias_dtype), _ptr(rows_arr), count,
        _ptr(ref), _ptr(mag), int(threads))
    if rc != 0:
        raise ValueError("oracle_gmm rejected its arguments")
    return ref, mag


def tgmm(lhs, dout, group_sizes, *, k_rows=None, lhs_dtype=None, dout_dtype=None, threads=0):
    """Per-group lhs_g^T @ dout_g in fp64.  Returns (ref, mag), each [G, k_rows, n]."""
    lhs, dout = _c(lhs), _c(dout)
    gs = np.ascontiguousarray(group_sizes, dtype=np.int32)
    m, k = lhs.shape
    n = dout.shape[1]
    kr = None if k_rows is None else np.ascontiguousarray(k_rows, dtype=np.int64)
    kc = k if kr is None else kr.shape[0]
    ref = np.zeros((gs.shape[0], kc, n), dtype=np.float64)
    mag = np.zeros((gs.shape[0], kc, n), dtype=np.float64)
    rc = _load().oracle_tgmm(_ptr(lhs), _dtype_code(lhs, lhs_dtype), m, k, _ptr(dout),
                             _dtype_code(dout, dout_dtype), n, _ptr(gs), gs.shape[0], _ptr(kr), kc,
                             _ptr(ref), _ptr(mag), int(threads))
    if rc != 0:
        raise ValueError("oracle_tgmm rejected its arguments")
    return ref, mag


def quantize_e4m3(x_bf16_bits: np.ndarray, group: int = 128):
    """Per-token-group e4m3 quantisation of bf16 activations [m, k] (stored bits, uint16).
    Returns (codes uint8 [m, k], scales f32 [m, k / group])."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    m, k = x.shape
    q = np.zeros((m, k), np.uint8)
    sc = np.zeros((m, k // group), np.float32)
    if _load().oracle_quantize_e4m3(_ptr(x), m, k, group, _ptr(q), _ptr(sc)) != 0:
        raise ValueError("bad quantisation arguments")
    return q, sc


def decode(stored: np.ndarray, dtype: int | None = None) -> np.ndarray:
    """Decodes stored values to fp64 by the format definitions.  For the packed 4-bit
    formats the last axis doubles (two values per byte, low nibble first)."""
    a = np.ascontiguousarray(stored)
    code = _dtype_code(a, dtype)
    count = a.size * (2 if code in PACKED else 1)
    out = np.zeros(count, dtype=np.float64)
    if _load().oracle_decode(_ptr(a), code, count, _ptr(out)) != 0:
        raise ValueError("bad dtype")
    shape = a.shape[:-1] + (a.shape[-1] * 2,) if code in PACKED else a.shape
    return out.reshape(shape)
