"""Grouped matrix multiplication (gmm / NT gmm / tgmm) for GB300, behind the C ABI of libgmm.

This module only marshals arguments: every step of the computation runs in
the CUDA kernels of ``libgmm.so`` (sources in ``csrc/``, ABI in
``include/libgmm.h``).  PyTorch supplies device memory and streams.  If the
library is not built, importing the ops raises: there is no fallback.

    gmm(lhs, rhs, group_sizes, rhs_scale=None, rhs_bias=None, transpose_rhs=True,
        group_offset=0, out=None, out_dtype=torch.bfloat16)
    tgmm(lhs, dout, group_sizes, out=None, out_dtype=torch.float32)

Definitions: page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230",
tpu_inference/kernels/megablox/gmm.py (gmm), and page "Megablox:
transposed-RHS gmm_v2 kernel for the backward dlhs" (NT dlhs, drhs).
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["gmm", "gmm_into", "tgmm", "tgmm_local", "quantize_e4m3", "tune", "tuning_set", "tuning_get", "tuning_clear",
           "tuning_save", "tuning_load", "tuning_rows_log2", "read_device_errors", "get_device_error", "workspace_for",
           "release_workspaces", "options", "GmmOptions", "GmmError", "LIB_PATH", "load_library",
           "DEVERR_NEGATIVE_GROUP_SIZE", "DEVERR_GROUP_SIZES_EXCEED_M", "DEVERR_TIMEOUT"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgmm.so")

DTYPE_BF16, DTYPE_F32, DTYPE_E4M3, DTYPE_E5M2, DTYPE_INT8, DTYPE_INT4, DTYPE_UINT4, DTYPE_E2M1, DTYPE_E8M0 = range(9)
# Packed 4-bit weight formats (uint8 tensors [L, n, k / 2], even k in the low nibble), by name.
PACKED_FORMATS = {"int4": DTYPE_INT4, "uint4": DTYPE_UINT4, "e2m1": DTYPE_E2M1}
# bf16 forward kernels, as the tiling table and the options name them.
KERNEL_AUTO, KERNEL_PAIR, KERNEL_SWAP_PAIR, KERNEL_SWAP, KERNEL_SINGLE = range(5)
KERNEL_IDS = {"auto": KERNEL_AUTO, "pair": KERNEL_PAIR, "swap_pair": KERNEL_SWAP_PAIR, "swap": KERNEL_SWAP,
              "single": KERNEL_SINGLE}
E4M3_KERNELS = {"auto": 0, "tensor": 1, "decode": 2}
ACT_SPLITS = {"auto": 0, "pass": 1, "kernel": 2}
TGMM_KERNELS = {"auto": 0, "single": 1, "pair": 2}
DEVERR_NEGATIVE_GROUP_SIZE, DEVERR_GROUP_SIZES_EXCEED_M, DEVERR_TIMEOUT, DEVERR_GROUP_OFFSET = 0x1, 0x2, 0x4, 0x8

_TORCH_TO_CODE = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32, torch.float8_e4m3fn: DTYPE_E4M3,
                  torch.float8_e5m2: DTYPE_E5M2, torch.int8: DTYPE_INT8}

_lock = threading.Lock()
_lib = None
_workspaces: dict[tuple[int, int], torch.Tensor] = {}
_defaults = threading.local()


class GmmOptions(ctypes.Structure):
    """gmm_options of the C ABI: per-call kernel choices (0 everywhere = every default)."""
    _fields_ = [("bf16_kernel", ctypes.c_int32), ("e4m3_kernel", ctypes.c_int32), ("act_split", ctypes.c_int32),
                ("tgmm_kernel", ctypes.c_int32), ("wait_limit_cycles", ctypes.c_int64),
                ("test_drop_stage", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def _make_options(bf16_kernel="auto", e4m3_kernel="auto", act_split="auto", tgmm_kernel="auto", wait_limit_cycles=0,
                  test_drop_stage=0, **unknown):
    if unknown:
        raise TypeError(f"unknown options {sorted(unknown)}")
    o = GmmOptions()
    o.bf16_kernel = bf16_kernel if isinstance(bf16_kernel, int) else KERNEL_IDS[bf16_kernel]
    o.e4m3_kernel = e4m3_kernel if isinstance(e4m3_kernel, int) else E4M3_KERNELS[e4m3_kernel]
    o.act_split = act_split if isinstance(act_split, int) else ACT_SPLITS[act_split]
    o.tgmm_kernel = tgmm_kernel if isinstance(tgmm_kernel, int) else TGMM_KERNELS[tgmm_kernel]
    o.wait_limit_cycles = int(wait_limit_cycles)
    o.test_drop_stage = int(test_drop_stage)
    return o


class options:
    """Kernel choices for the calls made on this thread inside the block, e.g.
    ``with options(bf16_kernel="pair"): gmm(...)``; passed to the library as its
    per-call gmm_options (the library reads no environment variable for them)."""

    def __init__(self, **kw):
        self.kw = kw

    def __enter__(self):
        self.saved = getattr(_defaults, "kw", {})
        _defaults.kw = {**self.saved, **self.kw}
        return self

    def __exit__(self, *exc):
        _defaults.kw = self.saved
        return False


def _current_options(extra):
    kw = {**getattr(_defaults, "kw", {}), **(extra or {})}
    return _make_options(**kw) if kw else None

# Every function the header declares, with its ctypes signature.
_P, _I, _I32, _I64, _SZ, _U32P = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                                  ctypes.POINTER(ctypes.c_uint32))
_IP = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "gmm_workspace_bytes": ([], _SZ),
    "gmm_workspace_bytes_for": ([_I64, _I64, _I64, _I32, _I32, _I, _I], _SZ),
    "gmm": ([_P, _I, _I64, _I64, _P, _I, _I32, _I64, _I, _P, _I32, _I32, _P, _I32, _P, _I, _P, _I, _P, _SZ, _P], _I),
    "tgmm": ([_P, _I, _P, _I, _I64, _I64, _I64, _P, _I32, _P, _I, _P, _SZ, _P], _I),
    "gmm_into": ([_P, _I, _I64, _I64, _P, _I, _I32, _I64, _I, _P, _I32, _I32, _P, _I32, _P, _I, _P, _I, _P, _SZ, _P], _I),
    "gmm_device_offset": ([_P, _I, _I64, _I64, _P, _I, _I32, _I64, _I, _P, _I32, _P, _P, _I32, _P, _I, _P, _I, _I, _P,
                           _SZ, _P], _I),
    "tgmm_local": ([_P, _I, _P, _I, _I64, _I64, _I64, _P, _I32, _I32, _I32, _P, _I, _P, _SZ, _P], _I),
    "gmm_noalloc": ([_P, _I, _I64, _I64, _P, _I, _I32, _I64, _I, _P, _I32, _I32, _P, _I32, _P, _I, _P, _I, _P], _I),
    "gmm_quantize_e4m3": ([_P, _I, _I64, _I64, _I64, _P, _P, _P], _I),
    "gmm_ex": ([_P, _I, _P, _I32, _I64, _I64, _P, _I, _I32, _I64, _I, _P, _I32, _I32, _P, _P, _I, _I32, _P, _I, _I32, _P,
                _I, _P, _I, _I, _P, _P, _SZ, _P], _I),
    "tgmm_ex": ([_P, _I, _P, _I, _I64, _I64, _I64, _P, _I32, _I32, _I32, _P, _I, _P, _P, _SZ, _P], _I),
    "gmm_tuning_set": ([_I32, _I64, _I64, _I32, _I, _I, _I, _I], _I),
    "gmm_tuning_get": ([_I32, _I64, _I64, _I32, _I, _I, _IP, _IP], _I),
    "gmm_tuning_clear": ([], _I),
    "gmm_tuning_save": ([ctypes.c_char_p], _I),
    "gmm_tuning_load": ([ctypes.c_char_p], _I),
    "gmm_tune": ([_P, _I, _I64, _I64, _P, _I, _I32, _I64, _I, _P, _I32, _I32, _P, _I, _P, _I, _P, _SZ, _P, _I, _IP,
                  _IP, ctypes.POINTER(ctypes.c_float)], _I),
    "gmm_read_device_errors": ([_P, _P, _U32P], _I),
    "gmm_get_device_error": ([_P, _P], _I),
    "gmm_status_string": ([_I], ctypes.c_char_p),
    "gmm_last_cuda_error": ([], _I),
}


class GmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = load_library()
        msg = lib.gmm_status_string(status).decode()
        extra = f" (CUDA error {lib.gmm_last_cuda_error()})" if status == 8 else ""
        super().__init__(f"{fn}: status {status}: {msg}{extra}")
        self.status = status


def load_library() -> ctypes.CDLL:
    """Loads libgmm.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with `python -m moe_grouped_matrix_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def workspace_for(device: torch.device, stream=None) -> torch.Tensor:
    """A zero-filled workspace of gmm_workspace_bytes() bytes for calls on `stream` (default:
    the device's current stream), cached per (device, stream).  The workspace holds per-call
    scratch (the split activation rows of the 8- and 4-bit weight kernels) as well as the
    error flags, so calls on different streams, which may run at the same time, each get
    their own; calls on one stream are ordered and share it."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    dev = torch.device("cuda", idx)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    key = (idx, s.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None:
        nbytes = int(load_library().gmm_workspace_bytes())
        with torch.cuda.stream(s):  # zero-filled in order with the stream's calls
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def release_workspaces(device=None) -> None:
    """Drops the cached default workspaces (of one device, or of all), e.g. after using
    many short-lived streams.  Their device error flags go with them."""
    idx = None if device is None else torch.device(device).index
    for key in [k for k in _workspaces if idx is None or k[0] == idx]:
        del _workspaces[key]


def _code(t: torch.Tensor) -> int:
    try:
        return _TORCH_TO_CODE[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _stream(device, stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _gmm_call(fn, lhs, rhs, group_sizes, rhs_scale, rhs_bias, transpose_rhs, group_offset, out, out_dtype,
              workspace, stream, rhs_format, lhs_scale=None, rhs_block_scale=None, opts=None):
    lib = load_library()
    opt = _current_options(opts)
    _dev(lhs, "lhs"), _dev(rhs, "rhs"), _dev(group_sizes, "group_sizes")
    if group_sizes.dtype != torch.int32:
        raise TypeError("group_sizes must be int32")
    if rhs_format is None:
        rcode = _code(rhs)
    else:
        if rhs_format not in PACKED_FORMATS or rhs.dtype != torch.uint8:
            raise TypeError("rhs_format names a packed 4-bit format (int4, uint4, e2m1) of a uint8 tensor")
        rcode = PACKED_FORMATS[rhs_format]
    m, k = lhs.shape
    n = rhs.shape[1] if transpose_rhs else rhs.shape[2]
    kr = (rhs.shape[2] if transpose_rhs else rhs.shape[1]) * (2 if rhs_format is not None else 1)
    if kr != k:
        raise ValueError(f"lhs has k={k} but rhs has k={kr}")
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=lhs.device)
    _dev(out, "out")
    if tuple(out.shape) != (m, n):
        raise ValueError(f"out must be [{m}, {n}], got {list(out.shape)}")
    ws = workspace if workspace is not None else workspace_for(lhs.device, stream)
    nb = 0
    if rhs_scale is not None:
        _dev(rhs_scale, "rhs_scale")
        nb = rhs_scale.shape[1]
    if rhs_bias is not None:
        _dev(rhs_bias, "rhs_bias")
    e8m0 = rhs_scale is not None and rhs_scale.dtype == torch.uint8
    if rhs_block_scale is not None:
        _dev(rhs_block_scale, "rhs_block_scale")
        if rhs_block_scale.dim() != 3 or k % rhs_block_scale.shape[2] != 0:
            raise ValueError("rhs_block_scale must be [G_local, n, k / block_size]")
    if (lhs.dtype == torch.float8_e4m3fn or lhs_scale is not None or e8m0 or rhs_block_scale is not None
            or opt is not None):
        # e4m3 activations with their scales, E8M0 weight scales, block scales or options: gmm_ex
        if lhs_scale is not None:
            _dev(lhs_scale, "lhs_scale")
            if lhs_scale.dtype != torch.float32 or lhs_scale.dim() != 2 or lhs_scale.shape[0] != m:
                raise ValueError("lhs_scale must be float32 [m, num_lhs_blocks]")
        dev_off = isinstance(group_offset, torch.Tensor)
        if dev_off:
            _dev(group_offset, "group_offset")
            if group_offset.dtype != torch.int32 or group_offset.numel() != 1:
                raise TypeError("a tensor group_offset must be one int32 on the device")
        rc = lib.gmm_ex(lhs.data_ptr(), _code(lhs), None if lhs_scale is None else lhs_scale.data_ptr(),
                        0 if lhs_scale is None else lhs_scale.shape[1], m, k, rhs.data_ptr(), rcode, rhs.shape[0], n,
                        int(bool(transpose_rhs)), group_sizes.data_ptr(), group_sizes.shape[0],
                        0 if dev_off else int(group_offset), group_offset.data_ptr() if dev_off else None,
                        None if rhs_scale is None else rhs_scale.data_ptr(), DTYPE_E8M0 if e8m0 else DTYPE_F32, nb,
                        None if rhs_block_scale is None else rhs_block_scale.data_ptr(),
                        DTYPE_E8M0 if rhs_block_scale is None or rhs_block_scale.dtype == torch.uint8 else
                        _code(rhs_block_scale),
                        0 if rhs_block_scale is None else k // rhs_block_scale.shape[2],
                        None if rhs_bias is None else rhs_bias.data_ptr(),
                        0 if rhs_bias is None else _code(rhs_bias), out.data_ptr(), _code(out),
                        int(fn == "gmm_into"), None if opt is None else ctypes.byref(opt), ws.data_ptr(), ws.numel(),
                        _stream(lhs.device, stream))
        if rc != 0:
            raise GmmError("gmm_ex", rc)
        return out
    head = (lhs.data_ptr(), _code(lhs), m, k, rhs.data_ptr(), rcode, rhs.shape[0], n, int(bool(transpose_rhs)),
            group_sizes.data_ptr(), group_sizes.shape[0])
    tail = (None if rhs_scale is None else rhs_scale.data_ptr(), nb,
            None if rhs_bias is None else rhs_bias.data_ptr(), 0 if rhs_bias is None else _code(rhs_bias),
            out.data_ptr(), _code(out))
    if isinstance(group_offset, torch.Tensor):
        # a device scalar, read by the kernel when it runs (gmm_device_offset)
        _dev(group_offset, "group_offset")
        if group_offset.dtype != torch.int32 or group_offset.numel() != 1:
            raise TypeError("a tensor group_offset must be one int32 on the device")
        rc = lib.gmm_device_offset(*head, group_offset.data_ptr(), *tail, int(fn == "gmm_into"), ws.data_ptr(),
                                   ws.numel(), _stream(lhs.device, stream))
        fn = "gmm_device_offset"
    else:
        rc = getattr(lib, fn)(*head, int(group_offset), *tail, ws.data_ptr(), ws.numel(), _stream(lhs.device, stream))
    if rc != 0:
        raise GmmError(fn, rc)
    return out


def gmm(lhs, rhs, group_sizes, rhs_scale=None, rhs_bias=None, transpose_rhs=True, group_offset=0, out=None,
        out_dtype=torch.bfloat16, workspace=None, stream=None, rhs_format=None, lhs_scale=None,
        rhs_block_scale=None, options=None):
    """out[r] = lhs[r] @ W_g^T (NT, rhs [G_local, n, k]) or lhs[r] @ W_g (NN, rhs [G_local, k, n])
    for each row r of local group g; all other rows of out are zero.  group_offset is an int, or a
    one-element int32 CUDA tensor that the kernel reads when it runs.  rhs is bf16, float8_e4m3fn,
    float8_e5m2 or int8, or a uint8 tensor [G_local, n, k / 2] of packed 4-bit weights with
    rhs_format = "int4", "uint4" or "e2m1".  rhs_scale is float32 [G_local, nb, 1, n], or uint8
    E8M0 codes of that shape.  lhs may be float8_e4m3fn (W8A8) with lhs_scale float32
    [m, num_lhs_blocks] (quantize_e4m3's scales).  rhs_block_scale: microscaling scales, uint8 E8M0
    [G_local, n, k / 32] of float8_e4m3fn weights (MXFP8) or float8_e4m3fn [G_local, n, k / 16] of
    packed e2m1 weights (NVFP4).  options: a dict of gmm_options fields (bf16_kernel, e4m3_kernel,
    act_split, wait_limit_cycles, test_drop_stage), over those of an enclosing ``options`` block."""
    return _gmm_call("gmm", lhs, rhs, group_sizes, rhs_scale, rhs_bias, transpose_rhs, group_offset, out,
                     out_dtype, workspace, stream, rhs_format, lhs_scale, rhs_block_scale, options)


def gmm_into(lhs, rhs, group_sizes, out, rhs_scale=None, rhs_bias=None, transpose_rhs=True, group_offset=0,
             workspace=None, stream=None, rhs_format=None, lhs_scale=None, rhs_block_scale=None, options=None):
    """As gmm, but only the local groups' rows of `out` are written; every other row keeps the
    caller's contents (the existing-output mode)."""
    if out is None:
        raise ValueError("gmm_into needs an output tensor")
    return _gmm_call("gmm_into", lhs, rhs, group_sizes, rhs_scale, rhs_bias, transpose_rhs, group_offset, out,
                     out.dtype, workspace, stream, rhs_format, lhs_scale, rhs_block_scale, options)


def tgmm_local(lhs, dout, group_sizes, group_offset=0, num_local_groups=None, out=None, out_dtype=torch.float32,
               workspace=None, stream=None, options=None):
    """out[l] = lhs_g^T @ dout_g for g = group_offset + l, 0 <= l < num_local_groups (zero blocks for
    empty groups); group rows come from all of group_sizes."""
    lib = load_library()
    _dev(lhs, "lhs"), _dev(dout, "dout"), _dev(group_sizes, "group_sizes")
    if group_sizes.dtype != torch.int32:
        raise TypeError("group_sizes must be int32")
    m, k = lhs.shape
    if dout.shape[0] != m:
        raise ValueError("lhs and dout must have the same number of rows")
    n = dout.shape[1]
    G = group_sizes.shape[0]
    L = G - int(group_offset) if num_local_groups is None else int(num_local_groups)
    if out is None:
        out = torch.empty((max(L, 0), k, n), dtype=out_dtype, device=lhs.device)
    _dev(out, "out")
    if tuple(out.shape) != (L, k, n):
        raise ValueError(f"out must be [{L}, {k}, {n}], got {list(out.shape)}")
    ws = workspace if workspace is not None else workspace_for(lhs.device, stream)
    opt = _current_options(options)
    rc = lib.tgmm_ex(lhs.data_ptr(), _code(lhs), dout.data_ptr(), _code(dout), m, k, n, group_sizes.data_ptr(),
                     G, int(group_offset), L, out.data_ptr(), _code(out), None if opt is None else ctypes.byref(opt),
                     ws.data_ptr(), ws.numel(), _stream(lhs.device, stream))
    if rc != 0:
        raise GmmError("tgmm_ex", rc)
    return out


def tgmm(lhs, dout, group_sizes, out=None, out_dtype=torch.float32, workspace=None, stream=None, options=None):
    """out[g] = lhs_g^T @ dout_g for every group g (zero blocks for empty groups)."""
    lib = load_library()
    _dev(lhs, "lhs"), _dev(dout, "dout"), _dev(group_sizes, "group_sizes")
    if group_sizes.dtype != torch.int32:
        raise TypeError("group_sizes must be int32")
    m, k = lhs.shape
    if dout.shape[0] != m:
        raise ValueError("lhs and dout must have the same number of rows")
    n = dout.shape[1]
    G = group_sizes.shape[0]
    if out is None:
        out = torch.empty((G, k, n), dtype=out_dtype, device=lhs.device)
    _dev(out, "out")
    ws = workspace if workspace is not None else workspace_for(lhs.device, stream)
    opt = _current_options(options)
    if opt is not None:
        rc = lib.tgmm_ex(lhs.data_ptr(), _code(lhs), dout.data_ptr(), _code(dout), m, k, n, group_sizes.data_ptr(), G,
                         0, G, out.data_ptr(), _code(out), ctypes.byref(opt), ws.data_ptr(), ws.numel(),
                         _stream(lhs.device, stream))
        if rc != 0:
            raise GmmError("tgmm_ex", rc)
        return out
    rc = lib.tgmm(lhs.data_ptr(), _code(lhs), dout.data_ptr(), _code(dout), m, k, n, group_sizes.data_ptr(), G,
                  out.data_ptr(), _code(out), ws.data_ptr(), ws.numel(), _stream(lhs.device, stream))
    if rc != 0:
        raise GmmError("tgmm", rc)
    return out


def quantize_e4m3(x, group=128, out=None, scale=None, stream=None):
    """Per-token-group e4m3 quantisation of bf16 activations [m, k]: returns (q float8_e4m3fn
    [m, k], scale f32 [m, k / group])."""
    _dev(x, "x")
    m, k = x.shape
    q = out if out is not None else torch.empty((m, k), dtype=torch.float8_e4m3fn, device=x.device)
    sc = scale if scale is not None else torch.empty((m, k // group), dtype=torch.float32, device=x.device)
    _dev(q, "out"), _dev(sc, "scale")
    _check("gmm_quantize_e4m3", load_library().gmm_quantize_e4m3(x.data_ptr(), _code(x), m, k, group, q.data_ptr(),
                                                                 sc.data_ptr(), _stream(x.device, stream)))
    return q, sc


def tuning_rows_log2(m: int, num_total_groups: int) -> int:
    """The table's row class: floor(log2(m // num_total_groups)), 0 when that is 0."""
    avg = m // num_total_groups if num_total_groups > 0 else m
    return max(avg.bit_length() - 1, 0)


def _check(fn, rc):
    if rc != 0:
        raise GmmError(fn, rc)


def tuning_set(rows_log2, k, n, num_total_groups, transpose_rhs, out_dtype, kernel, raster=0):
    """Records the bf16 kernel (KERNEL_*) and raster for a problem class."""
    _check("gmm_tuning_set", load_library().gmm_tuning_set(rows_log2, k, n, num_total_groups, int(bool(transpose_rhs)),
                                                           _TORCH_TO_CODE[out_dtype], kernel, raster))


def tuning_get(rows_log2, k, n, num_total_groups, transpose_rhs, out_dtype):
    """(kernel, raster) recorded for a problem class; kernel is KERNEL_AUTO if none."""
    kern, ras = ctypes.c_int(0), ctypes.c_int(0)
    _check("gmm_tuning_get", load_library().gmm_tuning_get(rows_log2, k, n, num_total_groups, int(bool(transpose_rhs)),
                                                           _TORCH_TO_CODE[out_dtype], ctypes.byref(kern),
                                                           ctypes.byref(ras)))
    return kern.value, ras.value


def tuning_clear():
    _check("gmm_tuning_clear", load_library().gmm_tuning_clear())


def tuning_save(path: str):
    _check("gmm_tuning_save", load_library().gmm_tuning_save(os.fsencode(path)))


def tuning_load(path: str):
    _check("gmm_tuning_load", load_library().gmm_tuning_load(os.fsencode(path)))


def tune(lhs, rhs, group_sizes, rhs_bias=None, transpose_rhs=True, group_offset=0, out=None,
         out_dtype=torch.bfloat16, iterations=10, workspace=None, stream=None):
    """Times every bf16 kernel choice on this problem (writing `out`), records the fastest in the
    tiling table and returns (kernel, raster, mean ms)."""
    lib = load_library()
    _dev(lhs, "lhs"), _dev(rhs, "rhs"), _dev(group_sizes, "group_sizes")
    m, k = lhs.shape
    n = rhs.shape[1] if transpose_rhs else rhs.shape[2]
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=lhs.device)
    _dev(out, "out")
    ws = workspace if workspace is not None else workspace_for(lhs.device, stream)
    kern, ras, ms = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_float(0)
    rc = lib.gmm_tune(lhs.data_ptr(), _code(lhs), m, k, rhs.data_ptr(), _code(rhs), rhs.shape[0], n,
                      int(bool(transpose_rhs)), group_sizes.data_ptr(), group_sizes.shape[0], int(group_offset),
                      None if rhs_bias is None else rhs_bias.data_ptr(), 0 if rhs_bias is None else _code(rhs_bias),
                      out.data_ptr(), _code(out), ws.data_ptr(), ws.numel(), _stream(lhs.device, stream),
                      int(iterations), ctypes.byref(kern), ctypes.byref(ras), ctypes.byref(ms))
    _check("gmm_tune", rc)
    return kern.value, ras.value, ms.value


def get_device_error(device=None, workspace=None, stream=None) -> int:
    """Synchronises the stream and returns the device's report as one status (0 = none),
    clearing the flags (gmm_get_device_error)."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = workspace if workspace is not None else workspace_for(dev, stream)
    return int(lib.gmm_get_device_error(ws.data_ptr(), _stream(dev, stream)))


def read_device_errors(device=None, workspace=None, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the sticky device error flags."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = workspace if workspace is not None else workspace_for(dev, stream)
    flags = ctypes.c_uint32(0)
    rc = lib.gmm_read_device_errors(ws.data_ptr(), _stream(dev, stream), ctypes.byref(flags))
    if rc != 0:
        raise GmmError("gmm_read_device_errors", rc)
    return int(flags.value)
