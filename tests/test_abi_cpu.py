"""The C-ABI library builds, loads and exports every symbol include/libgmm.h declares,
and rejects bad host-side arguments before touching the device (no GPU needed)."""

import ctypes
import os
import re

import pytest
import torch

import moe_grouped_matrix_gb300 as G
from moe_grouped_matrix_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "libgmm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return G.load_library()


def test_header_declares_the_expected_calls():
    assert declared_functions() == sorted(
        ["gmm", "tgmm", "gmm_workspace_bytes", "gmm_read_device_errors", "gmm_status_string", "gmm_last_cuda_error",
         "gmm_noalloc", "gmm_into", "tgmm_local", "gmm_device_offset", "gmm_tuning_set", "gmm_tuning_get",
         "gmm_tuning_clear", "gmm_tuning_save", "gmm_tuning_load", "gmm_tune", "gmm_quantize_e4m3", "gmm_ex",
         "tgmm_ex", "gmm_get_device_error", "gmm_workspace_bytes_for"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in G.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert lib.gmm_status_string(0) == b"ok"
    for code in range(1, 12):
        assert lib.gmm_status_string(code) != b"unknown status"
    assert lib.gmm_status_string(12) == b"unknown status"
    # the error flags (256 bytes, the smallest workspace a call accepts), then scratch
    assert lib.gmm_workspace_bytes() > 256 and lib.gmm_workspace_bytes() % 256 == 0


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first


def call_gmm(lib, fn="gmm", **over):
    a = dict(lhs=FAKE, lhs_dtype=0, m=256, k=128, rhs=FAKE, rhs_dtype=0, L=4, n=256, trhs=1, gs=FAKE, G=4, go=0,
             scale=None, nb=0, bias=None, bias_dtype=0, out=FAKE, out_dtype=0, ws=FAKE, ws_bytes=256, stream=None)
    a.update(over)
    return getattr(lib, fn)(a["lhs"], a["lhs_dtype"], a["m"], a["k"], a["rhs"], a["rhs_dtype"], a["L"], a["n"], a["trhs"],
                                a["gs"], a["G"], a["go"], a["scale"], a["nb"], a["bias"], a["bias_dtype"],
                                a["out"], a["out_dtype"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(lhs=None), 1), (dict(gs=None), 1), (dict(out=None), 1),
    (dict(lhs_dtype=1), 2), (dict(rhs_dtype=1), 2), (dict(out_dtype=2), 2), (dict(rhs_dtype=2, trhs=0), 2),
    (dict(bias=FAKE, bias_dtype=2), 2),
    (dict(k=100), 3), (dict(n=12), 3), (dict(m=-1), 3), (dict(L=5), 3), (dict(G=0), 3), (dict(G=2000, L=4), 3),
    (dict(scale=FAKE, nb=3), 3), (dict(scale=FAKE, nb=2, k=128), 3), (dict(rhs_dtype=2, k=200), 3),
    (dict(scale=FAKE, nb=1, trhs=0), 2), (dict(rhs_dtype=8), 2), (dict(rhs_dtype=5, trhs=0), 2),
    (dict(rhs_dtype=4, trhs=0), 2), (dict(rhs_dtype=7, k=200), 3), (dict(rhs_dtype=3, k=192, scale=FAKE, nb=2), 3),
    (dict(G=8, L=4, go=5), 5), (dict(G=8, L=4, go=-1), 5),
    (dict(lhs=ctypes.c_void_p((1 << 20) + 8)), 4), (dict(out=ctypes.c_void_p((1 << 20) + 4)), 4),
    (dict(ws=None), 6), (dict(ws_bytes=8), 6), (dict(ws_bytes=255), 6),
])
@pytest.mark.parametrize("fn", ["gmm", "gmm_into"])
def test_gmm_host_validation(lib, fn, over, status):
    assert call_gmm(lib, fn, **over) == status


def call_gmm_ex(lib, **over):
    a = dict(lhs=FAKE, lhs_dtype=2, lscale=FAKE, nlb=2, m=256, k=256, rhs=FAKE, rhs_dtype=2, L=4, n=256, trhs=1,
             gs=FAKE, G=4, go=0, godev=None, scale=FAKE, scale_dtype=8, nb=2, bscale=None, bscale_dtype=8, bsize=0,
             bias=None, bias_dtype=0, out=FAKE, out_dtype=0, keep=0, options=None, ws=FAKE, ws_bytes=256,
             stream=None)
    a.update(over)
    return lib.gmm_ex(*a.values())


@pytest.mark.parametrize("over,status", [
    (dict(lhs=None), 1), (dict(out=None), 1),
    (dict(rhs_dtype=0), 2),                         # e4m3 activations need 8- or 4-bit weights
    (dict(lhs_dtype=0), 2),                         # lhs_scale with bf16 activations
    (dict(lhs_dtype=1, lscale=None), 2),
    (dict(scale_dtype=0), 2), (dict(scale_dtype=2), 2),
    (dict(lhs_dtype=0, lscale=None, rhs_dtype=0), 2),  # E8M0 scales with bf16 weights
    (dict(trhs=0), 2),
    (dict(nlb=0), 3), (dict(nlb=3), 3), (dict(nlb=4), 3),  # lhs blocks must be 128-multiples wide
    (dict(nb=4), 3), (dict(k=200), 3),
    (dict(lscale=ctypes.c_void_p((1 << 20) + 2)), 4), (dict(godev=ctypes.c_void_p((1 << 20) + 2)), 4),
    (dict(G=8, go=5), 5),
    (dict(ws=None), 6),
    # microscaling block scales: MXFP8 only (e4m3 weights, E8M0 per 32, bf16 activations)
    (dict(lhs_dtype=0, lscale=None, scale_dtype=1, bscale=FAKE, bsize=32, rhs_dtype=3), 2),
    (dict(lhs_dtype=0, lscale=None, scale_dtype=1, bscale=FAKE, bsize=32, bscale_dtype=2), 2),
    (dict(bscale=FAKE, bsize=32), 2),                                     # e4m3 activations
    (dict(lhs_dtype=0, lscale=None, scale_dtype=1, bscale=FAKE, bsize=16), 3),
    (dict(lhs_dtype=0, lscale=None, scale_dtype=1, bscale=FAKE, bsize=32, rhs_dtype=7, bscale_dtype=2), 3),
    (dict(lhs_dtype=0, lscale=None, scale_dtype=1, bscale=FAKE, bsize=16, rhs_dtype=7, bscale_dtype=8), 2),
])
def test_gmm_ex_host_validation(lib, over, status):
    assert call_gmm_ex(lib, **over) == status


def opts(**kw):
    return ctypes.byref(G._make_options(**kw))


def test_options_layout():
    # gmm_options: four int32 choices, an int64 wait bound, the drop-stage test hook, a reserved word
    assert ctypes.sizeof(G.GmmOptions) == 32
    assert G.GmmOptions.wait_limit_cycles.offset == 16 and G.GmmOptions.test_drop_stage.offset == 24


@pytest.mark.parametrize("over", [
    dict(bf16_kernel=5), dict(bf16_kernel=-1), dict(e4m3_kernel=3), dict(act_split=3), dict(tgmm_kernel=3),
    dict(wait_limit_cycles=-5), dict(test_drop_stage=-1)])
def test_bad_options_are_rejected(lib, over):
    # checked before anything else reads the (fake) pointers: GMM_ERR_SHAPE
    assert call_gmm_ex(lib, lhs_dtype=0, lscale=None, rhs_dtype=0, scale=None, nb=0, options=opts(**over)) == 3
    bad = G._make_options()
    bad.reserved = 1
    assert call_gmm_ex(lib, lhs_dtype=0, lscale=None, rhs_dtype=0, scale=None, nb=0, options=ctypes.byref(bad)) == 3


def test_options_reach_the_checks(lib):
    # the e4m3 decoding kernel takes neither e4m3 activations nor E8M0 scales (GMM_ERR_DTYPE)
    assert call_gmm_ex(lib, options=opts(e4m3_kernel="decode")) == 2
    # the split pass is requested but the workspace (256 bytes) cannot hold it: GMM_ERR_WORKSPACE,
    # unless the device check comes first (GMM_ERR_ARCH / GMM_ERR_CUDA on a machine without a GB300)
    st = call_gmm_ex(lib, lhs_dtype=0, lscale=None, scale_dtype=1, options=opts(act_split="pass"))
    assert st in (6, 7, 8)


def test_workspace_bytes_for(lib):
    f = lib.gmm_workspace_bytes_for
    assert f(256, 4096, 2048, 64, 64, G.DTYPE_BF16, G.DTYPE_BF16) == 256          # bf16 weights: flags only
    assert f(256, 4096, 2048, 64, 64, G.DTYPE_E4M3, G.DTYPE_E4M3) == 256          # e4m3 activations
    # bf16 activations, e4m3 weights: 4 m k bytes of split terms, then (s1, s2) per 256-wide step
    assert f(256, 4096, 2048, 64, 64, G.DTYPE_BF16, G.DTYPE_E4M3) == 256 + 4 * 256 * 4096 + 8 * 256 * 16
    # int8 / int4 weights: the fp16 split, 2 m k bytes rounded up to 256, then (scale, mark) per
    # 128-wide step
    assert f(3, 640, 128, 1, 1, G.DTYPE_BF16, G.DTYPE_INT8) == 256 + 3840 + 8 * 3 * 5
    assert f(5, 640, 128, 1, 1, G.DTYPE_BF16, G.DTYPE_INT4) == 256 + 6400 + 8 * 5 * 5  # 6656 is 256-aligned
    # uint4 stays on the e4m3 split: 4 m k bytes, then (s1, s2) per 256-wide step
    assert f(5, 640, 128, 1, 1, G.DTYPE_BF16, G.DTYPE_UINT4) == 256 + 12800 + 8 * 5 * 3
    assert f(-1, 128, 128, 1, 1, G.DTYPE_BF16, G.DTYPE_E4M3) == 0
    assert f(256, 4096, 2048, 64, 64, G.DTYPE_BF16, G.DTYPE_E4M3) > lib.gmm_workspace_bytes() // 8


def test_device_error_needs_a_workspace(lib):
    assert lib.gmm_get_device_error(None, None) == 1


def test_quantize_host_validation(lib):
    q = lambda **o: lib.gmm_quantize_e4m3(o.get("x", FAKE), o.get("xd", 0), o.get("m", 4), o.get("k", 256),
                                          o.get("group", 128), o.get("q", FAKE), o.get("s", FAKE), None)
    assert q(x=None) == 1 and q(q=None) == 1 and q(s=None) == 1
    assert q(xd=1) == 2 and q(xd=2) == 2
    assert q(group=32) == 3 and q(group=96) == 3 and q(k=320) == 3 and q(m=-1) == 3
    assert q(x=ctypes.c_void_p((1 << 20) + 2)) == 4 and q(s=ctypes.c_void_p((1 << 20) + 2)) == 4


def test_tgmm_host_validation(lib):
    t = lambda **o: lib.tgmm(o.get("lhs", FAKE), o.get("ld", 0), o.get("dout", FAKE), o.get("dd", 0), o.get("m", 64),
                             o.get("k", 128), o.get("n", 256), o.get("gs", FAKE), o.get("G", 4), o.get("out", FAKE),
                             o.get("od", 1), o.get("ws", FAKE), o.get("wb", 256), None)
    assert t(lhs=None) == 1
    assert t(ld=2) == 2
    assert t(od=2) == 2
    assert t(k=12) == 3
    assert t(G=0) == 3
    assert t(out=ctypes.c_void_p((1 << 20) + 2)) == 4
    assert t(wb=0) == 6


def test_tgmm_ex_options(lib):
    t = lambda o: lib.tgmm_ex(FAKE, 0, FAKE, 0, 64, 128, 256, FAKE, 8, 2, 4, FAKE, 1, o, FAKE, 256, None)
    assert t(opts(tgmm_kernel=3)) == 3
    assert t(opts(bf16_kernel=7)) == 3


def test_tgmm_local_host_validation(lib):
    t = lambda **o: lib.tgmm_local(o.get("lhs", FAKE), 0, FAKE, 0, o.get("m", 64), 128, 256, o.get("gs", FAKE),
                                   o.get("G", 8), o.get("go", 2), o.get("L", 4), o.get("out", FAKE), 1, FAKE, 256,
                                   None)
    assert t(lhs=None) == 1
    assert t(gs=None) == 1
    assert t(L=0) == 3
    assert t(L=9) == 3
    assert t(G=2000, L=4) == 3
    assert t(go=5) == 5
    assert t(go=-1) == 5
    assert t(out=ctypes.c_void_p((1 << 20) + 4)) == 4


# ------------------------------------------------------------------ tiling table (host only)
def test_tiling_table_set_get_save_load(lib, tmp_path):
    G.tuning_clear()
    assert G.tuning_get(7, 4096, 28672, 8, True, torch.bfloat16) == (G.KERNEL_AUTO, 0)
    G.tuning_set(7, 4096, 28672, 8, True, torch.bfloat16, G.KERNEL_SINGLE, 16)
    G.tuning_set(3, 2048, 2048, 128, False, torch.float32, G.KERNEL_SWAP)
    G.tuning_set(9, 1024, 2048, 16, True, torch.bfloat16, G.KERNEL_PAIR, -8)  # group-major blocks of 8 m tiles
    assert G.tuning_get(7, 4096, 28672, 8, True, torch.bfloat16) == (G.KERNEL_SINGLE, 16)
    assert G.tuning_get(9, 1024, 2048, 16, True, torch.bfloat16) == (G.KERNEL_PAIR, -8)
    assert G.tuning_get(7, 4096, 28672, 8, False, torch.bfloat16) == (G.KERNEL_AUTO, 0)
    path = tmp_path / "table.txt"
    G.tuning_save(str(path))
    lines = path.read_text().splitlines()
    assert lines[0] == "# libgmm tiling table 1"
    assert sorted(lines[1:]) == sorted(["7 4096 28672 8 1 0 4 16", "3 2048 2048 128 0 1 3 0", "9 1024 2048 16 1 0 1 -8"])
    G.tuning_clear()
    assert G.tuning_get(3, 2048, 2048, 128, False, torch.float32) == (G.KERNEL_AUTO, 0)
    G.tuning_load(str(path))
    assert G.tuning_get(3, 2048, 2048, 128, False, torch.float32) == (G.KERNEL_SWAP, 0)
    assert G.tuning_get(7, 4096, 28672, 8, True, torch.bfloat16) == (G.KERNEL_SINGLE, 16)
    assert G.tuning_get(9, 1024, 2048, 16, True, torch.bfloat16) == (G.KERNEL_PAIR, -8)
    G.tuning_clear()


@pytest.mark.parametrize("body", ["7 4096 28672 8 1 0 9 0\n", "7 4096 28672 8 1 0 1\n", "7 4096 x 8 1 0 1 0\n",
                                  "7 4096 28672 8 1 0 1 65\n", "7 4096 28672 8 1 0 1 -65\n",
                                  "7 4096 28672 8 1 0 1 0 extra\n"])
def test_tiling_table_rejects_malformed_files(lib, tmp_path, body):
    G.tuning_clear()
    good = "3 2048 2048 128 0 1 3 0\n"
    path = tmp_path / "bad.txt"
    path.write_text("# libgmm tiling table 1\n" + good + body)
    assert lib.gmm_tuning_load(str(path).encode()) == 9
    assert G.tuning_get(3, 2048, 2048, 128, False, torch.float32) == (G.KERNEL_AUTO, 0), "nothing added"
    path.write_text("no header\n" + good)
    assert lib.gmm_tuning_load(str(path).encode()) == 9
    assert lib.gmm_tuning_load(str(tmp_path / "missing.txt").encode()) == 9


def test_tiling_table_rejects_bad_entries(lib):
    assert lib.gmm_tuning_set(7, 4096, 4096, 8, 1, 0, 0, 0) == 3   # AUTO is not an entry
    assert lib.gmm_tuning_set(7, 4096, 4096, 8, 1, 0, 5, 0) == 3
    assert lib.gmm_tuning_set(7, 4096, 4096, 8, 1, 0, 1, 99) == 3
    assert lib.gmm_tuning_set(7, 4096, 4096, 8, 1, 0, 1, -65) == 3
    assert lib.gmm_tuning_set(-1, 4096, 4096, 8, 1, 0, 1, 0) == 3
    assert G.tuning_rows_log2(16384, 8) == 11 and G.tuning_rows_log2(5, 8) == 0 and G.tuning_rows_log2(32768, 128) == 8
