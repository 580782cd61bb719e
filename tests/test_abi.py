"""CPU checks of the C ABI: the library builds, loads, exports every function
that include/*.h declares, and rejects bad arguments on the host before any
device work (these calls never touch a GPU)."""
import ctypes
import os
import re

import pytest

import block_sparse_spatio_gb300 as bss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(bss_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from block_sparse_spatio_gb300 import build
    build.build()
    return bss.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(bss.EXPORTED)


def test_status_strings(lib):
    assert lib.bss_status_string(0) == b"BSS_OK"
    assert lib.bss_status_string(4) == b"BSS_ERR_TIMEOUT"
    assert lib.bss_version() >= 100


def _params(**kw):
    base = dict(F=8, Hs=16, Ws=24, head_dim=128, spatial_frame_window=2, temporal_raster_window=40)
    base.update(kw)
    return bss.MaskParams(**base).c()


@pytest.mark.parametrize("kw,code", [
    (dict(F=0), 1), (dict(Hs=-1), 1), (dict(head_dim=96), 2), (dict(spatial_frame_window=-1), 1),
    (dict(sink_frames=2), 2), (dict(rounding=3), 1), (dict(rounding=-1), 1), (dict(temporal_permuted=2), 1),
])
def test_build_tile_map_rejects_bad_params(lib, kw, code):
    h = ctypes.c_void_p()
    p = _params(**kw)
    assert lib.bss_build_tile_map(ctypes.byref(p), 128, 128, ctypes.byref(h), None) == code
    assert h.value is None
    assert lib.bss_last_error_message() != b""


def test_build_tile_map_rejects_bad_tiles_and_null(lib):
    h = ctypes.c_void_p()
    p = _params()
    assert lib.bss_build_tile_map(ctypes.byref(p), 8, 128, ctypes.byref(h), None) == 1
    assert lib.bss_build_tile_map(ctypes.byref(p), 128, 0, ctypes.byref(h), None) == 1
    assert lib.bss_build_tile_map(None, 128, 128, ctypes.byref(h), None) == 1
    assert lib.bss_build_tile_map(ctypes.byref(p), 128, 128, None, None) == 1


def test_calls_with_stale_or_null_handles(lib):
    bogus = ctypes.c_void_p(0x1234)
    out = (ctypes.c_int64 * 7)()
    assert lib.bss_tile_map_stats(bogus, 0, out) == 1
    assert lib.bss_tile_map_stats(None, 0, out) == 1
    dims = (ctypes.c_int32 * 4)()
    assert lib.bss_tile_map_dims(bogus, 0, dims) == 1
    assert lib.bss_tile_map_copy_csr(bogus, 0, None, None) == 1
    x = ctypes.c_void_p(0x10000)
    assert lib.bss_sparse_attention(x, x, x, x, None, bogus, None, 2, 0.0, None) == 1
    lib.bss_destroy_tile_map(None)
    lib.bss_destroy_tile_map(bogus)  # unknown handles are ignored


def test_permute_rejects_bad_pointers(lib):
    p = _params()
    a, b = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20008)
    assert lib.bss_permute(None, a, None, 2, ctypes.byref(p), 0, None) == 1
    assert lib.bss_permute(a, b, None, 2, ctypes.byref(p), 0, None) == 1          # misaligned
    assert lib.bss_permute(a, ctypes.c_void_p(0x10010), None, 2, ctypes.byref(p), 0, None) == 1  # overlap
    assert lib.bss_permute(a, ctypes.c_void_p(0x1000000000), None, 0, ctypes.byref(p), 0, None) == 1  # H
    assert lib.bss_permute(a, ctypes.c_void_p(0x1000000000), None, 2, ctypes.byref(p), 5, None) == 1  # inverse


def test_dense_attention_rejects_bad_args(lib):
    a = ctypes.c_void_p(0x10000)
    assert lib.bss_dense_attention(None, a, a, a, None, 1, 256, 128, 0.0, None) == 1
    assert lib.bss_dense_attention(a, a, a, ctypes.c_void_p(0x10004), None, 1, 256, 128, 0.0, None) == 1
    assert lib.bss_dense_attention(a, a, a, a, None, 0, 256, 128, 0.0, None) == 1
    assert lib.bss_dense_attention(a, a, a, a, None, 1, 256, 80, 0.0, None) == 2
    assert lib.bss_dense_attention(a, a, a, a, None, 1, 256, 128, float("nan"), None) == 1


def test_diag_rejects_bad_args(lib):
    a = ctypes.c_void_p(0x10000)
    assert lib.bss_diag_mma_tile(None, a, a, a, a, a, 128, None) == 1
    assert lib.bss_diag_mma_tile(a, a, a, a, a, a, 32, None) == 2


def test_product_package_does_not_import_oracle():
    import ast
    pkg = os.path.join(ROOT, "block_sparse_spatio_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith(".py"):
                tree = ast.parse(open(os.path.join(dirpath, fn)).read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert all(not a.name.startswith("oracle") for a in node.names), fn
                    if isinstance(node, ast.ImportFrom):
                        assert not (node.module or "").startswith("oracle"), fn
            if fn.endswith((".cu", ".cuh", ".h")):
                assert "oracle" not in open(os.path.join(dirpath, fn)).read().lower(), fn


def test_noalloc_rejects_oversized_and_bad_buffers(lib):
    # host-side checks only: nothing is launched and no device is touched
    a = ctypes.c_void_p(0x10000)
    big = bss.MaskParams(F=21, Hs=180, Ws=320, head_dim=128, spatial_frame_window=3,
                         temporal_raster_window=2450).c()
    assert lib.bss_build_tile_map_csr_noalloc(ctypes.byref(big), 0, 128, 128, a, a, 1 << 40, a, None) == 2
    assert b"scratch" in lib.bss_last_error_message()
    small = _params()
    assert lib.bss_build_tile_map_csr_noalloc(ctypes.byref(small), 0, 128, 128, None, a, 1 << 20, a, None) == 1
    assert lib.bss_build_tile_map_csr_noalloc(ctypes.byref(small), 2, 128, 128, a, a, 1 << 20, a, None) == 1
    assert lib.bss_build_tile_map_csr_noalloc(ctypes.byref(small), 0, 128, 128, a, a, 10, a, None) == 1
    assert lib.bss_build_tile_map_csr_noalloc(ctypes.byref(small), 0, 128, 128, a, a, 1 << 20,
                                              ctypes.c_void_p(0x10004), None) == 1


@pytest.mark.parametrize("limit", [0, 999, 1_000_000_001, -5])
def test_wait_timeout_diag_rejects_limits_before_any_launch(lib, limit):
    assert lib.bss_diag_wait_timeout(limit, None, None) == 1  # BSS_ERR_INVALID_ARG


def test_permute_flagged_needs_flags(lib):
    p = _params()
    buf = ctypes.c_void_p(16)  # never dereferenced: the call is rejected on the host
    assert lib.bss_permute_flagged(buf, ctypes.c_void_p(1 << 40), None, 2, ctypes.byref(p), 0, None) == 1


def _cuda_include():
    for root in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime_api.h")):
            return os.path.join(root, "include")
    pytest.skip("no CUDA headers")


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_headers_compile_as_plain_c_and_cxx_and_link(lib, tmp_path, lang):
    """A program that includes only include/*.h, takes the address of every
    declared entry point, and calls host-side ones, builds with gcc / g++ and
    links against the shared library: the headers are the whole interface."""
    import shutil
    import subprocess
    cc = "gcc" if lang == "c99" else "g++"
    if shutil.which(cc) is None:
        pytest.skip(f"no {cc}")
    names = declared_functions()
    table = "\n".join(f"    (fnptr)&{n}," for n in names)
    src = f"""#include <stdio.h>
#include "bss.h"
#include "bss_diag.h"

typedef void (*fnptr)(void);
static const fnptr every_entry_point[] = {{
{table}
}};

int main(void) {{
    bss_tile_map h = 0;
    bss_status st = bss_build_tile_map(NULL, 128, 128, &h, 0);
    printf("%d %d %s %s %d\\n", (int)(sizeof(every_entry_point) / sizeof(every_entry_point[0])), bss_version(),
           bss_status_string(BSS_ERR_TIMEOUT), bss_status_string(st), h == 0);
    return st == BSS_ERR_INVALID_ARG ? 0 : 1;
}}
"""
    prog = tmp_path / "prog.c"
    prog.write_text(src)
    libdir = os.path.dirname(lib._name)
    flags = ["-std=c99"] if lang == "c99" else ["-std=c++17", "-x", "c++"]
    cmd = [cc, *flags, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", _cuda_include(),
           str(prog), "-L", libdir, "-lbss", f"-Wl,-rpath,{libdir}", "-o", str(tmp_path / "prog")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(tmp_path / "prog")], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split() == [str(len(names)), str(lib.bss_version()), "BSS_ERR_TIMEOUT", "BSS_ERR_INVALID_ARG", "1"]


def test_route_heads_rejects_bad_args_before_any_launch(lib):
    p, bad = _params(), _params(head_dim=96)
    a, r, f, e = (ctypes.c_void_p(x) for x in (0x10000, 0x20000, 0x30000, 0x40000))
    pp = ctypes.byref(p)
    assert lib.bss_route_heads(a, a, a, 2, None, r, 4, f, e, None) == 1                  # no params
    assert lib.bss_route_heads(a, a, a, 2, ctypes.byref(bad), r, 4, f, e, None) == 2     # head_dim
    assert lib.bss_route_heads(None, a, a, 2, pp, r, 4, f, e, None) == 1                 # NULL Q
    assert lib.bss_route_heads(a, a, a, 2, pp, None, 4, f, e, None) == 1                 # NULL rows
    assert lib.bss_route_heads(a, a, a, 2, pp, r, 4, None, e, None) == 1                 # NULL flags
    assert lib.bss_route_heads(a, a, a, 2, pp, r, 4, f, None, None) == 1                 # NULL errors
    assert lib.bss_route_heads(ctypes.c_void_p(0x10008), a, a, 2, pp, r, 4, f, e, None) == 1  # Q misaligned
    assert lib.bss_route_heads(a, a, a, 2, pp, ctypes.c_void_p(0x20002), 4, f, e, None) == 1  # rows misaligned
    assert lib.bss_route_heads(a, a, a, 0, pp, r, 4, f, e, None) == 1                    # H
    assert lib.bss_route_heads(a, a, a, 2, pp, r, 0, f, e, None) == 1                    # R
    assert lib.bss_last_error_message() != b""


def test_split_and_fused_attention_reject_bad_args_before_any_launch(lib):
    a, m = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x1234)
    # the temporal heads' buffers: NULL or misaligned
    assert lib.bss_sparse_attention_split(a, a, a, a, None, a, a, None, None, m, None, 2, 0.0, None) == 1
    assert lib.bss_sparse_attention_split(a, a, a, a, a, a, ctypes.c_void_p(0x10004), None, None, m, None, 2,
                                          0.0, None) == 1
    assert lib.bss_sparse_attention_split(a, a, a, a, a, a, a, ctypes.c_void_p(0x10004), None, m, None, 2,
                                          0.0, None) == 1
    # a map handle the library did not hand out
    assert lib.bss_sparse_attention_split(a, a, a, a, a, a, a, None, None, m, None, 2, 0.0, None) == 1
    assert lib.bss_sparse_attention_fused(a, a, a, a, None, m, None, 2, 0.0, None) == 1
    assert lib.bss_sparse_attention_fused(a, a, a, a, None, None, None, 2, 0.0, None) == 1


def test_step_calls_reject_bad_args_before_any_device_work(lib):
    bogus = ctypes.c_void_p(0x1234)
    x = ctypes.c_void_p(0x10000)
    p = _params()
    assert lib.bss_attention_step(x, x, x, x, None, bogus, None, 2, None, None, None, None) == 1
    assert lib.bss_attention_step(x, x, x, x, None, None, None, 2, None, None, None, None) == 1
    out = ctypes.c_void_p()
    assert lib.bss_step_workspace_create(ctypes.byref(p), 0, 3, 1, ctypes.byref(out)) == 1        # H
    assert lib.bss_step_workspace_create(ctypes.byref(p), 4, 0, 1, ctypes.byref(out)) == 1        # depth
    assert lib.bss_step_workspace_create(ctypes.byref(p), 4, 9, 1, ctypes.byref(out)) == 1
    assert lib.bss_step_workspace_create(ctypes.byref(p), 4, 3, 5, ctypes.byref(out)) == 1        # group
    assert lib.bss_step_workspace_create(ctypes.byref(p), 4, 3, 0, ctypes.byref(out)) == 1
    assert lib.bss_step_workspace_create(ctypes.byref(p), 4, 3, 1, None) == 1
    bad = _params(head_dim=96)
    assert lib.bss_step_workspace_create(ctypes.byref(bad), 4, 3, 1, ctypes.byref(out)) == 2
    assert out.value is None
    assert lib.bss_attention_step_host(x, x, x, x, x, bogus, bogus, None, None) == 1
    assert lib.bss_step_workspace_wait_stream(bogus, None) == 1
    lib.bss_step_workspace_destroy(None)
    lib.bss_step_workspace_destroy(bogus)  # unknown handles are ignored


def test_permute_flagged_multi_rejects_bad_args(lib):
    p = _params()
    a = [ctypes.c_void_p(0x10000 + i * 0x10000000) for i in range(6)]
    arr = lambda *xs: (ctypes.c_void_p * len(xs))(*xs)  # noqa: E731
    fl = ctypes.c_void_p(0x9000)
    ins, outs = arr(a[0], a[1], a[2]), arr(a[3], a[4], a[5])
    assert lib.bss_permute_flagged_multi(ins, outs, 0, fl, 2, ctypes.byref(p), 0, None) == 1   # count
    assert lib.bss_permute_flagged_multi(ins, outs, 4, fl, 2, ctypes.byref(p), 0, None) == 1
    assert lib.bss_permute_flagged_multi(ins, outs, 3, None, 2, ctypes.byref(p), 0, None) == 1  # flags
    assert lib.bss_permute_flagged_multi(None, outs, 3, fl, 2, ctypes.byref(p), 0, None) == 1
    assert lib.bss_permute_flagged_multi(ins, arr(a[3], a[1], a[5]), 3, fl, 2, ctypes.byref(p), 0, None) == 1
    assert lib.bss_permute_flagged_multi(ins, arr(a[3], a[3], a[5]), 3, fl, 2, ctypes.byref(p), 0, None) == 1
    assert lib.bss_permute_flagged_multi(ins, arr(a[3], ctypes.c_void_p(0x30000008), a[5]), 3, fl, 2,
                                         ctypes.byref(p), 0, None) == 1                        # misaligned
    assert lib.bss_permute_flagged_multi(ins, outs, 3, fl, 0, ctypes.byref(p), 0, None) == 1   # H
