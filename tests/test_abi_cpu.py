"""The C-ABI library builds, loads without a GPU, exports every function that
include/paged_kv.h declares, and rejects bad arguments on the host before
touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_236_gb300 import build
    build.build()
    import paged_kv_cache_236_gb300 as pkv
    return pkv.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"paged_kv_write", "paged_attention_forward", "paged_attention_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert b"sm_103a" in lib.pkv_version()


def test_workspace_sizes_are_host_arithmetic(lib):
    s = lib.paged_attention_workspace_size(64, 64, 32, 8, 128)
    m = lib.paged_attention_workspace_min(64, 64, 32, 8, 128)
    assert 0 < m < s
    assert lib.paged_attention_workspace_size(64, 64, 32, 0, 128) == 0


def test_host_checks_need_no_gpu(lib):
    # num_q_heads not a multiple of num_kv_heads: rejected before any CUDA call
    st = lib.paged_attention_forward(None, None, None, None, None, None, None, 1, 1, 6, 4, 128, 4, 16, 1, 0,
                                     ctypes.c_float(0.1), 1, 0, None, 0, 1, None)
    assert st == 1 and b"num_kv_heads" in lib.pkv_last_error()
    st = lib.paged_attention_forward(None, None, None, None, None, None, None, 1, 1, 8, 4, 96, 4, 16, 1, 0,
                                     ctypes.c_float(0.1), 1, 0, None, 0, 1, None)
    assert st == 2 and b"head_dim" in lib.pkv_last_error()
    st = lib.paged_attention_forward(None, None, None, None, None, None, None, 1, 1, 8, 4, 128, 4, 24, 1, 0,
                                     ctypes.c_float(0.1), 1, 0, None, 0, 1, None)
    assert st == 2 and b"block_size" in lib.pkv_last_error()
    st = lib.paged_attention_forward(None, None, None, None, None, None, None, 1, 1, 8, 4, 128, 4, 16, 1, 0,
                                     ctypes.c_float(0.1), 1, 0, None, 0, 7, None)
    assert st == 2
    # empty batches are no-ops
    assert lib.paged_attention_forward(None, None, None, None, None, None, None, 0, 0, 8, 4, 128, 4, 16, 1, 0,
                                       ctypes.c_float(0.1), 1, 0, None, 0, 1, None) == 0
    assert lib.paged_kv_write(None, None, None, None, None, 0, 4, 16, 4, 128, 0, 0, 1, None) == 0
    # bad token stride
    assert lib.paged_kv_write(None, None, None, None, None, 3, 4, 16, 4, 128, 100, 0, 1, None) == 1
    # null pointers with work to do
    assert lib.paged_kv_write(None, None, None, None, None, 3, 4, 16, 4, 128, 0, 0, 1, None) == 1


def test_fp8_host_checks_need_no_gpu(lib):
    import ctypes as C
    f = C.c_float
    # FP8 attention: scales must be positive, head_dim 128 only
    st = lib.paged_attention_forward_fp8kv(None, None, None, None, None, None, None, 1, 1, 8, 4, 128, 4, 16, 1, 0,
                                           f(0.1), 1, f(0.0), f(1.0), 0, None, 0, None)
    assert st == 1 and b"scale" in lib.pkv_last_error()
    st = lib.paged_attention_forward_fp8kv(None, None, None, None, None, None, None, 1, 1, 8, 4, 64, 4, 16, 1, 0,
                                           f(0.1), 1, f(1.0), f(1.0), 0, None, 0, None)
    assert st == 2 and b"head_dim" in lib.pkv_last_error()
    # an empty batch is a no-op
    assert lib.paged_attention_forward_fp8kv(None, None, None, None, None, None, None, 0, 0, 8, 4, 128, 4, 16, 1, 0,
                                             f(0.1), 1, f(1.0), f(1.0), 0, None, 0, None) == 0
    # FP8 write: scales, row multiple of 16, source dtype
    assert lib.paged_kv_write_fp8(None, None, None, None, None, 3, 4, 16, 4, 128, 0, 0, 1, f(-1.0), f(1.0), None) == 1
    assert lib.paged_kv_write_fp8(None, None, None, None, None, 3, 4, 16, 1, 8, 0, 0, 1, f(1.0), f(1.0), None) == 2
    assert lib.paged_kv_write_fp8(None, None, None, None, None, 3, 4, 16, 4, 128, 0, 0, 2, f(1.0), f(1.0), None) == 2
    assert lib.paged_kv_write_fp8(None, None, None, None, None, 0, 4, 16, 4, 128, 0, 0, 1, f(1.0), f(1.0), None) == 0


def test_headers_compile_as_plain_c(tmp_path):
    """The public headers are C: each compiles alone with a C99 compiler."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = tmp_path / f"use_{h}.c"
        src.write_text(f'#include "{h}"\nint main(void) {{ return 0; }}\n')
        r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                            "-I" + os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
        assert r.returncode == 0, (h, r.stderr)
