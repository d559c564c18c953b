"""The C-ABI library without a GPU: it loads, exports every entry point that
include/gf.h declares, and rejects invalid arguments before touching a device."""
import ctypes
import os
import re

import pytest

import gemm_epilogue_tmem_gb300 as gf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"GF_API\s+[\w\s\*]+?\b(gf_\w+)\s*\(", src)
    return names


@pytest.fixture(scope="module")
def L():
    gf.build()
    return gf.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"gf_matmul_plan", "gf_matmul_execute", "gf_plan_free"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {gf.LIB}").read().split()
    exported = {s for s in out if s.startswith("gf_")}
    assert exported == set(names)


def test_status_strings(L):
    for s in range(7):
        assert gf.gf_status_string(s).startswith("GF_")
    assert "unknown" in gf.gf_status_string(99)


@pytest.mark.parametrize("args,status", [
    ((-1, 8, 8, 0, 1, 0, 0), gf.GF_ERR_INVALID_VALUE),        # negative m
    ((8, 8, 8, 7, 1, 0, 0), gf.GF_ERR_INVALID_VALUE),         # dtype
    ((8, 8, 8, 0, 9, 0, 0), gf.GF_ERR_INVALID_VALUE),         # epilog
    ((8, 8, 8, 0, 1, 5, 0), gf.GF_ERR_INVALID_VALUE),         # bias axis
    ((8, 8, 8, 0, 1, 0, 3), gf.GF_ERR_INVALID_VALUE),         # b layout
    ((8, 12, 8, 0, 1, 0, 0), gf.GF_ERR_UNSUPPORTED),          # n % 8
    ((8, 8, 12, 0, 1, 0, 0), gf.GF_ERR_UNSUPPORTED),          # k % 8
    ((8, 8, 8, 0, 3, 1, 0), gf.GF_ERR_UNSUPPORTED),           # DRELU_BGRAD with a row bias
    ((1 << 31, 8, 8, 0, 1, 0, 0), gf.GF_ERR_INVALID_VALUE),   # m too large
])
def test_plan_rejects_before_device(L, args, status):
    h = L.gf_matmul_plan_ex(*args)
    assert not h
    assert L.gf_last_error() == status


def test_null_plan_calls(L):
    assert L.gf_matmul_execute(None, None, None, None, None, None, None, None, None) == \
        gf.GF_ERR_INVALID_VALUE
    assert L.gf_plan_status(None, None) == gf.GF_ERR_INVALID_VALUE
    assert L.gf_plan_set_option(None, 0, 0) == gf.GF_ERR_INVALID_VALUE
    assert L.gf_matmul_autotune(None, None, None, None, None, None, None, None, None, 3) == \
        gf.GF_ERR_INVALID_VALUE
    ks = ctypes.c_int32(-1)
    assert L.gf_plan_k_splits(None, ctypes.byref(ks)) == gf.GF_ERR_INVALID_VALUE
    assert ks.value == -1
    assert L.gf_plan_launches(None, ctypes.byref(ks)) == gf.GF_ERR_INVALID_VALUE
    assert ks.value == -1
    L.gf_plan_free(None)


def test_no_device_here(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = L.gf_matmul_plan(256, 256, 256, 0, 1, 0)
    assert not h and L.gf_last_error() == gf.GF_ERR_NO_DEVICE


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "gf.h"\nint main(void){ return (int)GF_OK + (int)sizeof(gf_status); }\n')
    rc = os.system(f"gcc -std=c99 -Wall -Werror -I{ROOT}/include -c {src} -o {tmp_path}/t.o")
    assert rc == 0


def test_noalloc_rejection_is_the_last_error(L):
    """A rejected gf_drelu_bgrad_noalloc is what gf_last_error reports (the
    checks run before any device is touched)."""
    assert L.gf_plan_set_option(None, 0, 0) == gf.GF_ERR_INVALID_VALUE
    assert L.gf_last_error() == gf.GF_ERR_INVALID_VALUE
    # n not a multiple of 8
    assert L.gf_drelu_bgrad_noalloc(8, 12, 8, 0, 1, None, None, None, None, None, None) == \
        gf.GF_ERR_UNSUPPORTED
    assert L.gf_last_error() == gf.GF_ERR_UNSUPPORTED
    # negative m
    assert L.gf_drelu_bgrad_noalloc(-1, 8, 8, 0, 1, None, None, None, None, None, None) == \
        gf.GF_ERR_INVALID_VALUE
    assert L.gf_last_error() == gf.GF_ERR_INVALID_VALUE
