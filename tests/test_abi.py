"""The C-ABI library loads and exports every symbol include/hb.h declares;
argument errors are reported synchronously (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from chunked_prefill_hybrid_tau_gb300 import _lib as L
from chunked_prefill_hybrid_tau_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "hb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(hb_\w+)\s*\(", src, flags=re.M)))


def test_header_lists_the_boundary():
    names = header_functions()
    for required in ["hb_plan_batch", "hb_kv_append", "hb_attention", "hb_layer_forward"]:
        assert required in names
    assert set(names) == set(L.PROTOTYPES), set(names) ^ set(L.PROTOTYPES)


def test_library_exports_every_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    assert lib.hb_version() >= 100
    assert lib.hb_status_string(0) == b"ok"
    assert lib.hb_status_string(3) == b"out of KV pages"


def test_library_is_in_tree(lib):
    path = L.library_path()
    assert os.path.commonpath([path, ROOT]) == ROOT
    assert os.path.exists(path)


def test_argument_errors_are_synchronous(lib):
    # null operands are rejected before any device work
    st = lib.hb_gemm(None, None, None, None, 128, 128, 128, 0, None)
    assert st == L.HB_ERR_INVALID_ARG
    assert b"null" in lib.hb_last_error()
    st = lib.hb_gemm(C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), None, 128, 100, 128, 0, None)
    assert st == L.HB_ERR_INVALID_ARG  # N not a multiple of 64
    bad = L.hb_layer_dims(256, 4, 3, 64, 688, 16, 1e-6, 1e4)  # n_q % n_kv != 0
    st = lib.hb_kv_append(None, 0, None, None, None, 1, C.byref(bad), None, None, None, 1, None)
    assert st == L.HB_ERR_INVALID_ARG
    # the wait self-test checks its limit before touching a device
    assert lib.hb_selftest_wait_timeout(0, None) == L.HB_ERR_INVALID_ARG
    assert lib.hb_selftest_wait_timeout(1000001, None) == L.HB_ERR_INVALID_ARG
    with pytest.raises(B.HBError):
        B._check(L.HB_ERR_INVALID_ARG, "x")


def test_workspace_sizes(lib):
    import workloads as wl
    ds = B.dims_struct(wl.MISTRAL)
    a = lib.hb_attention_workspace_bytes(C.byref(ds), 512, 33, 4097)
    assert a > 0 and a % 256 == 0
    w = lib.hb_layer_workspace_bytes(C.byref(ds), 512, 33, 4097)
    assert w > a + 512 * 4096 * 2 * 5
