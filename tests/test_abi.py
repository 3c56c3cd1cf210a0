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
    assert st == L.HB_ERR_INVALID_ARG  # N not a multiple of 8
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


def test_idle_iteration_is_a_no_op(lib):
    """An iteration with nothing planned (no decodes, no prompt tokens) is
    accepted and returns before any device work, so it runs without a GPU;
    the same call with one row would need the device."""
    import workloads as wl
    ds = B.dims_struct(wl.TINY)
    fake = C.c_void_p(4096)  # never dereferenced
    w = L.hb_layer_weights(fake, fake, fake, fake, None, None, None, None, L.HB_WEIGHTS_BF16)
    plan = L.hb_device_plan(0, 0, 1, None, None, None, None, None, 0, 0, 0)
    st = lib.hb_layer_forward(C.byref(w), C.byref(ds), C.byref(plan), fake, 64, fake, fake, fake, fake, 8, 64,
                              None, 0, None, None)
    assert st == L.HB_OK, lib.hb_last_error()
    # a planned row with null plan arrays is an argument error, found before the device
    plan.n_rows, plan.n_seqs = 1, 1
    st = lib.hb_layer_forward(C.byref(w), C.byref(ds), C.byref(plan), fake, 64, fake, fake, fake, fake, 8, 64,
                              None, 0, None, None)
    assert st == L.HB_ERR_INVALID_ARG and b"null plan array" in lib.hb_last_error()


def test_layer_stack_checks_every_layer_before_launching(lib):
    """hb_layers_forward validates all layers' arguments before any device
    work: an idle iteration is a no-op, and a bad later layer is an argument
    error (no GPU needed for either)."""
    import workloads as wl
    ds = B.dims_struct(wl.TINY)
    fake = C.c_void_p(4096)  # never dereferenced
    good = L.hb_layer_weights(fake, fake, fake, fake, None, None, None, None, L.HB_WEIGHTS_BF16)
    e4m3_no_scales = L.hb_layer_weights(fake, fake, fake, fake, None, None, None, None, L.HB_WEIGHTS_E4M3)
    plan = L.hb_device_plan(0, 0, 1, None, None, None, None, None, 0, 0, 0)
    ks = (C.c_void_p * 3)(4096, 4096, 4096)
    vs = (C.c_void_p * 3)(4096, 4096, 4096)

    def call(ws, n, k=ks, v=vs):
        return lib.hb_layers_forward(ws, n, C.byref(ds), C.byref(plan), fake, 64, fake, fake, k, v, 8, 64, None, 0,
                                     None)

    st = call((L.hb_layer_weights * 3)(good, good, good), 3)
    assert st == L.HB_OK, lib.hb_last_error()
    assert call((L.hb_layer_weights * 3)(good, good, good), 0) == L.HB_OK
    assert call((L.hb_layer_weights * 3)(good, good, e4m3_no_scales), 3) == L.HB_ERR_INVALID_ARG
    assert b"scales" in lib.hb_last_error()
    v_null = (C.c_void_p * 3)(4096, None, 4096)
    assert call((L.hb_layer_weights * 3)(good, good, good), 3, v=v_null) == L.HB_ERR_INVALID_ARG
    assert b"layer 1" in lib.hb_last_error()
    assert call((L.hb_layer_weights * 3)(good, good, good), -1) == L.HB_ERR_INVALID_ARG
    assert lib.hb_layers_forward(None, 1, C.byref(ds), C.byref(plan), fake, 64, fake, fake, ks, vs, 8, 64, None, 0,
                                 None) == L.HB_ERR_INVALID_ARG


def test_launch_counter_needs_no_device(lib):
    """hb_kernel_launches is readable without a GPU, and calls that fail
    their argument checks launch nothing."""
    n0 = lib.hb_kernel_launches()
    assert lib.hb_gemm(None, None, None, None, 128, 128, 128, 0, None) == L.HB_ERR_INVALID_ARG
    assert lib.hb_selftest_wait_timeout(0, None) == L.HB_ERR_INVALID_ARG
    assert lib.hb_kernel_launches() == n0
    assert B.hb_kernel_launches() == n0
