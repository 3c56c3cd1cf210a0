"""ctypes declarations of the C ABI in include/hb.h (structs and prototypes)."""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

i32 = C.c_int32
p_i32 = C.POINTER(C.c_int32)
vp = C.c_void_p


class hb_layer_dims(C.Structure):
    _fields_ = [("d_model", i32), ("n_q", i32), ("n_kv", i32), ("d_head", i32), ("d_ff", i32),
                ("page_size", i32), ("rms_eps", C.c_float), ("rope_theta", C.c_float)]


class hb_request(C.Structure):
    _fields_ = [("prompt_len", i32), ("done", i32), ("n_pages", i32), ("page_cap", i32), ("pages", p_i32)]


class hb_page_pool(C.Structure):
    _fields_ = [("pages", p_i32), ("count", i32), ("head", i32)]


class hb_plan(C.Structure):
    _fields_ = [("row_cap", i32), ("row_seq", p_i32), ("row_pos", p_i32), ("slot_mapping", p_i32),
                ("seq_cap", i32), ("seq_q_start", p_i32), ("seq_pos0", p_i32), ("seq_kv_len", p_i32),
                ("seq_kind", p_i32), ("seq_req", p_i32), ("max_pages", i32), ("block_table", p_i32),
                ("pf_cap", i32), ("pf_take", p_i32), ("pf_finished", p_i32),
                ("n_rows", i32), ("n_seqs", i32), ("n_decode_seqs", i32), ("pages_used", i32),
                ("over_budget", i32), ("need_rows", i32), ("need_seqs", i32), ("need_max_pages", i32),
                ("need_pages", i32), ("decode_pairs", C.c_int64), ("chunk_pairs", C.c_int64),
                ("chunk_rows", C.c_int64)]


class hb_device_plan(C.Structure):
    _fields_ = [("n_rows", i32), ("n_seqs", i32), ("max_pages", i32), ("row_pos", vp), ("slot_mapping", vp),
                ("seq_q_start", vp), ("seq_kv_len", vp), ("block_table", vp),
                ("decode_pairs", C.c_int64), ("chunk_pairs", C.c_int64), ("chunk_rows", C.c_int64)]


class hb_layer_weights(C.Structure):
    _fields_ = [("w_qkv", vp), ("w_o", vp), ("w_gu", vp), ("w_d", vp),
                ("s_qkv", vp), ("s_o", vp), ("s_gu", vp), ("s_d", vp), ("format", i32)]


class hb_profile(C.Structure):
    _fields_ = [("events", C.POINTER(vp)), ("n_events", i32)]


HB_LAYER_STAGES = 8
HB_EPI_STORE, HB_EPI_RESIDUAL, HB_EPI_SWIGLU, HB_EPI_F32 = 0, 1, 2, 3
HB_WEIGHTS_BF16, HB_WEIGHTS_E4M3 = 0, 1
HB_OK, HB_ERR_INVALID_ARG, HB_ERR_CAPACITY, HB_ERR_OUT_OF_PAGES = 0, 1, 2, 3
HB_ERR_CUDA, HB_ERR_TIMEOUT, HB_ERR_UNSUPPORTED, HB_ERR_DEVICE = 4, 5, 6, 7

# name -> (restype, argtypes); every symbol include/hb.h declares
PROTOTYPES = {
    "hb_status_string": (C.c_char_p, [C.c_int]),
    "hb_last_error": (C.c_char_p, []),
    "hb_version": (i32, []),
    "hb_plan_batch": (C.c_int, [C.POINTER(hb_request), i32, C.POINTER(hb_request), i32, C.POINTER(hb_page_pool),
                                i32, i32, i32, C.POINTER(hb_plan)]),
    "hb_sched_create": (C.c_int, [i32, i32, i32, p_i32, i32, C.POINTER(vp)]),
    "hb_sched_destroy": (None, [vp]),
    "hb_sched_add": (C.c_int, [vp, i32, i32, p_i32]),
    "hb_sched_plan": (C.c_int, [vp, C.POINTER(hb_plan), p_i32]),
    "hb_sched_commit": (C.c_int, [vp]),
    "hb_sched_info": (C.c_int, [vp, i32, p_i32, p_i32, p_i32, p_i32]),
    "hb_sched_active": (i32, [vp]),
    "hb_sched_free_pages": (i32, [vp]),
    "hb_rope_table": (C.c_int, [vp, i32, i32, C.c_double, vp]),
    "hb_rmsnorm": (C.c_int, [vp, vp, vp, i32, i32, C.c_float, vp]),
    "hb_kv_append": (C.c_int, [vp, i32, vp, vp, vp, i32, C.POINTER(hb_layer_dims), vp, vp, vp, i32, vp]),
    "hb_attention_workspace_bytes": (C.c_size_t, [C.POINTER(hb_layer_dims), i32, i32, i32]),
    "hb_attention": (C.c_int, [vp, vp, vp, i32, C.POINTER(hb_device_plan), C.POINTER(hb_layer_dims), i32, vp, vp,
                               C.c_size_t, vp]),
    "hb_attention_noalloc": (C.c_int, [vp, vp, vp, i32, C.POINTER(hb_device_plan), C.POINTER(hb_layer_dims), i32,
                                       vp, vp]),
    "hb_gemm": (C.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, vp]),
    "hb_gemm_e4m3": (C.c_int, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]),
    "hb_quantize_e4m3": (C.c_int, [vp, vp, vp, i32, i32, vp]),
    "hb_interleave_gate_up": (C.c_int, [vp, vp, vp, i32, i32, vp]),
    "hb_fold_gamma": (C.c_int, [vp, vp, vp, i32, i32, vp]),
    "hb_layer_workspace_bytes": (C.c_size_t, [C.POINTER(hb_layer_dims), i32, i32, i32]),
    "hb_layer_kernel_count": (C.c_int, [C.POINTER(hb_layer_dims), i32, i32, p_i32]),
    "hb_layers_forward": (C.c_int, [C.POINTER(hb_layer_weights), i32, C.POINTER(hb_layer_dims),
                                    C.POINTER(hb_device_plan), vp, i32, vp, vp, C.POINTER(vp), C.POINTER(vp), i32,
                                    i32, vp, C.c_size_t, vp]),
    "hb_layer_forward": (C.c_int, [C.POINTER(hb_layer_weights), C.POINTER(hb_layer_dims),
                                   C.POINTER(hb_device_plan), vp, i32, vp, vp, vp, vp, i32, i32, vp, C.c_size_t, vp,
                                   C.POINTER(hb_profile)]),
    "hb_final_logits": (C.c_int, [vp, i32, vp, i32, vp, vp, i32, i32, C.c_float, vp, vp, C.c_size_t, vp]),
    "hb_check_status": (C.c_int, [vp]),
    "hb_device_info": (C.c_int, [p_i32, p_i32]),
    "hb_kernel_launches": (C.c_uint64, []),
    "hb_selftest_wait_timeout": (C.c_int, [i32, vp]),
}

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load():
    """Build (if needed) and load libhb.so; raises if it cannot be built or loaded."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libhb.so missing at {path}")
            lib = C.CDLL(path)
            for name, (res, args) in PROTOTYPES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
