"""GB300-native hybrid-iteration forward for chunked prefill (sm_103a).

One hybrid iteration packs every active decode with prompt chunks under a
token budget tau and runs a decoder-layer forward over the packed rows with a
16-token paged KV cache.  The compute path is the C-ABI library libhb.so
(include/hb.h, CUDA kernels in csrc/); this package holds its build script
and a thin ctypes binding whose functions carry the C names.
"""
from .binding import (DevicePlan, HBError, HostPlan, LayerWeights, Scheduler, dims_struct, hb_attention,
                      hb_attention_workspace_bytes, hb_check_status, hb_device_info, hb_final_logits, hb_fold_gamma,
                      hb_gemm, hb_gemm_e4m3, hb_interleave_gate_up, hb_kernel_launches, hb_kv_append,
                      hb_layer_forward, hb_layer_kernel_count, hb_layer_workspace_bytes, hb_layers_forward,
                      hb_plan_batch, hb_quantize_e4m3, hb_rmsnorm, hb_rope_table, hb_selftest_wait_timeout,
                      hb_version, lib, prepare_layer_weights)

__all__ = [
    "DevicePlan", "HBError", "HostPlan", "LayerWeights", "Scheduler", "dims_struct", "hb_attention",
    "hb_attention_workspace_bytes", "hb_check_status", "hb_device_info", "hb_final_logits", "hb_fold_gamma",
    "hb_gemm", "hb_gemm_e4m3", "hb_interleave_gate_up", "hb_kernel_launches", "hb_kv_append", "hb_layer_forward",
    "hb_layer_kernel_count", "hb_layer_workspace_bytes", "hb_layers_forward", "hb_plan_batch", "hb_quantize_e4m3",
    "hb_rmsnorm", "hb_rope_table", "hb_selftest_wait_timeout", "hb_version", "lib", "prepare_layer_weights",
]
