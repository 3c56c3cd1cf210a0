// hb_attention_noalloc: the hybrid attention for callers that cannot hand the
// library a device workspace.
//
// Some callers cannot allocate device memory at all: a plug-in that runs
// inside another engine's execution step, where that engine owns every
// device allocation and forbids cudaMalloc (which can also synchronise the
// whole device), or a host runtime that has no spare buffer to pass down.
// This entry point needs nothing from them but the inputs and the output:
// its scratch (split-KV partial results and counters) lives in a fixed
// file-scope device array of kNoAllocScratchBytes that every GPU loading the
// library holds until the process exits.
#include <mutex>

#include "runtime.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// Host code must not use this name as a device address: on the host it is a
// stand-in, so its device address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_attention_scratch[kNoAllocScratchBytes];

void* g_scratch_ptr[hb::kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on `device` (the current device),
// looked up once per device.
hb_status scratch_address(int device, void** out) {
  if (device < 0 || device >= hb::kMaxDevices) {
    hb::set_error("hb_attention_noalloc: device ordinal %d out of range", device);
    return HB_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[device] == nullptr) {
    void* p = nullptr;
    hb_status st = hb::cuda_status(cudaGetSymbolAddress(&p, g_attention_scratch),
                                   "cudaGetSymbolAddress(attention scratch)");
    if (st != HB_OK) return st;
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return HB_OK;
}

}  // namespace

extern "C" hb_status hb_attention_noalloc(const void* q, const void* k_cache, const void* v_cache, int32_t num_pages,
                                          const hb_device_plan* plan, const hb_layer_dims* dims, int32_t max_kv_len,
                                          void* out, void* stream) {
  hb::clear_error();
  hb_status st = hb::check_dims(dims);
  if (st != HB_OK) return st;
  HB_REQUIRE(plan != nullptr, "hb_attention_noalloc: null plan");
  HB_REQUIRE(q && k_cache && v_cache && out, "hb_attention_noalloc: null pointer");
  HB_REQUIRE(plan->n_seqs == 0 || (plan->seq_q_start && plan->seq_kv_len && plan->block_table),
             "hb_attention_noalloc: null plan array");
  HB_REQUIRE(num_pages > 0 && max_kv_len >= 1 && plan->n_seqs >= 0, "hb_attention_noalloc: bad sizes");
  const size_t need = hb::attention_workspace_bytes(*dims, plan->n_seqs, max_kv_len);
  if (need > kNoAllocScratchBytes) {
    hb::set_error("hb_attention_noalloc: %d sequences with up to %d keys need %zu bytes of scratch; the fixed "
                  "scratch holds %zu bytes (use hb_attention with a workspace)",
                  plan->n_seqs, max_kv_len, need, kNoAllocScratchBytes);
    return HB_ERR_CAPACITY;
  }
  hb::DeviceCtx ctx;
  st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  void* scratch = nullptr;
  st = scratch_address(ctx.device, &scratch);
  if (st != HB_OK) return st;
  return hb::attention_launch(ctx, q, k_cache, v_cache, num_pages, *plan, *dims, max_kv_len, out, scratch,
                              kNoAllocScratchBytes, static_cast<cudaStream_t>(stream), false);
}
