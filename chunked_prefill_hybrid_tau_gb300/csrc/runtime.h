// Host-side runtime helpers shared by the CUDA translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.h"

namespace hb {

// Device ordinals the per-device state covers (device_context rejects others).
constexpr int kMaxDevices = 64;

struct DeviceCtx {
  int device;
  int num_sms;
  int* status;  // device address of the status word of this device
};

// Current device, checked to be sm_103; status-word address cached per device.
hb_status device_context(DeviceCtx* ctx);

hb_status cuda_status(cudaError_t e, const char* what);
// After a <<<...>>> launch: its error, and the launch counted when accepted.
hb_status launch_status(const char* what);
// Counts one accepted kernel launch (hb_kernel_launches reads the total).
void count_launch();

// 2D tensor map of bf16 (elem_bytes 2), byte (elem_bytes 1: E4M3 codes) or
// fp32 (elem_bytes 4) elements: `outer` rows of `inner` elements, rows
// `row_stride_bytes` apart; box of box_inner x box_outer elements.
hb_status encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128,
                         int elem_bytes = 2);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Raises a kernel's dynamic shared-memory limit once per device.  `done` is
// that kernel's per-device flag array (kMaxDevices entries, static storage).
// Host threads that make their first call at the same time may each set the
// attribute; setting it is idempotent, and the flags are atomics, so this is
// free of data races.
template <typename Kernel>
hb_status smem_limit_once(std::atomic<bool>* done, int device, Kernel kernel, int bytes, const char* what) {
  if (done[device].load(std::memory_order_acquire)) return HB_OK;
  hb_status st = cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), what);
  if (st == HB_OK) done[device].store(true, std::memory_order_release);
  return st;
}

// Launch with programmatic stream serialization: the kernel may start while
// its predecessor on the stream is still running (once every predecessor CTA
// has signalled griddepcontrol.launch_dependents) and must execute
// griddepcontrol.wait before it touches memory the predecessor writes or
// reads.  Every kernel of this library does both, so kernels complete in
// stream order.  Behind anything that is not such a kernel (a copy, an event,
// another library's kernel) the launch waits as usual.
template <typename... KArgs, typename... Args>
hb_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     const char* what, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const hb_status st = cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...), what);
  if (st == HB_OK) count_launch();
  return st;
}

hb_status encode_tmap_q3d(CUtensorMap* map, const void* q, int T, int n_q, int d_head);
// 3-D map over a paged K or V pool [page][n_kv][16][d_head] bf16 seen as
// (64 dims, rows = (page * n_kv + head) * 16 + key, d_head / 64 halves): one
// box of 64 x 16 x (d_head / 64) loads a whole 16-key page of one kv head as
// [half][key][128 bytes] with the 128-byte swizzle, the layout of two
// separate 64-dim boxes placed 2 KB apart.
hb_status encode_tmap_kv_pages(CUtensorMap* map, const void* pool, uint64_t rows, int d_head);
hb_status chunk_tc_launch(const DeviceCtx& ctx, const void* q, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const hb_device_plan& plan, const hb_layer_dims& dims, int num_pages, int max_kv_len,
                          void* out, int* work_counter, int grid, cudaStream_t stream);

// Shape checks shared by the layer entry points.
hb_status check_dims(const hb_layer_dims* dims);

// Launchers (arguments already checked; asynchronous on `stream`).
hb_status rmsnorm_launch(const DeviceCtx& ctx, const void* x, const int* rows, const void* gamma, void* y,
                         int n_rows, int d, float eps, int n_src, cudaStream_t stream);
// zero / n_zero: ints cleared after the kernel's wait for its inputs (the
// layer's split-K and attention counters; nullptr, 0 for none).
hb_status kv_append_launch(const DeviceCtx& ctx, const void* qkv, int T, const int* row_pos, const int* slots,
                           const void* rope, int max_pos, const hb_layer_dims& dims, void* q_out, void* k_cache,
                           void* v_cache, int num_pages, cudaStream_t stream, int* zero = nullptr, int n_zero = 0);
hb_status gemm_check(const void* A, const void* B, void* C, const void* R, int M, int N, int K, int epi);

// RMSNorm folded into the projections.  Row statistics are 32-column partial
// sums of squares, float [rows][parts] with parts = d / 32, always grouped
// the same way whatever the tile shape, so a row's factor never depends on
// its batch.  ss_in: scale each output row by rsqrt(sum / d + eps) (STORE,
// SWIGLU; the gamma is folded into the weights).  ss_out: write the
// statistics of the rounded output rows (RESIDUAL).
struct GemmNorm {
  const float* ss_in = nullptr;
  float* ss_out = nullptr;
  int parts = 0;
  float inv_d = 0.f, eps = 0.f;
};

// Split-K workspace for RESIDUAL projections (fp32 partial tiles and arrival
// counters; the counters must be zero at launch and are not cleared by the
// kernel: a kernel ahead of the projections zeroes them).  Used when
// gemm_split_k(N, K, epi) holds, which depends on the shape only.
struct GemmSplit {
  float* part = nullptr;
  int* flags = nullptr;
};
bool gemm_split_k(int N, int K, int epi);

// QKV projection with the RoPE rotation and the paged KV append in its
// epilogue (the layer's fused path with E4M3 weights, epilogue id kEpiRope,
// internal, gemm_e4m3_launch only): the
// rotated q rows go to q_out [rows][n_q][d_head], the rotated K row and the
// V row of each token to its slot of the [page][n_kv][16][d_head] pools.
// rope, row_pos and slots as for kv_append_launch; the arithmetic and the
// rounding points are those of the projection's STORE epilogue followed by
// kv_append_kernel, so the fused and the two-kernel paths give the same bits.
struct GemmRope {
  const float2* rope = nullptr;
  const int* row_pos = nullptr;
  const int* slots = nullptr;
  void* q_out = nullptr;
  void* k_cache = nullptr;
  void* v_cache = nullptr;
  int n_q = 0, n_kv = 0, d_head = 0, max_pos = 0;
  long long num_slots = 0;
};
constexpr int kEpiRope = 16;
// The fused path applies when whole heads fall in every 128- and 256-column tile.
bool gemm_rope_ok(int N, const hb_layer_dims& dims);
// Tile width of CTA-pair tiles (tcgen05 cta_group::2, 256 rows) for a
// projection, or 0 for one-CTA tiles.
int gemm_pair_bn(int M, int N, int epi, bool split, int num_sms);
size_t gemm_split_part_bytes(int M, int N);  // fp32 partial tiles
int gemm_split_flags(int M, int N);          // arrival counters (ints)

// E4M3 projections: A [M][K] and B [N][K] codes (row stride lda bytes for A,
// K for B) with per-row fp32 scales sa [M] and sb [N]; the epilogues are the
// bf16 ones applied to sa[m] sb[n] acc.
hb_status gemm_e4m3_launch(const DeviceCtx& ctx, const void* A, int lda, const float* sa, const void* B,
                           const float* sb, void* C, int ldc, const void* R, int M, int N, int K, int epi,
                           cudaStream_t stream, const GemmNorm* norm = nullptr, const GemmSplit* split = nullptr,
                           const GemmRope* rope = nullptr);
hb_status gemm_e4m3_check(const void* A, const float* sa, const void* B, const float* sb, void* C, const void* R,
                          int M, int N, int K, int epi);

// Per-row E4M3 quantization of bf16 rows x [rows][cols] (row stride cols):
// codes q [rows][cols], scales [rows]; with ss != nullptr also the row
// statistics of x in the GemmNorm layout (cols % 32 == 0), and n_zero ints
// at `zero` cleared (as row_sumsq_launch).
hb_status quant_rows_launch(const DeviceCtx& ctx, const void* x, void* q, float* scale, int rows, int cols,
                            float* ss, int* zero, int n_zero, cudaStream_t stream);

// A [M][K] with row stride lda, B [N][K], C/R with row stride ldc (elements).
hb_status gemm_launch(const DeviceCtx& ctx, const void* A, int lda, const void* B, void* C, int ldc, const void* R,
                      int M, int N, int K, int epi, cudaStream_t stream, const GemmNorm* norm = nullptr,
                      const GemmSplit* split = nullptr);

// Row statistics of x [rows][d] bf16 in the GemmNorm layout; also zeroes
// n_zero ints at `zero` (split-K counters of the launches that follow).
hb_status row_sumsq_launch(const DeviceCtx& ctx, const void* x, float* ss, int rows, int d, int* zero, int n_zero,
                           cudaStream_t stream);
size_t attention_workspace_bytes(const hb_layer_dims& dims, int max_seqs, int max_kv_len);
// Bytes at the start of the attention workspace that must be zero when the
// attention kernels start (work and combine counters).
size_t attention_counter_bytes(const hb_layer_dims& dims, int n_seqs);
// counters_zeroed: the caller has zeroed the counters on the stream (the
// layer does it in a kernel ahead of the attention), else they are cleared
// here.
hb_status attention_launch(const DeviceCtx& ctx, const void* q, const void* k_cache, const void* v_cache,
                           int num_pages, const hb_device_plan& plan, const hb_layer_dims& dims, int max_kv_len,
                           void* out, void* ws, size_t ws_bytes, cudaStream_t stream, bool counters_zeroed);

}  // namespace hb
