// Host runtime pieces: device status word, device properties, TMA tensor-map
// encoding through the driver entry point (no link-time libcuda dependency,
// so the library also loads on machines without a GPU driver).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "runtime.h"

// Device status word: 0 = ok, else the first error a kernel recorded.
__device__ int g_hb_status_word;

namespace hb {

namespace {
// Per-device state, filled once under g_mu.  The status pointer is published
// last with release order: a thread that reads it non-null (acquire) also
// sees that device's SM count and compute capability.
std::atomic<int*> g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
int g_cc[kMaxDevices];
std::mutex g_mu;
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};
}  // namespace

hb_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return HB_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return HB_ERR_CUDA;
}

static hb_status init_device(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_status_ptr[dev].load(std::memory_order_relaxed) != nullptr) return HB_OK;
  void* p = nullptr;
  hb_status st = cuda_status(cudaGetSymbolAddress(&p, g_hb_status_word), "cudaGetSymbolAddress(status word)");
  if (st != HB_OK) return st;
  cudaDeviceProp prop;
  st = cuda_status(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
  if (st != HB_OK) return st;
  g_num_sms[dev] = prop.multiProcessorCount;
  g_cc[dev] = prop.major * 10 + prop.minor;
  g_status_ptr[dev].store(static_cast<int*>(p), std::memory_order_release);
  return HB_OK;
}

hb_status device_context(DeviceCtx* ctx) {
  int dev = 0;
  hb_status st = cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != HB_OK) return st;
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d out of range", dev);
    return HB_ERR_UNSUPPORTED;
  }
  int* status = g_status_ptr[dev].load(std::memory_order_acquire);
  if (status == nullptr) {
    st = init_device(dev);
    if (st != HB_OK) return st;
    status = g_status_ptr[dev].load(std::memory_order_acquire);
  }
  if (g_cc[dev] != 103) {
    set_error("the library is built for sm_103a; device %d is sm_%d", dev, g_cc[dev]);
    return HB_ERR_UNSUPPORTED;
  }
  ctx->device = dev;
  ctx->num_sms = g_num_sms[dev];
  ctx->status = status;
  return HB_OK;
}

static hb_status resolve_encode() {
  if (g_encode.load(std::memory_order_acquire) != nullptr) return HB_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode.load(std::memory_order_relaxed) != nullptr) return HB_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  hb_status st =
      cuda_status(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q),
                  "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
  if (st != HB_OK) return st;
  if (q != cudaDriverEntryPointSuccess || fn == nullptr) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return HB_ERR_UNSUPPORTED;
  }
  g_encode.store(reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn), std::memory_order_release);
  return HB_OK;
}

hb_status encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128,
                         int elem_bytes) {
  hb_status st = resolve_encode();
  if (st != HB_OK) return st;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = g_encode.load(std::memory_order_acquire)(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, box %u x %u", static_cast<int>(r),
              static_cast<unsigned long long>(inner), static_cast<unsigned long long>(outer), box_inner, box_outer);
    return HB_ERR_INVALID_ARG;
  }
  return HB_OK;
}

// 3-D map over q [T][n_q][d_head] bf16: box of 64 dims x 1 head x 128 tokens,
// 128-byte swizzle (one K-major half tile of a 128-row attention unit).
hb_status encode_tmap_q3d(CUtensorMap* map, const void* q, int T, int n_q, int d_head) {
  hb_status st = resolve_encode();
  if (st != HB_OK) return st;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d_head), static_cast<cuuint64_t>(n_q), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d_head) * 2, static_cast<cuuint64_t>(n_q) * d_head * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = g_encode.load(std::memory_order_acquire)(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (q, 3-D) failed (%d)", static_cast<int>(res));
    return HB_ERR_INVALID_ARG;
  }
  return HB_OK;
}

hb_status encode_tmap_kv_pages(CUtensorMap* map, const void* pool, uint64_t rows, int d_head) {
  hb_status st = resolve_encode();
  if (st != HB_OK) return st;
  const cuuint32_t halves = static_cast<cuuint32_t>(d_head / 64);
  cuuint64_t dims[3] = {64, rows, halves};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d_head) * 2, 128};
  cuuint32_t box[3] = {64, 16, halves};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = g_encode.load(std::memory_order_acquire)(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (kv pages, 3-D) failed (%d)", static_cast<int>(res));
    return HB_ERR_INVALID_ARG;
  }
  return HB_OK;
}

// Kernels launched by this library in this process (all devices and host
// threads).
static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

hb_status launch_status(const char* what) {
  const hb_status st = cuda_status(cudaGetLastError(), what);
  if (st == HB_OK) count_launch();
  return st;
}

}  // namespace hb

extern "C" uint64_t hb_kernel_launches(void) { return hb::g_launches.load(std::memory_order_relaxed); }

extern "C" hb_status hb_check_status(void* stream) {
  hb::clear_error();
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  st = hb::cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  if (st != HB_OK) return st;
  int word = 0;
  st = hb::cuda_status(cudaMemcpy(&word, ctx.status, sizeof(int), cudaMemcpyDeviceToHost), "read status word");
  if (st != HB_OK) return st;
  if (word == 0) return HB_OK;
  const int zero = 0;
  st = hb::cuda_status(cudaMemcpy(ctx.status, &zero, sizeof(int), cudaMemcpyHostToDevice), "clear status word");
  if (st != HB_OK) return st;
  if (word == hb::kDevTimeout) {
    hb::set_error("a bounded device-side wait expired");
    return HB_ERR_TIMEOUT;
  }
  hb::set_error("a device-side index check failed (code %d)", word);
  return HB_ERR_DEVICE;
}

extern "C" hb_status hb_device_info(int32_t* num_sms, int32_t* is_sm103) {
  hb::clear_error();
  HB_REQUIRE(num_sms && is_sm103, "hb_device_info: null output");
  int dev = 0;
  hb_status st = hb::cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != HB_OK) return st;
  cudaDeviceProp prop;
  st = hb::cuda_status(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
  if (st != HB_OK) return st;
  *num_sms = prop.multiProcessorCount;
  *is_sm103 = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
  return HB_OK;
}
