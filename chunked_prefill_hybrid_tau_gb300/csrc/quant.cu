// Per-row E4M3 quantization of bf16 rows: the operand preparation of the
// FP8 projections (weights once, activations every layer).
//
// Format: OCP E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
// largest finite magnitude 448, no infinities).  Per row r:
//   amax = max_c |x[r][c]|,  inv = 448 / amax,  scale[r] = amax / 448
// (both divisions correctly rounded in fp32), and
//   q[r][c] = E4M3(fp32(x[r][c] * inv)), rounded to nearest even, saturating,
// so x[r][c] ~ scale[r] * q[r][c].  An all-zero row gets inv = 0 and
// scale = 0.  The scaling is per row because a row's result must not depend
// on the other rows of its batch (a token's codes are the same whether its
// prompt runs in one chunk or several).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "device.cuh"
#include "runtime.h"

namespace hb {
namespace {

using namespace dev;

constexpr int kQuantThreads = 128;

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi, float inv) {
  const __nv_fp8x2_storage_t v =
      __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(lo, inv), __fmul_rn(hi, inv)), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(v);
}

// One CTA per row; thread t holds 16-byte pieces t, t + 128, ... of the row
// in registers.  SS: also the 32-column partial sums of squares of the bf16
// row (the GemmNorm layout: four adjacent pieces, reduced over four adjacent
// lanes by a fixed xor pattern, the same arithmetic as row_sumsq_kernel).
template <int NV, bool SS>
__global__ void __launch_bounds__(kQuantThreads)
    quant_rows_kernel(const uint4* __restrict__ x, uint2* __restrict__ q, float* __restrict__ scale, int c8,
                      float* __restrict__ ss, int* zero, int n_zero) {
  griddep_launch_dependents();
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0;
  __shared__ float red[kQuantThreads / 32];
  const int r = blockIdx.x;
  const int t = threadIdx.x, lane = t & 31;
  const uint4* xr = x + static_cast<size_t>(r) * c8;
  uint4 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = t + kQuantThreads * k;
    v[k] = i < c8 ? xr[i] : make_uint4(0, 0, 0, 0);
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      if (SS) {
        a = __fmaf_rn(f.x, f.x, a);
        a = __fmaf_rn(f.y, f.y, a);
      }
    }
    if (SS) {
      a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 1));
      a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 2));
      const int i = t + kQuantThreads * k;
      if ((lane & 3) == 0 && i < c8) ss[static_cast<size_t>(r) * (c8 / 4) + i / 4] = a;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[t >> 5] = amax;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const bool nz = amax > 0.f;
  const float inv = nz ? __fdiv_rn(448.0f, amax) : 0.f;
  if (t == 0) scale[r] = nz ? __fdiv_rn(amax, 448.0f) : 0.f;
  uint2* qr = q + static_cast<size_t>(r) * c8;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = t + kQuantThreads * k;
    if (i >= c8) break;
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    uint32_t b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      b[j] = e4m3x2(f.x, f.y, inv);
    }
    qr[i] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
  }
}

}  // namespace

hb_status quant_rows_launch(const DeviceCtx& ctx, const void* x, void* q, float* scale, int rows, int cols,
                            float* ss, int* zero, int n_zero, cudaStream_t stream) {
  (void)ctx;
  if (rows == 0) return HB_OK;
  const int c8 = cols / 8;
  const int nv = (c8 + kQuantThreads - 1) / kQuantThreads;
  auto* xp = static_cast<const uint4*>(x);
  auto* qp = static_cast<uint2*>(q);
#define HB_Q(NV_)                                                                                               \
  if (nv <= NV_) {                                                                                              \
    if (ss)                                                                                                     \
      return launch_pdl(quant_rows_kernel<NV_, true>, rows, kQuantThreads, 0, stream, "quant_rows_kernel launch", \
                        xp, qp, scale, c8, ss, zero, n_zero);                                                   \
    return launch_pdl(quant_rows_kernel<NV_, false>, rows, kQuantThreads, 0, stream, "quant_rows_kernel launch",  \
                      xp, qp, scale, c8, ss, zero, n_zero);                                                     \
  }
  HB_Q(1)
  HB_Q(2)
  HB_Q(4)
  HB_Q(8)
  HB_Q(16)
  HB_Q(32)
#undef HB_Q
  set_error("E4M3 quantization: %d columns above the supported 32768", cols);
  return HB_ERR_UNSUPPORTED;
}

}  // namespace hb

extern "C" hb_status hb_quantize_e4m3(const void* x, void* q, float* scale, int32_t rows, int32_t cols,
                                      void* stream) {
  hb::clear_error();
  HB_REQUIRE(x && q && scale, "hb_quantize_e4m3: null pointer");
  HB_REQUIRE(rows >= 0 && cols > 0 && cols % 16 == 0, "hb_quantize_e4m3: rows >= 0 and cols %% 16 == 0 required");
  HB_REQUIRE(hb::aligned16(x) && hb::aligned16(q), "hb_quantize_e4m3: 16-byte alignment");
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  return hb::quant_rows_launch(ctx, x, q, scale, rows, cols, nullptr, nullptr, 0, static_cast<cudaStream_t>(stream));
}
