// Memory-bound kernels of the layer: RMSNorm, the RoPE table, and the fused
// RoPE + paged KV append.
#include <cuda_bf16.h>

#include "device.cuh"
#include "runtime.h"

namespace hb {
namespace {

using namespace dev;

// ---------------------------------------------------------------- RMSNorm
// One warp per row, four rows per CTA.  The row is held in registers (NV
// 16-byte vectors per lane, all loads issued before the reduction), fp32
// sum of squares, shuffle reduction, y = x * rsqrt(mean(x^2) + eps) * gamma
// rounded once to bf16.  `rows` (optional) gathers source rows (final norm
// of selected rows).
constexpr int kNormWarps = 4;

template <int NV>
__global__ void __launch_bounds__(kNormWarps * 32)
    rmsnorm_kernel(const uint4* __restrict__ x, const int* __restrict__ rows, const uint4* __restrict__ gamma,
                   uint4* __restrict__ y, int n_rows, int d8, float inv_d, float eps, int n_src, int* status) {
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kNormWarps + warp;
  if (r >= n_rows) return;
  int src = r;
  if (rows) {
    src = rows[r];
    if (src < 0 || src >= n_src) {
      if (lane == 0) flag_error(status, kStatusIndex);
      return;
    }
  }
  const uint4* xr = x + static_cast<size_t>(src) * d8;
  uint4 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = lane + 32 * k;
    v[k] = i < d8 ? xr[i] : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      ss += f.x * f.x + f.y * f.y;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss * inv_d + eps);
  uint4* yr = y + static_cast<size_t>(r) * d8;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = lane + 32 * k;
    if (i >= d8) break;
    const uint4 g = gamma[i];
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]), gg = unpack_bf16x2(gw[j]);
      o[j] = pack_bf16x2(f.x * inv * gg.x, f.y * inv * gg.y);
    }
    yr[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------- row statistics
// 32-column partial sums of squares of bf16 rows (the layout of GemmNorm):
// one warp per row, lane i holds 16-byte pieces i, i+32, ...; four adjacent
// pieces make one 32-column group, reduced over the four lanes by a fixed
// xor pattern.
template <int NV>
__global__ void __launch_bounds__(kNormWarps * 32)
    row_sumsq_kernel(const uint4* __restrict__ x, float* __restrict__ ss, int n_rows, int d8, int* zero,
                     int n_zero) {
  griddep_launch_dependents();
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kNormWarps + warp;
  if (r >= n_rows) return;
  const uint4* xr = x + static_cast<size_t>(r) * d8;
  uint4 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int i = lane + 32 * k;
    v[k] = i < d8 ? xr[i] : make_uint4(0, 0, 0, 0);
  }
  float* out = ss + static_cast<size_t>(r) * (d8 / 4);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      a = __fmaf_rn(f.x, f.x, a);
      a = __fmaf_rn(f.y, f.y, a);
    }
    // parts of 32 columns: (lane 4q + lane 4q+1) + (lane 4q+2 + lane 4q+3)
    a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const int i = lane + 32 * k;
    if ((lane & 3) == 0 && i < d8) out[i / 4] = a;
  }
}

// ---------------------------------------------------------------- gamma folding
// out[r][c] = bf16(w[r][c] * gamma[c]): RMSNorm's gain moved into the
// projection that consumes the normalised rows (x * inv * g) W^T =
// inv * x (W diag(g))^T.  out may alias w.
__global__ void fold_gamma_kernel(const uint4* w, const uint4* __restrict__ gamma, uint4* out, size_t total, int d8) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 a = w[i], g = gamma[i % d8];
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 fa = unpack_bf16x2(aw[j]), fg = unpack_bf16x2(gw[j]);
      o[j] = pack_bf16x2(fa.x * fg.x, fa.y * fg.y);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------- RoPE table
// table[p][i] = (cos, sin)(p * theta^(-2i/d_head)) in double, rounded to float.
__global__ void rope_table_kernel(float2* __restrict__ t, int max_pos, int half, int d_head, double theta) {
  const size_t total = static_cast<size_t>(max_pos) * half;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
    const double inv_freq = pow(theta, -2.0 * i / d_head);
    double s, c;
    sincos(static_cast<double>(p) * inv_freq, &s, &c);
    t[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

// ---------------------------------------------------------------- RoPE + KV append
// One CTA per row.  A "rotating" thread owns 8 elements of the first half of
// a q or k head and the matching 8 of the second half (rotate-half pairs i
// and i + d/2); a "copy" thread moves 8 elements of a v head.  All global
// accesses are 16 bytes.  K/V land at slot = page*16 + offset of the
// [page][kv head][16][d_head] pools.
template <int DH>
__global__ void kv_append_kernel(const __nv_bfloat16* __restrict__ qkv, const int* __restrict__ row_pos,
                                 const int* __restrict__ slots, const float2* __restrict__ rope, int max_pos, int n_q,
                                 int n_kv, __nv_bfloat16* __restrict__ q_out, __nv_bfloat16* __restrict__ kc,
                                 __nv_bfloat16* __restrict__ vc, long long num_slots, int* status, int* zero,
                                 int n_zero) {
  constexpr int HALF = DH / 2;
  constexpr int RC = HALF / 8;  // rotating threads per head
  constexpr int VC = DH / 8;    // copy threads per v head
  griddep_launch_dependents();
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0;
  const int r = blockIdx.x;
  const int pos = row_pos[r];
  const int slot = slots[r];
  const int ld = (n_q + 2 * n_kv) * DH;
  const bool pos_ok = pos >= 0 && pos < max_pos;
  const bool slot_ok = slot >= 0 && slot < num_slots;
  if (threadIdx.x == 0) {
    if (!pos_ok || slot >= num_slots) flag_error(status, kStatusIndex);
  }
  if (!pos_ok) return;
  const int page = slot / 16, off = slot % 16;
  const __nv_bfloat16* src_row = qkv + static_cast<size_t>(r) * ld;
  const int rot = (n_q + n_kv) * RC;
  const int total = rot + n_kv * VC;
  for (int t = threadIdx.x; t < total; t += blockDim.x) {
    if (t < rot) {
      const int h = t / RC, c = t % RC;
      const __nv_bfloat16* src = src_row + h * DH + c * 8;
      uint4 a = *reinterpret_cast<const uint4*>(src);
      uint4 b = *reinterpret_cast<const uint4*>(src + HALF);
      const float4* cs = reinterpret_cast<const float4*>(rope + static_cast<size_t>(pos) * HALF + c * 8);
      uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w}, o1[4], o2[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 t2 = cs[j];  // (cos, sin) of element 2j and 2j+1
        const float2 x1 = unpack_bf16x2(aw[j]), x2 = unpack_bf16x2(bw[j]);
        // each product and sum rounded to fp32 (no contraction), as in the
        // fused QKV epilogue, so both paths give the same bits
        o1[j] = pack_bf16x2(__fsub_rn(__fmul_rn(x1.x, t2.x), __fmul_rn(x2.x, t2.y)),
                            __fsub_rn(__fmul_rn(x1.y, t2.z), __fmul_rn(x2.y, t2.w)));
        o2[j] = pack_bf16x2(__fadd_rn(__fmul_rn(x2.x, t2.x), __fmul_rn(x1.x, t2.y)),
                            __fadd_rn(__fmul_rn(x2.y, t2.z), __fmul_rn(x1.y, t2.w)));
      }
      __nv_bfloat16* dst;
      if (h < n_q) {
        dst = q_out + (static_cast<size_t>(r) * n_q + h) * DH;
      } else {
        if (!slot_ok) continue;
        dst = kc + ((static_cast<size_t>(page) * n_kv + (h - n_q)) * 16 + off) * DH;
      }
      *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
      *reinterpret_cast<uint4*>(dst + HALF + c * 8) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
    } else {
      if (!slot_ok) continue;
      const int t2 = t - rot;
      const int g = t2 / VC, c = t2 % VC;
      const uint4 v = *reinterpret_cast<const uint4*>(src_row + (n_q + n_kv + g) * DH + c * 8);
      *reinterpret_cast<uint4*>(vc + ((static_cast<size_t>(page) * n_kv + g) * 16 + off) * DH + c * 8) = v;
    }
  }
}

}  // namespace

hb_status rmsnorm_launch(const DeviceCtx& ctx, const void* x, const int* rows, const void* gamma, void* y,
                         int n_rows, int d, float eps, int n_src, cudaStream_t stream) {
  if (n_rows == 0) return HB_OK;
  const int blocks = (n_rows + kNormWarps - 1) / kNormWarps;
  const int d8 = d / 8;
  const int nv = (d8 + 31) / 32;
  auto* xp = static_cast<const uint4*>(x);
  auto* gp = static_cast<const uint4*>(gamma);
  auto* yp = static_cast<uint4*>(y);
#define HB_NORM(NV_)                                                                                           \
  if (nv <= NV_) {                                                                                             \
    return launch_pdl(rmsnorm_kernel<NV_>, blocks, kNormWarps * 32, 0, stream, "rmsnorm_kernel launch", xp, rows, \
                      gp, yp, n_rows, d8, 1.0f / d, eps, n_src, ctx.status);                                     \
  }
  HB_NORM(1)
  HB_NORM(2)
  HB_NORM(4)
  HB_NORM(8)
  HB_NORM(16)
  HB_NORM(32)
#undef HB_NORM
  set_error("rmsnorm: d = %d above the supported 8192", d);
  return HB_ERR_UNSUPPORTED;
}

hb_status row_sumsq_launch(const DeviceCtx& ctx, const void* x, float* ss, int rows, int d, int* zero, int n_zero,
                           cudaStream_t stream) {
  if (rows == 0) return HB_OK;
  const int blocks = (rows + kNormWarps - 1) / kNormWarps;
  const int d8 = d / 8;
  const int nv = (d8 + 31) / 32;
  auto* xp = static_cast<const uint4*>(x);
  (void)ctx;
#define HB_SS(NV_)                                                                                                 \
  if (nv <= NV_)                                                                                                   \
    return launch_pdl(row_sumsq_kernel<NV_>, blocks, kNormWarps * 32, 0, stream, "row_sumsq_kernel launch", xp, ss, \
                      rows, d8, zero, n_zero);
  HB_SS(1)
  HB_SS(2)
  HB_SS(4)
  HB_SS(8)
  HB_SS(16)
  HB_SS(32)
#undef HB_SS
  set_error("row statistics: d = %d above the supported 8192", d);
  return HB_ERR_UNSUPPORTED;
}

hb_status kv_append_launch(const DeviceCtx& ctx, const void* qkv, int T, const int* row_pos, const int* slots,
                           const void* rope, int max_pos, const hb_layer_dims& dm, void* q_out, void* k_cache,
                           void* v_cache, int num_pages, cudaStream_t stream, int* zero, int n_zero) {
  if (T == 0) return HB_OK;
  const int per_row = (dm.n_q + dm.n_kv) * (dm.d_head / 16) + dm.n_kv * (dm.d_head / 8);
  const int threads = per_row < 1024 ? ((per_row + 31) / 32) * 32 : 1024;
  const long long num_slots = static_cast<long long>(num_pages) * 16;
  auto* qo = static_cast<__nv_bfloat16*>(q_out);
  auto* kc = static_cast<__nv_bfloat16*>(k_cache);
  auto* vc = static_cast<__nv_bfloat16*>(v_cache);
  auto* in = static_cast<const __nv_bfloat16*>(qkv);
  auto* rp = static_cast<const float2*>(rope);
  if (dm.d_head == 128)
    return launch_pdl(kv_append_kernel<128>, T, threads, 0, stream, "kv_append_kernel launch", in, row_pos, slots, rp,
                      max_pos, dm.n_q, dm.n_kv, qo, kc, vc, num_slots, ctx.status, zero, n_zero);
  return launch_pdl(kv_append_kernel<64>, T, threads, 0, stream, "kv_append_kernel launch", in, row_pos, slots, rp,
                    max_pos, dm.n_q, dm.n_kv, qo, kc, vc, num_slots, ctx.status, zero, n_zero);
}

hb_status check_dims(const hb_layer_dims* dm) {
  HB_REQUIRE(dm != nullptr, "null hb_layer_dims");
  HB_REQUIRE(dm->d_model > 0 && dm->d_model % 64 == 0, "d_model must be a positive multiple of 64");
  HB_REQUIRE(dm->n_q > 0 && dm->n_kv > 0 && dm->n_q % dm->n_kv == 0, "n_q must be a multiple of n_kv");
  HB_REQUIRE(dm->n_q / dm->n_kv <= 16, "at most 16 query heads per kv head");
  HB_REQUIRE(dm->d_head == 64 || dm->d_head == 128, "d_head must be 64 or 128");
  HB_REQUIRE(dm->d_ff > 0 && dm->d_ff % 8 == 0, "d_ff must be a positive multiple of 8");
  HB_REQUIRE(dm->page_size == 16, "page_size must be 16");
  HB_REQUIRE(dm->rms_eps >= 0.f, "rms_eps must be >= 0");
  return HB_OK;
}

}  // namespace hb

extern "C" hb_status hb_rmsnorm(const void* x, const void* gamma, void* y, int32_t rows, int32_t d, float eps,
                                void* stream) {
  hb::clear_error();
  HB_REQUIRE(x && gamma && y, "hb_rmsnorm: null pointer");
  HB_REQUIRE(rows >= 0 && d > 0 && d % 8 == 0, "hb_rmsnorm: rows >= 0 and d %% 8 == 0 required");
  HB_REQUIRE(hb::aligned16(x) && hb::aligned16(gamma) && hb::aligned16(y), "hb_rmsnorm: 16-byte alignment");
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  return hb::rmsnorm_launch(ctx, x, nullptr, gamma, y, rows, d, eps, rows, static_cast<cudaStream_t>(stream));
}

extern "C" hb_status hb_rope_table(void* table, int32_t max_pos, int32_t d_head, double theta, void* stream) {
  hb::clear_error();
  HB_REQUIRE(table != nullptr, "hb_rope_table: null table");
  HB_REQUIRE(max_pos > 0 && d_head > 0 && d_head % 16 == 0 && theta > 1.0, "hb_rope_table: bad arguments");
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  hb::rope_table_kernel<<<ctx.num_sms * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<float2*>(table), max_pos, d_head / 2, d_head, theta);
  return hb::launch_status("rope_table_kernel launch");
}

extern "C" hb_status hb_kv_append(const void* qkv, int32_t T, const int32_t* row_pos, const int32_t* slot_mapping,
                                  const void* rope, int32_t max_pos, const hb_layer_dims* dims, void* q_out,
                                  void* k_cache, void* v_cache, int32_t num_pages, void* stream) {
  hb::clear_error();
  hb_status st = hb::check_dims(dims);
  if (st != HB_OK) return st;
  HB_REQUIRE(T >= 0 && max_pos > 0 && num_pages > 0, "hb_kv_append: bad sizes");
  HB_REQUIRE(qkv && row_pos && slot_mapping && rope && q_out && k_cache && v_cache, "hb_kv_append: null pointer");
  HB_REQUIRE(hb::aligned16(qkv) && hb::aligned16(q_out) && hb::aligned16(k_cache) && hb::aligned16(v_cache) &&
                 hb::aligned16(rope),
             "hb_kv_append: 16-byte alignment");
  hb::DeviceCtx ctx;
  st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  return hb::kv_append_launch(ctx, qkv, T, row_pos, slot_mapping, rope, max_pos, *dims, q_out, k_cache, v_cache,
                              num_pages, static_cast<cudaStream_t>(stream));
}

extern "C" hb_status hb_fold_gamma(const void* w, const void* gamma, void* out, int32_t rows, int32_t cols,
                                   void* stream) {
  hb::clear_error();
  HB_REQUIRE(w && gamma && out, "hb_fold_gamma: null pointer");
  HB_REQUIRE(rows > 0 && cols > 0 && cols % 8 == 0, "hb_fold_gamma: rows > 0 and cols %% 8 == 0 required");
  HB_REQUIRE(hb::aligned16(w) && hb::aligned16(gamma) && hb::aligned16(out), "hb_fold_gamma: 16-byte alignment");
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  const size_t total = static_cast<size_t>(rows) * (cols / 8);
  hb::fold_gamma_kernel<<<ctx.num_sms * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(w), static_cast<const uint4*>(gamma), static_cast<uint4*>(out), total, cols / 8);
  return hb::launch_status("fold_gamma_kernel launch");
}

namespace hb {
namespace {
// One thread waits on a barrier that nothing ever completes: the bounded
// wait gives up after timeout_ns and records a timeout in the status word,
// the path every kernel takes when a copy or a partner never arrives.
__global__ void wait_selftest_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, nullptr, status, timeout_ns);
}
}  // namespace
}  // namespace hb

extern "C" hb_status hb_selftest_wait_timeout(int32_t timeout_us, void* stream) {
  hb::clear_error();
  HB_REQUIRE(timeout_us >= 1 && timeout_us <= 1000000, "hb_selftest_wait_timeout: timeout_us in [1, 1000000]");
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  hb::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      ctx.status, static_cast<unsigned long long>(timeout_us) * 1000ull);
  return hb::launch_status("wait_selftest_kernel launch");
}
