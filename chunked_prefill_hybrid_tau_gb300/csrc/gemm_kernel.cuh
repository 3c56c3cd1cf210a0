// The persistent tcgen05 GEMM kernel template shared by the bf16 and the
// E4M3 projections (instantiated in gemm.cu and gemm_e4m3.cu).
//
// Packed-token projections on the 5th-generation tensor cores:
//   C = epilogue(A B^T),  A [M][K] (activations), B [N][K] (weights), both
//   bf16 (kind::f16) or both E4M3 with per-row scales of A and B applied to
//   the fp32 accumulators in the epilogue (kind::f8f6f4).
//
// These are the linear layers whose cost model the pages use (Sarathi-Serve
// reading notes, section 1.6: T = max(T_math, T_mem) with
// T_math = 2 n d_in d_out / FLOPS and T_mem = (d_in d_out bytes_w + ...) / BW).
//
// Design (sm_103a):
//   * persistent grid (<= one CTA per SM), 128 x BN output tiles walked with
//     the M index fastest, so the CTAs that share a weight tile run together
//     and the weights stream from HBM once;
//   * warp 0: TMA producer.  128-byte swizzled 128-row (A) and BN-row (B)
//     boxes of one 128-byte k-block (64 bf16 or 128 E4M3 elements)
//     into a STAGES-deep shared-memory ring, completion via mbarrier tx bytes;
//   * warp 1: one elected thread issues tcgen05.mma (M=128, N=BN, 32 bytes
//     of K per instruction) into a TMEM accumulator; tcgen05.commit frees a ring slot
//     and, after the last K block, signals the epilogue;
//   * warps 2-5: epilogue.  tcgen05.ld 32x32b (warp w reads TMEM lanes
//     32*(w%4)..), fused STORE / RESIDUAL / SWIGLU / F32 epilogue, then the
//     accumulator buffer is handed back.  Two accumulator buffers let the
//     epilogue of one tile overlap the main loop of the next.  A CTA's last
//     tile has nothing to overlap, so its epilogue uses the then idle ring:
//     the residual tile (and a split-K partner's partial) arrive by TMA /
//     bulk copy, the outputs are staged in 128-byte swizzled rows and leave
//     by TMA stores, instead of one row per thread through the load/store
//     units.
//   * every wait is bounded (device.cuh); on expiry the kernel unwinds.
#pragma once
#include <cuda_bf16.h>

#include "device.cuh"
#include "runtime.h"

namespace hb {
namespace {

using namespace dev;

constexpr int BM = 128;
// K elements per k-block: one 128-byte swizzle row of the operand type
// (64 bf16 or 128 E4M3), so both types use the same shared-memory layout.
template <bool F8>
constexpr int bk_elems() { return F8 ? 128 : 64; }
constexpr int kThreads = 192;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 192 ? 5 : 6);
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
};

struct Params {
  int M, N, K;
  void* C;
  const void* R;
  int ldc;       // row stride of C and R (elements)
  int out_cols;  // valid output columns (N, or N/2 for SWIGLU)
  int* status;
  GemmNorm norm;  // folded RMSNorm: row scaling in (STORE, SWIGLU), row statistics out (RESIDUAL)
  int ksplit;     // 1, or 2: each tile's K range in two halves (RESIDUAL only)
  float* part;    // ksplit 2: fp32 partial tiles [tile][half][BN][BM] (column-major)
  int* flags;     // ksplit 2: per 128-row tile arrival counters (index 4 x tile), zero at launch
  const float* sa;  // E4M3 operands: per-row scales of A [M] and of B [N] (null for bf16)
  const float* sb;
  GemmRope rope;    // kEpiRope: destinations and RoPE table of the fused QKV epilogue
};

// Work unit u: tile u / ksplit, K half u % ksplit (k-blocks [kb0, kb1)).
// The two halves of a tile are consecutive units, so they run at the same
// time on neighbouring CTAs.
struct Unit {
  int tile, half, m0, n_blk, kb0, kb1;
};

template <int BN>
__device__ __forceinline__ Unit unit_of(const Params& p, int u, int m_tiles, int kblocks) {
  Unit w;
  w.tile = u / p.ksplit;
  w.half = u - w.tile * p.ksplit;
  w.m0 = (w.tile % m_tiles) * BM;
  w.n_blk = w.tile / m_tiles;
  const int per = (kblocks + p.ksplit - 1) / p.ksplit;
  w.kb0 = w.half * per;
  w.kb1 = w.kb0 + per < kblocks ? w.kb0 + per : kblocks;
  return w;
}

// silu(g) = g / (1 + e^-g).  The fast divide (2 ulp) is far below the bf16
// rounding of the result; an IEEE divide here made the SwiGLU epilogue the
// most expensive part of the gate/up projection.  For g -> -inf the
// denominator overflows to inf and the quotient is 0, the correct limit.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, __fadd_rn(1.0f, __expf(-g))); }

// Inverse RMS of one row from its 32-column partial sums of squares, summed
// in column order: rsqrt(sum / d + eps).
__device__ __forceinline__ float row_inv_rms(const GemmNorm& nm, int row) {
  const float2* sp = reinterpret_cast<const float2*>(nm.ss_in + static_cast<size_t>(row) * nm.parts);
  float ss = 0.f;
  for (int i = 0; i < nm.parts / 2; ++i) {
    const float2 v = sp[i];
    ss += v.x;
    ss += v.y;
  }
  return rsqrtf(ss * nm.inv_d + nm.eps);
}

// Store 32 accumulator columns [col, col+32) of one row, 16-byte segments
// past the last valid column skipped (STORE: scaled by `scale`, the row's
// folded RMSNorm factor, else 1; F32: as is).
template <int EPI>
__device__ __forceinline__ void store_chunk(const Params& p, int row, int col, const uint32_t (&r)[32], float scale) {
  const int ncols = p.out_cols;
  if constexpr (EPI == HB_EPI_F32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.C) + static_cast<size_t>(row) * p.ldc + col);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (col + 4 * i < ncols)
        dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                             __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
  } else {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack_bf16x2(__fmul_rn(__uint_as_float(r[2 * i]), scale), __fmul_rn(__uint_as_float(r[2 * i + 1]), scale));
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.C) + static_cast<size_t>(row) * p.ldc + col);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (col + 8 * i < ncols) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// Sum of squares of 32 bf16 values held as 16 packed pairs, formed as
// row_sumsq_kernel forms a 32-column part: an fma chain over each 8-value
// vector, then (v0 + v1) + (v2 + v3).  Every producer of row statistics
// uses this order, so a row's statistics have the same bits whichever
// kernel wrote them.
__device__ __forceinline__ float sumsq32(const uint32_t (&w)[16]) {
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[4 * i + j]);
      a = __fmaf_rn(f.x, f.x, a);
      a = __fmaf_rn(f.y, f.y, a);
    }
    v[i] = a;
  }
  return __fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3]));
}

// RESIDUAL: C = R + acc for 32 columns, with the residual already loaded
// (rv); writes the sum of squares of the 32 rounded outputs to ss_dst when
// it is given.
__device__ __forceinline__ void residual_chunk(const Params& p, int row, int col, const uint32_t (&r)[32],
                                               const uint4 (&rv)[4], float* ss_dst) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t rr[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(rr[j]);
      const int e = 8 * i + 2 * j;
      w[4 * i + j] = pack_bf16x2(__fadd_rn(f.x, __uint_as_float(r[e])), __fadd_rn(f.y, __uint_as_float(r[e + 1])));
    }
  }
  if (ss_dst) *ss_dst = sumsq32(w);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.C) + static_cast<size_t>(row) * p.ldc + col);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (col + 8 * i < p.out_cols) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// E4M3 operands: acc * rowf * sb[col + j] for 32 accumulator columns, in
// place (rowf = the row's scale times its folded RMSNorm factor, if any);
// columns at or past N get scale 0.
// The products are rounded explicitly (no contraction into a later add), so
// every epilogue path produces the same bits.
__device__ __forceinline__ void scale_cols(uint32_t (&r)[32], float rowf, const float* sb, int col, int N) {
  const float4* s4 = reinterpret_cast<const float4*>(sb + col);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 s = col + 4 * i < N ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    r[4 * i] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[4 * i]), rowf), s.x));
    r[4 * i + 1] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[4 * i + 1]), rowf), s.y));
    r[4 * i + 2] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[4 * i + 2]), rowf), s.z));
    r[4 * i + 3] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[4 * i + 3]), rowf), s.w));
  }
}

// Split K: the two halves of a 128-row tile exchange partial sums by
// columns.  Each CTA has written its fp32 partial of the other half's
// columns; here it arrives on the tile's counter and waits (bounded) for the
// partner's arrival, after which the partner's partial of its own columns is
// in place.  Own + partner is commutative, so either half's sum has the same
// bits.  The counters must be zero at launch (the layer clears them in a
// kernel ahead of its projections); both halves of a tile run in the same round of the
// persistent grid (consecutive units on an even number of clusters).
__device__ __forceinline__ bool split_exchange(const Params& p, int stile, bool leader, volatile int* ep_flag,
                                               volatile int* abort_flag) {
  __threadfence();
  named_barrier_sync(1, 128);
  if (leader) {
    int* arrive = p.flags + stile * 4;
    atomicAdd(arrive, 1);
    int ok = 1;
    const uint64_t t0 = globaltimer();
    while (*reinterpret_cast<volatile int*>(arrive) < 2) {
      if (*abort_flag || globaltimer() - t0 > kWaitTimeoutNs) {
        if (!*abort_flag) flag_error(p.status, kStatusTimeout);
        *abort_flag = 1;
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    *ep_flag = ok;
  }
  named_barrier_sync(1, 128);
  return *ep_flag != 0;
}

// Epilogue of one 128 x BN accumulator block in TMEM (t_base: this warp's
// 32 lanes) for output row `row` of the warp's thread: SwiGLU, residual (with
// the split-K exchange on 128-row tile `stile`, K half `half`) or store.
// scale: the row's folded RMSNorm factor; rowf: scale times the row's E4M3
// scale (F8).
template <int BN, int EPI, bool F8>
__device__ __forceinline__ void epilogue_tile(const Params& p, uint32_t t_base, int row, bool row_ok, int rloc,
                                              int n_blk, int stile, int half, bool leader, volatile int* ep_flag,
                                              volatile int* abort_flag, float scale, float rowf) {
  if (EPI == HB_EPI_SWIGLU) {
#pragma unroll 1
    for (int j = 0; j < BN / 128; ++j) {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(t_base + j * 128 + h * 32, g);
        tmem_ld_32x32b_x32(t_base + j * 128 + 64 + h * 32, u);
        tmem_ld_wait();
        const int col = n_blk * (BN / 2) + j * 64 + h * 32;
        if (row_ok && col < p.out_cols) {
          if constexpr (F8) {
            // gate and up rows of w_gu have their own scales
            const int bcol = n_blk * BN + j * 128 + h * 32;
            scale_cols(g, rowf, p.sb, bcol, p.N);
            scale_cols(u, rowf, p.sb, bcol + 64, p.N);
          }
          const float sc = F8 ? 1.f : scale;
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = __fmul_rn(silu(__fmul_rn(__uint_as_float(g[2 * i]), sc)), __fmul_rn(__uint_as_float(u[2 * i]), sc));
            const float a1 =
                __fmul_rn(silu(__fmul_rn(__uint_as_float(g[2 * i + 1]), sc)), __fmul_rn(__uint_as_float(u[2 * i + 1]), sc));
            w[i] = pack_bf16x2(a0, a1);
          }
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.C) +
                                                static_cast<size_t>(row) * p.ldc + col);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (col + 8 * i < p.out_cols) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  } else {
    // columns this CTA finishes: all, or with split K its half of them (the
    // other half's partial goes to the partner CTA)
    constexpr int NC = BN / 32;
    int c_lo = 0, c_hi = NC;
    const float* other = nullptr;
    bool finish = true;
    if (p.ksplit == 2) {
      c_lo = half * (NC / 2);
      c_hi = c_lo + NC / 2;
      float* mine = p.part + (static_cast<size_t>(stile) * 2 + half) * BN * BM;
#pragma unroll 1
      for (int c = 0; c < NC; ++c) {
        if (c >= c_lo && c < c_hi) continue;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) mine[static_cast<size_t>(c * 32 + j) * BM + rloc] = __uint_as_float(r[j]);
      }
      finish = split_exchange(p, stile, leader, ep_flag, abort_flag);
      other = p.part + (static_cast<size_t>(stile) * 2 + (1 - half)) * BN * BM;
    }
    if (finish && EPI == HB_EPI_RESIDUAL) {
      // software-pipelined: the residual (and the other half's partial)
      // of chunk c + 1 is in flight while chunk c is combined and stored
      uint4 rv[2][4];
      float ov[2][32];
      auto fetch = [&](int c, int b) {
        const int col = n_blk * BN + c * 32;
        const uint4* res = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.R) +
                                                          static_cast<size_t>(row) * p.ldc + col);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          rv[b][i] = (row_ok && col + 8 * i < p.out_cols) ? res[i] : make_uint4(0, 0, 0, 0);
        if (other != nullptr) {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[b][j] = __ldcg(other + static_cast<size_t>(c * 32 + j) * BM + rloc);
        }
      };
      const int n_own = c_hi - c_lo;
      fetch(c_lo, 0);
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        if (i >= n_own) break;
        const int c = c_lo + i;
        const int b = i & 1;
        if (i + 1 < n_own) fetch(c + 1, b ^ 1);
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + c * 32, r);
        tmem_ld_wait();
        if (other != nullptr) {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), ov[b][j]));
        }
        const int col = n_blk * BN + c * 32;
        if constexpr (F8) scale_cols(r, rowf, p.sb, col, p.N);
        float* ss_dst = p.norm.ss_out != nullptr
                            ? p.norm.ss_out + static_cast<size_t>(row) * p.norm.parts + col / 32
                            : nullptr;
        if (row_ok && col < p.out_cols) residual_chunk(p, row, col, r, rv[b], ss_dst);
      }
    } else if (finish) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + c * 32, r);
        tmem_ld_wait();
        const int col = n_blk * BN + c * 32;
        if constexpr (F8) scale_cols(r, rowf, p.sb, col, p.N);
        if (row_ok && col < p.out_cols) store_chunk<EPI>(p, row, col, r, F8 ? 1.f : scale);
      }
    }
  }
}

// Byte offset of 16-byte chunk c (0..7) of row r in a staged slab of 128
// rows x 128 bytes with the 128-byte swizzle (the TMA box layout).
__device__ __forceinline__ uint32_t slab_off(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }
constexpr int kSlabBytes = 128 * 128;

// Epilogue of a CTA's last 128 x BN accumulator block, staged through the
// ring (idle once the tile's MMAs are done; at least 192 KB):
//   STORE / F32 / SWIGLU: outputs into 128-byte slabs, then TMA stores;
//   RESIDUAL: the residual tile arrives by TMA into the slabs (issued as soon
//   as the accumulator is ready) and is overwritten in place by the outputs;
//   with split K each of the tile's two CTAs finishes half of the columns:
//   it writes its fp32 partial of the other half (column-major, coalesced),
//   meets the partner on the tile's counter and fetches the partner's partial
//   of its own half with one bulk copy.
// Called by the 128 epilogue threads; `leader` is one of them.  Returns
// false when a bounded wait expired.  This code runs once per CTA and
// often cold, so its instruction fetches weigh as much as its arithmetic:
// the 32-column steps of the residual path are not unrolled (bf16 layer
// 233.0 -> 231.7 us), those of the SwiGLU and store paths only with E4M3
// operands (their longer code with the scales: E4M3 layer 206.1 -> 202.3
// us; with bf16, not unrolling them cost 2 us).  Measured on one GB300,
// 1500 steps per variant.
template <int BN, int EPI, bool F8>
__device__ __forceinline__ bool epilogue_last(const Params& p, const CUtensorMap* tmC, const CUtensorMap* tmR,
                                              uint8_t* ring, uint64_t* ep_bar, volatile int* ep_flag, uint32_t t_base,
                                              int m0, int row, bool row_ok, int rloc, int n_blk, int stile, int half,
                                              bool leader, float scale, float rowf, volatile int* abort_flag) {
  if constexpr (EPI == HB_EPI_RESIDUAL) {
    // the columns this CTA finishes: all, or with split K its half (the
    // other half's partial goes to the partner CTA, whose partial of these
    // columns comes in by one bulk copy)
    constexpr int NS_ALL = BN / 64;  // 64-column bf16 slabs
    const bool split = p.ksplit == 2;
    const int ns = split ? NS_ALL / 2 : NS_ALL;
    const int cl0 = split ? half * (BN / 2) : 0;  // first accumulator column finished here
    constexpr int NP = 2 * NS_ALL;  // 32-column statistics parts of the tile
    static_assert(NS_ALL * kSlabBytes + (BN / 2) * BM * 4 + BM * NP * 4 <= 192 * 1024,
                  "ring too small for the split epilogue");
    uint8_t* part_smem = ring + NS_ALL * kSlabBytes;
    // this thread's row statistics, collected here and written as one vector
    float* ss_sm = reinterpret_cast<float*>(part_smem + (BN / 2) * BM * 4) + rloc * NP;
    if (leader) {
      mbar_arrive_expect_tx(&ep_bar[0], ns * kSlabBytes);
      for (int s = 0; s < ns; ++s) tma_load_2d(ring + s * kSlabBytes, tmR, &ep_bar[0], n_blk * BN + cl0 + s * 64, m0);
    }
    if (split) {
      float* mine = p.part + (static_cast<size_t>(stile) * 2 + half) * BN * BM;
      const int o0 = (1 - half) * (BN / 2);  // the partner's columns
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + o0 + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) mine[static_cast<size_t>(o0 + c * 32 + j) * BM + rloc] = __uint_as_float(r[j]);
      }
      const bool ok = split_exchange(p, stile, leader, ep_flag, abort_flag);
      if (leader && ok) {
        fence_proxy_async_global();
        const float* other = p.part + (static_cast<size_t>(stile) * 2 + (1 - half)) * BN * BM + cl0 * BM;
        constexpr uint32_t kPiece = (BN / 2) * BM * 4 / 2;
        mbar_arrive_expect_tx(&ep_bar[1], 2 * kPiece);
        for (int i = 0; i < 2; ++i)
          bulk_load(part_smem + i * kPiece, reinterpret_cast<const uint8_t*>(other) + i * kPiece, kPiece, &ep_bar[1]);
      }
      if (!ok) {
        mbar_wait(&ep_bar[0], 0, nullptr, nullptr);  // the residual copies land before the CTA leaves
        return false;
      }
    }
    if (!mbar_wait(&ep_bar[0], 0, abort_flag, p.status)) return false;
    if (split && !mbar_wait(&ep_bar[1], 0, abort_flag, p.status)) return false;
    const float* other = reinterpret_cast<const float*>(part_smem);  // partner's partial of this CTA's columns
#pragma unroll 1
    for (int s = 0; s < ns; ++s) {
      uint8_t* slab = ring + s * kSlabBytes;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        const int cl = cl0 + s * 64 + h * 32;  // accumulator column within the tile
        tmem_ld_32x32b_x32(t_base + cl, r);
        tmem_ld_wait();
        if (split) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), other[(cl - cl0 + j) * BM + rloc]));
        }
        const int col = n_blk * BN + cl;
        if constexpr (F8) scale_cols(r, rowf, p.sb, col, p.N);
        uint32_t w[16];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint4* q = reinterpret_cast<uint4*>(slab + slab_off(rloc, h * 4 + c4));
          const uint4 rv = *q;
          const uint32_t rr[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = unpack_bf16x2(rr[j]);
            const int e = 8 * c4 + 2 * j;
            w[4 * c4 + j] =
                pack_bf16x2(__fadd_rn(f.x, __uint_as_float(r[e])), __fadd_rn(f.y, __uint_as_float(r[e + 1])));
          }
          *q = make_uint4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
        }
        ss_sm[2 * s + h] = sumsq32(w);
      }
    }
    if (p.norm.ss_out != nullptr && row_ok) {
      // parts (n_blk BN + cl0) / 32 .. + 2 ns - 1 of the row, consecutive
      const int col0 = n_blk * BN + cl0;
      float* dst = p.norm.ss_out + static_cast<size_t>(row) * p.norm.parts + col0 / 32;
      const bool vec = (p.norm.parts % 4) == 0 && (col0 / 32) % 4 == 0 && col0 + 2 * ns * 32 <= p.out_cols;
      if (vec) {
        for (int i = 0; i < 2 * ns; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(ss_sm[i], ss_sm[i + 1], ss_sm[i + 2], ss_sm[i + 3]);
      } else {
        for (int i = 0; i < 2 * ns; ++i)
          if (col0 + i * 32 < p.out_cols) dst[i] = ss_sm[i];
      }
    }
    fence_proxy_async_smem();
    named_barrier_sync(1, 128);
    if (leader) {
      for (int s = 0; s < ns; ++s) tma_store_2d(tmC, ring + s * kSlabBytes, n_blk * BN + cl0 + s * 64, m0);
      bulk_commit_group();
    }
    return true;
  } else if constexpr (EPI == HB_EPI_SWIGLU) {
    constexpr int NS = BN / 128;  // each 128 accumulator columns (gate 64 | up 64) give a 64-column slab
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      uint8_t* slab = ring + s * kSlabBytes;
#pragma unroll(F8 ? 1 : 2)
      for (int h = 0; h < 2; ++h) {
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(t_base + s * 128 + h * 32, g);
        tmem_ld_32x32b_x32(t_base + s * 128 + 64 + h * 32, u);
        tmem_ld_wait();
        if constexpr (F8) {
          const int bcol = n_blk * BN + s * 128 + h * 32;
          scale_cols(g, rowf, p.sb, bcol, p.N);
          scale_cols(u, rowf, p.sb, bcol + 64, p.N);
        }
        const float sc = F8 ? 1.f : scale;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = 8 * c4 + 2 * j;
            const float a0 = __fmul_rn(silu(__fmul_rn(__uint_as_float(g[e]), sc)), __fmul_rn(__uint_as_float(u[e]), sc));
            const float a1 = __fmul_rn(silu(__fmul_rn(__uint_as_float(g[e + 1]), sc)), __fmul_rn(__uint_as_float(u[e + 1]), sc));
            w[j] = pack_bf16x2(a0, a1);
          }
          *reinterpret_cast<uint4*>(slab + slab_off(rloc, h * 4 + c4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    fence_proxy_async_smem();
    named_barrier_sync(1, 128);
    if (leader) {
      for (int s = 0; s < NS; ++s) tma_store_2d(tmC, ring + s * kSlabBytes, n_blk * (BN / 2) + s * 64, m0);
      bulk_commit_group();
    }
    return true;
  } else {
    // STORE (bf16, 64 columns per slab) or F32 (fp32, 32 columns per slab)
    constexpr int SC = EPI == HB_EPI_F32 ? 32 : 64;
    constexpr int NS = BN / SC;
#pragma unroll 1
    for (int s = 0; s < NS; ++s) {
      uint8_t* slab = ring + s * kSlabBytes;
#pragma unroll(F8 ? 1 : 2)
      for (int h = 0; h < SC / 32; ++h) {
        uint32_t r[32];
        const int cl = s * SC + h * 32;
        tmem_ld_32x32b_x32(t_base + cl, r);
        tmem_ld_wait();
        if constexpr (F8) scale_cols(r, rowf, p.sb, n_blk * BN + cl, p.N);
        if constexpr (EPI == HB_EPI_F32) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(slab + slab_off(rloc, c)) = make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
        } else {
          const float sc = F8 ? 1.f : scale;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int e = 8 * c4 + 2 * j;
              w[j] = pack_bf16x2(__fmul_rn(__uint_as_float(r[e]), sc), __fmul_rn(__uint_as_float(r[e + 1]), sc));
            }
            *reinterpret_cast<uint4*>(slab + slab_off(rloc, h * 4 + c4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    fence_proxy_async_smem();
    named_barrier_sync(1, 128);
    if (leader) {
      for (int s = 0; s < NS; ++s) tma_store_2d(tmC, ring + s * kSlabBytes, n_blk * BN + s * SC, m0);
      bulk_commit_group();
    }
    return true;
  }
}

// QKV epilogue with RoPE and the KV append (kEpiRope) for one 128 x BN
// accumulator block whose columns are whole heads (BN a multiple of
// d_head): per head and per 32 dimensions i of its first half, the thread's
// row takes accumulator columns i and i + d_head/2, rounds them to bf16 as
// the STORE epilogue would (the qkv activations), rotates q and k heads by
// the row's position (rotate-half: x_i cos - x_{i+d/2} sin and
// x_{i+d/2} cos + x_i sin, each product and sum rounded to fp32 as in
// kv_append_kernel) and writes q to its row, K and V to the row's slot.
// An out-of-range position skips the row; an out-of-range slot skips its
// K/V; both set the status word (as kv_append_kernel).  Each thread writes
// its own row in 16-byte pieces.  (Staging the rows in the idle ring and
// writing whole rows per warp measured slower.)
template <int BN, bool F8>
__device__ __forceinline__ void epilogue_rope(const Params& p, uint32_t t_base, int row, bool row_ok, int n_blk,
                                              float scale, float rowf) {
  const GemmRope& rp = p.rope;
  const int DH = rp.d_head, HALF = DH / 2;
  const int pos = row_ok ? __ldg(rp.row_pos + row) : 0;
  const int slot = row_ok ? __ldg(rp.slots + row) : 0;
  const bool pos_ok = row_ok && pos >= 0 && pos < rp.max_pos;
  const bool slot_ok = pos_ok && slot >= 0 && slot < rp.num_slots;
  if (row_ok && (!pos_ok || slot >= rp.num_slots)) flag_error(p.status, kStatusIndex);
  const int page = slot / 16, off = slot % 16;
  const float sc = F8 ? 1.f : scale;
  auto* q_out = static_cast<__nv_bfloat16*>(rp.q_out);
  auto* kc = static_cast<__nv_bfloat16*>(rp.k_cache);
  auto* vc = static_cast<__nv_bfloat16*>(rp.v_cache);
#pragma unroll 1
  for (int hb = 0; hb < BN; hb += DH) {
    const int col0 = n_blk * BN + hb;  // the head's first column
    const int head = col0 / DH;
    const bool rot = head < rp.n_q + rp.n_kv;
    __nv_bfloat16* dst = nullptr;
    if (head < rp.n_q) {
      dst = pos_ok ? q_out + (static_cast<size_t>(row) * rp.n_q + head) * DH : nullptr;
    } else if (rot) {
      dst = slot_ok ? kc + ((static_cast<size_t>(page) * rp.n_kv + (head - rp.n_q)) * 16 + off) * DH : nullptr;
    } else {
      dst = slot_ok ? vc + ((static_cast<size_t>(page) * rp.n_kv + (head - rp.n_q - rp.n_kv)) * 16 + off) * DH
                    : nullptr;
    }
#pragma unroll 1
    for (int c = 0; c < HALF; c += 32) {
      // (cos, sin) of dimensions c .. c + 31 at the row's position, all loads
      // in flight together (the accumulator loads overlap them)
      float4 cs[16];
      const float4* csp = reinterpret_cast<const float4*>(rp.rope + static_cast<size_t>(pos) * HALF + c);
#pragma unroll
      for (int i = 0; i < 16; ++i) cs[i] = rot && pos_ok ? __ldg(csp + i) : make_float4(1.f, 0.f, 1.f, 0.f);
      uint32_t r1[32], r2[32];
      tmem_ld_32x32b_x32(t_base + hb + c, r1);
      tmem_ld_32x32b_x32(t_base + hb + HALF + c, r2);
      tmem_ld_wait();
      if constexpr (F8) {
        scale_cols(r1, rowf, p.sb, col0 + c, p.N);
        scale_cols(r2, rowf, p.sb, col0 + HALF + c, p.N);
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {  // 8 dimensions (one 16-byte piece per half) at a time
        uint32_t w1[4], w2[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 8 * g + 2 * j;
          // the bf16 activations of the projection
          const float2 a = unpack_bf16x2(pack_bf16x2(__fmul_rn(__uint_as_float(r1[e]), sc),
                                                     __fmul_rn(__uint_as_float(r1[e + 1]), sc)));
          const float2 b = unpack_bf16x2(pack_bf16x2(__fmul_rn(__uint_as_float(r2[e]), sc),
                                                     __fmul_rn(__uint_as_float(r2[e + 1]), sc)));
          if (rot) {
            const float4 t = cs[e >> 1];  // (cos, sin) of dimensions e and e + 1
            w1[j] = pack_bf16x2(__fsub_rn(__fmul_rn(a.x, t.x), __fmul_rn(b.x, t.y)),
                                __fsub_rn(__fmul_rn(a.y, t.z), __fmul_rn(b.y, t.w)));
            w2[j] = pack_bf16x2(__fadd_rn(__fmul_rn(b.x, t.x), __fmul_rn(a.x, t.y)),
                                __fadd_rn(__fmul_rn(b.y, t.z), __fmul_rn(a.y, t.w)));
          } else {
            w1[j] = pack_bf16x2(a.x, a.y);
            w2[j] = pack_bf16x2(b.x, b.y);
          }
        }
        if (dst != nullptr) {
          *reinterpret_cast<uint4*>(dst + c + 8 * g) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
          *reinterpret_cast<uint4*>(dst + HALF + c + 8 * g) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
        }
      }
    }
  }
}

template <int BN, int EPI, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR, Params p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* ep_bar = drain + 1;  // last-tile epilogue: residual copies, partner partial
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ep_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ep_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (p.M + BM - 1) / BM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  const int units = tiles * p.ksplit;
  constexpr int BK = bk_elems<F8>();
  const int kblocks = (p.K + BK - 1) / BK;  // TMA zero-fills columns past K

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(drain, 1);
    mbar_init(&ep_bar[0], 1);
    mbar_init(&ep_bar[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t pending = 0;  // stages armed and not yet seen consumed (bit mask)
      uint32_t armed_parity = 0;
      // The weights do not come from the previous kernel: the first ring
      // fill of B is issued before waiting for it, then A follows.  Up to 8
      // row tiles, a weight box is read by the CTAs of its column tile at
      // about the same time and not again in the layer: first out of L2.
      // With more rows the larger activations push the box out between its
      // readers, and the default policy is faster (measured at 2048 and
      // 4096 rows).
      const uint64_t wpol = m_tiles <= 8 ? policy_evict_first() : policy_evict_normal();
      int pre = 0;
      if (static_cast<int>(blockIdx.x) < units) {
        const Unit w = unit_of<BN>(p, blockIdx.x, m_tiles, kblocks);
        pre = w.kb1 - w.kb0 < C::STAGES ? w.kb1 - w.kb0 : C::STAGES;
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
          tma_load_2d_hint(smem + i * C::STAGE_BYTES + C::A_BYTES, &tmB, &full[i], (w.kb0 + i) * BK, w.n_blk * BN,
                           wpol);
        }
      }
      griddep_wait();
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of<BN>(p, u, m_tiles, kblocks);
        const int m0 = w.m0;
        const int n0 = w.n_blk * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          if (u == static_cast<int>(blockIdx.x) && kb - w.kb0 < pre) {
            // stage armed and its B box issued above (fresh barrier, phase 0)
            pending |= 1u << stage;
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, m0);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            pending |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, m0);
            tma_load_2d_hint(sa + C::A_BYTES, &tmB, &full[stage], kb * BK, n0, wpol);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let copies already in flight land before the CTA exits; a stage
        // whose empty wait succeeded later was consumed, so only the last
        // STAGES arms can be outstanding
        for (int s = 0; s < C::STAGES; ++s)
          if (pending & (1u << s)) mbar_drain(&full[s], (armed_parity >> s) & 1u);
      }
    }
    if (lane != 0) griddep_wait();
  } else if (warp == 1) {
    griddep_wait();
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int t = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++t) {
        const Unit w = unit_of<BN>(p, u, m_tiles, kblocks);
        const int acc = t & 1;
        const uint32_t acc_phase = (t >> 1) & 1;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
          // four MMAs of 32 bytes of K each (16 bf16 or 32 E4M3 elements)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (F8)
              mma_e4m3(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), kIdesc,
                       (kb != w.kb0 || k != 0) ? 1u : 0u);
            else
              mma_bf16(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), kIdesc,
                       (kb != w.kb0 || k != 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(&acc_full[acc]);
      }
      if (!ok) {
        // make sure no MMA is still reading shared memory or writing TMEM
        mma_commit(drain);
        mbar_drain(drain, 0);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    griddep_wait();
    const int quarter = warp & 3;
    const bool leader = warp == 2 && lane == 0;
    int t = 0;
    for (int un = blockIdx.x; un < units; un += gridDim.x, ++t) {
      const Unit wu = unit_of<BN>(p, un, m_tiles, kblocks);
      const int acc = t & 1;
      const uint32_t acc_phase = (t >> 1) & 1;
      const int m0 = wu.m0;
      const int n_blk = wu.n_blk;
      const int rloc = quarter * 32 + lane;  // row within the tile
      const int row = m0 + rloc;
      const bool row_ok = row < p.M;
      // the row's folded RMSNorm factor, read before the accumulator is ready
      const float scale = (p.norm.ss_in != nullptr && row_ok) ? row_inv_rms(p.norm, row) : 1.f;
      const float rowf = F8 && row_ok ? scale * p.sa[row] : scale;
      bool ok = mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      if constexpr (EPI == kEpiRope) {
        epilogue_rope<BN, F8>(p, t_base, row, row_ok, n_blk, scale, rowf);
      } else if (un + static_cast<int>(gridDim.x) >= units) {
        // the CTA's last tile: the ring is idle, stage through it
        ok = epilogue_last<BN, EPI, F8>(p, &tmC, &tmR, smem, ep_bar, ep_flag, t_base, m0, row, row_ok, rloc, n_blk,
                                        wu.tile, wu.half, leader, scale, rowf, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
      } else {
        epilogue_tile<BN, EPI, F8>(p, t_base, row, row_ok, rloc, n_blk, wu.tile, wu.half, leader, ep_flag, abort_flag,
                                   scale, rowf);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
    if (leader) bulk_wait_group<0>();  // the TMA stores have left shared memory and are performed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- CTA pairs
// A cluster of two CTAs on neighbouring SMs computes 256 x BN tiles with
// tcgen05.mma.cta_group::2: each CTA holds its 128 rows of A and its BN / 2
// of the tile's BN B rows (the even CTA the first half) in shared memory, the
// even CTA's MMA thread issues M = 256, N = BN MMAs, and each CTA's tensor
// memory receives its own 128 accumulator rows.  At BN = 256 every SM streams
// 32 KB per k-block for the FLOPs a one-CTA 128 x 256 tile streams 48 KB for.
//   * both CTAs' TMA loads of a stage complete on the even CTA's `full`
//     barrier (armed once with both CTAs' bytes); the MMA commit frees the
//     stage in both CTAs (multicast), and after a tile's last k-block it
//     signals both CTAs' accumulator barriers;
//   * the epilogue warps of both CTAs hand the accumulator buffer back on the
//     even CTA's `acc_empty` (count 8);
//   * a tile of the pair covers 128-row tiles 2 pm and 2 pm + 1 of the
//     single-CTA numbering, so split-K partials and counters are shared with
//     gemm_kernel's layout.
constexpr int kPairBN = 256;  // the tile width of split-K pair projections
template <int BN>
struct CfgPair {
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = (BN / 2) * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 6 : (BN == 192 ? 7 : 8);
  static constexpr int TMEM_COLS = 512;  // two BN-column accumulators
  static_assert(BN == 128 || BN == 192 || BN == 256, "pair tile width");
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
};

struct PairUnit {
  int pm, n_blk, half, kb0, kb1;
};

__device__ __forceinline__ PairUnit pair_unit_of(const Params& p, int u, int pm_tiles, int kblocks) {
  PairUnit w;
  const int tile = u / p.ksplit;
  w.half = u - tile * p.ksplit;
  w.pm = tile % pm_tiles;
  w.n_blk = tile / pm_tiles;
  const int per = (kblocks + p.ksplit - 1) / p.ksplit;
  w.kb0 = w.half * per;
  w.kb1 = w.kb0 + per < kblocks ? w.kb0 + per : kblocks;
  return w;
}

template <int BN, int EPI, bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR, Params p) {
  using C = CfgPair<BN>;
  constexpr int BK = bk_elems<F8>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);  // even CTA's are used
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;  // even CTA's are used
  uint64_t* drain = acc_empty + 2;
  uint64_t* ep_bar = drain + 1;  // last-tile epilogue (this CTA's own): residual copies, partner partial
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ep_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* ep_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int m_tiles = (p.M + BM - 1) / BM;
  const int pm_tiles = (m_tiles + 1) / 2;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int units = pm_tiles * n_tiles * p.ksplit;
  const int kblocks = (p.K + BK - 1) / BK;
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int n_clusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);
    }
    mbar_init(drain, 1);
    mbar_init(&ep_bar[0], 1);
    mbar_init(&ep_bar[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t pending = 0, armed_parity = 0;  // stages loaded and not yet seen released
      // The weights do not come from the previous kernel: the first ring
      // fill of B is issued before waiting for it, then A follows.  Up to 4
      // pair row tiles (1024 rows), a weight box is read by the clusters of
      // its column tile at about the same time and not again in the layer:
      // first out of L2 (with the decode K/V stream also first out, the
      // 512-row layer is 2% faster).  With more rows the activations push
      // the box out between its readers, and the default policy is faster.
      const uint64_t wpol = pm_tiles <= 4 ? policy_evict_first() : policy_evict_normal();
      int pre = 0;
      if (cluster < units) {
        const PairUnit w = pair_unit_of(p, cluster, pm_tiles, kblocks);
        const int n0 = w.n_blk * BN + static_cast<int>(rank) * (BN / 2);
        pre = w.kb1 - w.kb0 < C::STAGES ? w.kb1 - w.kb0 : C::STAGES;
        for (int i = 0; i < pre; ++i) {
          if (leader) mbar_arrive_expect_tx(&full[i], 2 * C::STAGE_BYTES);  // both CTAs' boxes
          tma_load_2d_pair_hint(smem + i * C::STAGE_BYTES + C::A_BYTES, &tmB, cluster_addr(&full[i], 0),
                                (w.kb0 + i) * BK, n0, wpol);
        }
      }
      griddep_wait();
      for (int u = cluster; u < units && ok; u += n_clusters) {
        const PairUnit w = pair_unit_of(p, u, pm_tiles, kblocks);
        const int m0 = (2 * w.pm + static_cast<int>(rank)) * BM;
        const int n0 = w.n_blk * BN + static_cast<int>(rank) * (BN / 2);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          const uint32_t fb = cluster_addr(&full[stage], 0);
          if (u == cluster && kb - w.kb0 < pre) {
            // stage armed and its B box issued above (fresh barriers)
            pending |= 1u << stage;
            tma_load_2d_pair(sa, &tmA, fb, kb * BK, m0);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            pending |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);  // both CTAs' boxes
            tma_load_2d_pair(sa, &tmA, fb, kb * BK, m0);
            tma_load_2d_pair_hint(sa + C::A_BYTES, &tmB, fb, kb * BK, n0, wpol);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Normally every loaded stage is consumed by a pair MMA before the MMA
      // thread drains, and the final cluster barrier follows that drain.
      // After an expired wait, let the boxes still in flight land (their
      // stage is released once consumed; a short bounded wait otherwise).
      if (*abort_flag) raise_peer_abort(abort_flag, rank);
      if (!ok)
        for (int s2 = 0; s2 < C::STAGES; ++s2)
          if (pending & (1u << s2)) mbar_drain(&empty[s2], (armed_parity >> s2) & 1u);
    }
  } else if (warp == 1) {
    griddep_wait();
    // ---------------------------------------------------------- MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t kIdesc = F8 ? idesc_e4m3_f32(2 * BM, BN) : idesc_bf16_f32(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int t = 0;
      bool ok = true;
      for (int u = cluster; u < units && ok; u += n_clusters, ++t) {
        const PairUnit w = pair_unit_of(p, u, pm_tiles, kblocks);
        const int acc = t & 1;
        const uint32_t acc_phase = (t >> 1) & 1;
        if (!mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (F8)
              mma_e4m3_pair(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), kIdesc,
                            (kb != w.kb0 || k != 0) ? 1u : 0u);
            else
              mma_bf16_pair(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), kIdesc,
                            (kb != w.kb0 || k != 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty[stage], 3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit_pair(&acc_full[acc], 3);
      }
      if (*abort_flag) raise_peer_abort(abort_flag, rank);
      // no pair MMA may still read either CTA's shared memory or write its
      // tensor memory when the CTAs leave
      mma_commit_pair(drain, 1);
      mbar_drain(drain, 0);
    }
  } else {
    // ---------------------------------------------------------- epilogue (both CTAs)
    griddep_wait();
    const int quarter = warp & 3;
    const bool leader_thread = warp == 2 && lane == 0;
    int t = 0;
    for (int un = cluster; un < units; un += n_clusters, ++t) {
      const PairUnit wu = pair_unit_of(p, un, pm_tiles, kblocks);
      const int acc = t & 1;
      const uint32_t acc_phase = (t >> 1) & 1;
      const int mt = 2 * wu.pm + static_cast<int>(rank);  // this CTA's 128-row tile
      const int rloc = quarter * 32 + lane;
      const int row = mt * BM + rloc;
      const bool row_ok = row < p.M;
      const float scale = (p.norm.ss_in != nullptr && row_ok) ? row_inv_rms(p.norm, row) : 1.f;
      const float rowf = F8 && row_ok ? scale * p.sa[row] : scale;
      bool ok = mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      if (mt < m_tiles) {  // a 128-row tile wholly past M (odd tile count) has nothing to write
        const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
        const int stile = mt + m_tiles * wu.n_blk;
        if constexpr (EPI == kEpiRope) {
          epilogue_rope<BN, F8>(p, t_base, row, row_ok, wu.n_blk, scale, rowf);
        } else if (un + n_clusters >= units) {
          // the CTA's last tile: its ring is idle, stage through it
          ok = epilogue_last<BN, EPI, F8>(p, &tmC, &tmR, smem, ep_bar, ep_flag, t_base, mt * BM, row, row_ok, rloc,
                                          wu.n_blk, stile, wu.half, leader_thread, scale, rowf, abort_flag);
        } else {
          epilogue_tile<BN, EPI, F8>(p, t_base, row, row_ok, rloc, wu.n_blk, stile, wu.half, leader_thread, ep_flag,
                                     abort_flag, scale, rowf);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&acc_empty[acc], 0));
      if (!__all_sync(0xffffffffu, ok)) break;
    }
    if (leader_thread) bulk_wait_group<0>();  // the TMA stores have left shared memory and are performed
    if (lane == 0 && *abort_flag) raise_peer_abort(abort_flag, rank);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

// Tensor maps of the output and the residual for the last-tile epilogue:
// 128-row boxes of one 128-byte row (64 bf16 or 32 fp32 columns), 128-byte
// swizzle.
template <int EPI>
hb_status encode_out_maps(CUtensorMap* tmC, CUtensorMap* tmR, void* Cp, const void* R, int ldc, int M, int out_cols) {
  const int esz = EPI == HB_EPI_F32 ? 4 : 2;
  hb_status st = encode_tmap_2d(tmC, Cp, out_cols, M, static_cast<uint64_t>(ldc) * esz, 128 / esz, BM, true, esz);
  if (st != HB_OK) return st;
  if (EPI != HB_EPI_RESIDUAL) {
    *tmR = *tmC;
    return HB_OK;
  }
  return encode_tmap_2d(tmR, R, out_cols, M, static_cast<uint64_t>(ldc) * 2, 64, BM, true, 2);
}

template <int BN, int EPI, bool F8>
hb_status launch_pair(const DeviceCtx& ctx, const void* A, int lda, const float* sa, const void* B, const float* sb,
                      void* Cp, int ldc, const void* R, int M, int N, int K, const GemmNorm* norm,
                      const GemmSplit* split, cudaStream_t stream, const GemmRope* rope = nullptr) {
  using C = CfgPair<BN>;
  constexpr int BK = bk_elems<F8>();
  constexpr int ESZ = F8 ? 1 : 2;
  CUtensorMap tmA, tmB, tmC, tmR;
  hb_status st = encode_tmap_2d(&tmA, A, K, M, static_cast<uint64_t>(lda) * ESZ, BK, BM, true, ESZ);
  if (st != HB_OK) return st;
  st = encode_tmap_2d(&tmB, B, K, N, static_cast<uint64_t>(K) * ESZ, BK, BN / 2, true, ESZ);
  if (st != HB_OK) return st;
  if constexpr (EPI == kEpiRope) {
    tmC = tmA;  // no tiled stores: the fused epilogue writes q, K and V rows itself
    tmR = tmA;
  } else {
    st = encode_out_maps<EPI>(&tmC, &tmR, Cp, R, ldc, M, EPI == HB_EPI_SWIGLU ? N / 2 : N);
    if (st != HB_OK) return st;
  }
  static std::atomic<bool> attr_set[kMaxDevices];
  st = smem_limit_once(attr_set, ctx.device, gemm_pair_kernel<BN, EPI, F8>, C::SMEM, "cudaFuncSetAttribute(gemm pair)");
  if (st != HB_OK) return st;
  Params p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = Cp;
  p.R = R;
  p.ldc = ldc;
  p.out_cols = EPI == HB_EPI_SWIGLU ? N / 2 : N;
  p.status = ctx.status;
  p.norm = norm ? *norm : GemmNorm{};
  p.ksplit = split ? 2 : 1;
  p.part = split ? split->part : nullptr;
  p.flags = split ? split->flags : nullptr;
  p.sa = sa;
  p.sb = sb;
  p.rope = rope ? *rope : GemmRope{};
  const int m_tiles = (M + BM - 1) / BM;
  const int units = ((m_tiles + 1) / 2) * ((N + BN - 1) / BN) * p.ksplit;
  const int pairs = ctx.num_sms / 2;
  const int grid = 2 * (units < pairs ? units : pairs);
  return launch_pdl(gemm_pair_kernel<BN, EPI, F8>, grid, kThreads, C::SMEM, stream, "gemm_pair_kernel launch", tmA, tmB,
                    tmC, tmR, p);
}

// A [M][K] (row stride lda elements), B [N][K]; sa/sb: E4M3 scales (F8 only).
template <int BN, int EPI, bool F8>
hb_status launch(const DeviceCtx& ctx, const void* A, int lda, const float* sa, const void* B, const float* sb,
                 void* Cp, int ldc, const void* R, int M, int N, int K, const GemmNorm* norm, const GemmSplit* split,
                 cudaStream_t stream, const GemmRope* rope = nullptr) {
  using C = Cfg<BN>;
  constexpr int BK = bk_elems<F8>();
  constexpr int ESZ = F8 ? 1 : 2;
  CUtensorMap tmA, tmB, tmC, tmR;
  hb_status st = encode_tmap_2d(&tmA, A, K, M, static_cast<uint64_t>(lda) * ESZ, BK, BM, true, ESZ);
  if (st != HB_OK) return st;
  st = encode_tmap_2d(&tmB, B, K, N, static_cast<uint64_t>(K) * ESZ, BK, BN, true, ESZ);
  if (st != HB_OK) return st;
  if constexpr (EPI == kEpiRope) {
    tmC = tmA;  // no tiled stores: the fused epilogue writes q, K and V rows itself
    tmR = tmA;
  } else {
    st = encode_out_maps<EPI>(&tmC, &tmR, Cp, R, ldc, M, EPI == HB_EPI_SWIGLU ? N / 2 : N);
    if (st != HB_OK) return st;
  }
  static std::atomic<bool> attr_set[kMaxDevices];
  st = smem_limit_once(attr_set, ctx.device, gemm_kernel<BN, EPI, F8>, C::SMEM, "cudaFuncSetAttribute(gemm)");
  if (st != HB_OK) return st;
  Params p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = Cp;
  p.R = R;
  p.ldc = ldc;
  p.out_cols = EPI == HB_EPI_SWIGLU ? N / 2 : N;
  p.status = ctx.status;
  p.norm = norm ? *norm : GemmNorm{};
  p.ksplit = split ? 2 : 1;
  p.part = split ? split->part : nullptr;
  p.flags = split ? split->flags : nullptr;
  p.sa = sa;
  p.sb = sb;
  p.rope = rope ? *rope : GemmRope{};
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int units = tiles * p.ksplit;
  const int grid = units < ctx.num_sms ? units : ctx.num_sms;
  return launch_pdl(gemm_kernel<BN, EPI, F8>, grid, kThreads, C::SMEM, stream, "gemm_kernel launch", tmA, tmB, tmC,
                    tmR, p);
}

// Tile width: fewest waves of tiles over the SMs, weighted by a per-tile
// cost that grows with BN (plus a fixed per-tile overhead).
inline int choose_bn(int M, int N, int epi, int num_sms) {
  const int cands_swiglu[2] = {256, 128};
  const int cands[3] = {256, 192, 128};
  const bool whole = epi == HB_EPI_SWIGLU || epi == kEpiRope;  // tiles of whole 128-column groups
  const int* c = whole ? cands_swiglu : cands;
  const int nc = whole ? 2 : 3;
  const int m_tiles = (M + BM - 1) / BM;
  int best = 128;
  double best_cost = 1e30;
  for (int i = 0; i < nc; ++i) {
    const int bn = c[i];
    if (whole ? N % bn != 0 : (N % bn != 0 && bn != 128)) continue;
    const int tiles = m_tiles * ((N + bn - 1) / bn);
    const int waves = (tiles + num_sms - 1) / num_sms;
    const double cost = waves * (bn + 32.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

}  // namespace
}  // namespace hb
