// Varlen paged hybrid attention: chunk rows on the tensor cores
// (attention_tc.cu), decode rows here on the HBM path, and the split of the
// SMs between the two.
//
// What it computes (Sarathi-Serve reading notes, sections 3.1 and 7.5b;
// Chunked Prefill page, mechanism section): a prompt chunk's query at
// position p attends to keys 0..p of its request -- the cached prefix
// written by earlier chunks plus the causal part of its own chunk -- and a
// decode row attends to its whole context.  Keys are read through the
// sequence's block table from 16-token pages.
//
// Decode unit: one decode row x one kv head (its n_q/n_kv q heads as the
// rows of an m16n8k16 MMA) x one SPLIT-key range at fixed absolute
// positions, so the result of a row never depends on its batch companions.
// Each warp owns whole units and streams the unit's pages (K and V of one kv
// head, one TMA box of 16 keys x 64 dims per half) through its own ring with
// the 128-byte swizzle that makes the ldmatrix reads conflict-free.  Split
// results are combined in split order by the last warp to finish a
// (row, kv head).
#include <cuda_bf16.h>


#include "device.cuh"
#include "runtime.h"

namespace hb {
namespace {

using namespace dev;

constexpr int SPLIT = 1024;                 // keys per decode split
constexpr int HALF_BYTES = 16 * 128;        // one 64-dim half of a page: 16 keys x 128-byte rows
constexpr int MAX_SEQS = 1024;

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int* q_start;
  const int* kv_len;
  const int* block_table;
  int S, T, max_pages, num_pages, n_q, n_kv, grp, max_kv_len;
  float scale_log2;
  int* work_counter;
  int* combine_counters;
  float* partials;
  int* status;
  // 1 when the chunk kernel precedes this one on the stream: that kernel
  // waited for the inputs before letting this one start, so the wait here
  // is deferred to the end (this grid's completion then implies the chunk
  // kernel's, which the next kernel on the stream relies on)
  int wait_at_end;
};

__device__ __forceinline__ int upper_index(const int* pre, int n, int u) {
  // largest s in [0, n) with pre[s] <= u (pre non-decreasing, pre[0] = 0)
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------- MMA helpers
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Byte offset of (key 0..15, 16-byte chunk 0..D/8-1) in one swizzled K or V
// page: 64-dim halves of 16 rows x 128 bytes, chunk index XOR row.
__device__ __forceinline__ uint32_t blk_off(int key, int chunk) {
  const int r = key & 15;
  return (chunk >> 3) * HALF_BYTES + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
}

// One warp, one 16-key page: S = Q K^T (rows a = lane/4 and b = a + 8 of the
// q-head group; keys above `lim` masked), online-softmax update in log2
// units, O += P V with P rounded to bf16 for the MMA.
template <int D>
__device__ __forceinline__ void warp_page(uint32_t k_base, uint32_t v_base, int key0, const uint32_t (&qa)[D / 16][4],
                                          float (&o)[D / 8][4], float (&m)[2], float (&l)[2], int lim,
                                          float scale_log2, int lane) {
  const int mat = lane >> 3, rr = lane & 7, t = lane & 3;
  float s[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  {
    const int key = ((mat >> 1) << 3) + rr;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t b[4];
      ldsm_x4(k_base + blk_off(key, 2 * kk + (mat & 1)), b);
      mma16816(s[0], qa[kk], b[0], b[1]);
      mma16816(s[1], qa[kk], b[2], b[3]);
    }
  }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = key0 + 8 * j + 2 * t + (e & 1);
      const float v = key <= lim ? s[j][e] * scale_log2 : -INFINITY;
      s[j][e] = v;
      mx[e >> 1] = fmaxf(mx[e >> 1], v);
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
  }
  float alpha[2], muse[2];
  bool grew = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float mn = fmaxf(m[h], mx[h]);
    muse[h] = mn == -INFINITY ? 0.f : mn;
    grew |= mn > m[h];
    alpha[h] = ex2_approx(m[h] - muse[h]);  // 1 when the maximum did not grow
    m[h] = mn;
  }
  float rs[2] = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pv = ex2_approx(s[j][e] - muse[e >> 1]);
      s[j][e] = pv;
      rs[e >> 1] += pv;
    }
  }
  l[0] = l[0] * alpha[0] + rs[0];
  l[1] = l[1] * alpha[1] + rs[1];
  // rescale O only when some row's maximum grew (else alpha = 1 exactly)
  if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }
  }
  uint32_t pa[4];
  pa[0] = pack_bf16x2(s[0][0], s[0][1]);
  pa[1] = pack_bf16x2(s[0][2], s[0][3]);
  pa[2] = pack_bf16x2(s[1][0], s[1][1]);
  pa[3] = pack_bf16x2(s[1][2], s[1][3]);
  const int key = ((mat & 1) << 3) + rr;
#pragma unroll
  for (int jd = 0; jd < D / 16; ++jd) {
    uint32_t b[4];
    ldsm_x4_t(v_base + blk_off(key, 2 * jd + (mat >> 1)), b);
    mma16816(o[2 * jd], pa, b[0], b[1]);
    mma16816(o[2 * jd + 1], pa, b[2], b[3]);
  }
}

__device__ __forceinline__ uint32_t ld_q2(const __nv_bfloat16* rowp, int col, bool ok) {
  return ok ? __ldg(reinterpret_cast<const unsigned int*>(rowp + col)) : 0u;
}

// ---------------------------------------------------------------- decode rows
// HBM path.  Each warp owns whole units -- one decode row x one kv head (its
// q-head group as MMA rows) x one SPLIT-key range at fixed absolute
// positions -- and streams the unit's 16-token pages through its own
// DR-deep ring of TMA boxes, refilling a slot as soon as it has consumed it.
// No cross-warp synchronisation: partial results go straight from registers
// to the split records, and the last warp to finish a (row, kv head)
// combines the splits in split order.
constexpr int kDecWarps = 8;

template <int D>
struct DC {
  static constexpr int PAGE_BYTES = (D / 64) * HALF_BYTES;  // one page of one kv head, K or V
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;        // K page then V page
  static constexpr int DR = D == 128 ? 3 : 6;               // ring depth per warp
  static constexpr int REC_FLOATS = 16 * D + 32;
  static constexpr int RING_BYTES = kDecWarps * DR * STAGE_BYTES;  // multiple of 1024
  static constexpr int BAR_BYTES = kDecWarps * DR * 8;               // mbarriers: 8-byte aligned after the rings
  static constexpr int BT_BYTES = kDecWarps * (SPLIT / 16) * 4;    // per-warp copy of a unit's page ids
  static constexpr int SMEM = RING_BYTES + BAR_BYTES + BT_BYTES + (MAX_SEQS + 1) * 4 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kDecWarps * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Params p) {
  using C = DC<D>;
  constexpr int DR = C::DR, STAGE_BYTES = C::STAGE_BYTES, PAGE_BYTES = C::PAGE_BYTES, REC_FLOATS = C::REC_FLOATS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);
  int* btc_all = reinterpret_cast<int*>(smem + C::RING_BYTES + C::BAR_BYTES);
  int* dpre = btc_all + kDecWarps * (SPLIT / 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ga = lane >> 2, t4 = lane & 3;
  griddep_launch_dependents();
  if (!p.wait_at_end) griddep_wait();

  for (int s = tid; s < p.S; s += blockDim.x) {
    const int q0 = p.q_start[s], q1 = p.q_start[s + 1];
    const int kvl = p.kv_len[s];
    int d = 0;
    if (q1 - q0 == 1) {
      if (q0 < 0 || q1 > p.T || kvl < 1 || kvl > p.max_kv_len || (kvl + 15) / 16 > p.max_pages)
        flag_error(p.status, kStatusIndex);
      else
        d = p.n_kv * ((kvl + SPLIT - 1) / SPLIT);
    }
    dpre[s + 1] = d;
  }
  if (tid < kDecWarps * DR) mbar_init(&bars[tid], 1);
  if (tid == 0) fence_barrier_init();
  __syncthreads();
  if (tid == 0) {
    dpre[0] = 0;
    for (int s = 1; s <= p.S; ++s) dpre[s] += dpre[s - 1];
  }
  __syncthreads();
  const int total = dpre[p.S];
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }

  uint8_t* ring = smem + warp * DR * STAGE_BYTES;
  uint64_t* full = bars + warp * DR;
  int* btc = btc_all + warp * (SPLIT / 16);
  uint32_t phases = 0;  // bit s: parity to wait for on slot s
  while (true) {
    int u = 0;
    if (lane == 0) u = atomicAdd(p.work_counter + 1, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= total) break;
    const int s = upper_index(dpre, p.S, u);
    const int local = u - dpre[s];
    const int kvl = p.kv_len[s];
    const int g = local % p.n_kv;
    const int split = local / p.n_kv;
    const int key_begin = split * SPLIT;
    const int key_end = min(kvl, key_begin + SPLIT);
    const int nsplit = (kvl + SPLIT - 1) / SPLIT;
    const int npages = (key_end - key_begin + 15) / 16;
    const int page0 = key_begin / 16;
    const int* bt = p.block_table + static_cast<size_t>(s) * p.max_pages;
    const int row = p.q_start[s];
    // the unit's page ids, validated once, into this warp's shared copy
    for (int b = lane; b < npages; b += 32) {
      int page = bt[page0 + b];
      if (page < 0 || page >= p.num_pages) {
        flag_error(p.status, kStatusIndex);
        page = 0;
      }
      btc[b] = page;
    }
    __syncwarp();

    // page b of this unit into slot b % DR: lane 0 arms the slot, lanes 0
    // and 1 then issue one TMA box each (the whole K or V page, both halves)
    auto issue = [&](int b) {
      const int slot = b % DR;
      uint8_t* dst = ring + slot * STAGE_BYTES;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], STAGE_BYTES);
      __syncwarp();
      if (lane < 2) {
        const int page = btc[b];
        const int y = (page * p.n_kv + g) * 16;
        const bool is_v = lane & 1;
        // each decode K/V byte is read once: first out of L2, so the stream
        // does not push out what is read again (the chunk rows' prefix K/V,
        // activations, code)
        tma_load_3d_hint(dst + (is_v ? PAGE_BYTES : 0), is_v ? &tmV : &tmK, &full[slot], 0, y, 0,
                         policy_evict_first());
      }
    };
    for (int b = 0; b < min(DR, npages); ++b) issue(b);

    // q rows of this kv head's group (rows >= grp are zero padding)
    const bool oka = ga < p.grp, okb = ga + 8 < p.grp;
    const size_t qbase = static_cast<size_t>(row) * p.n_q + g * p.grp;
    const __nv_bfloat16* qra = p.q + (qbase + (oka ? ga : 0)) * D;
    const __nv_bfloat16* qrb = p.q + (qbase + (okb ? ga + 8 : 0)) * D;
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = ld_q2(qra, 16 * kk + 2 * t4, oka);
      qa[kk][1] = ld_q2(qrb, 16 * kk + 2 * t4, okb);
      qa[kk][2] = ld_q2(qra, 16 * kk + 8 + 2 * t4, oka);
      qa[kk][3] = ld_q2(qrb, 16 * kk + 8 + 2 * t4, okb);
    }
    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    const int lim = key_end - 1;

    bool ok = true;
    for (int b = 0; b < npages; ++b) {
      const int slot = b % DR;
      bool fok = mbar_wait(&full[slot], (phases >> slot) & 1u, nullptr, p.status);
      phases ^= 1u << slot;
      if (!__all_sync(0xffffffffu, fok)) {
        ok = false;
        break;
      }
      uint8_t* st = ring + slot * STAGE_BYTES;
      const int key0 = key_begin + 16 * b;
      const bool tail = key0 + 16 > key_end;
      if (tail) {
        // keys past key_end may hold uninitialised memory: zero their V rows
        uint4* vb = reinterpret_cast<uint4*>(st + PAGE_BYTES);
        const int first = key_end - key0;
        for (int i = lane; i < (16 - first) * (D / 8); i += 32) {
          const int key = first + i / (D / 8), c = i % (D / 8);
          vb[blk_off(key, c) / 16] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      const uint32_t kb = smem_u32(st);
      warp_page<D>(kb, kb + PAGE_BYTES, key0, qa, o, m, l, lim, p.scale_log2, lane);
      // slot consumed.  Reads are complete (their results fed the MMAs); the
      // zeroing writes of a tail page must be ordered before the next TMA write.
      if (tail) fence_proxy_async_smem();
      __syncwarp();
      if (b + DR < npages) issue(b + DR);
    }
    if (!ok) {
      // unwind: let this warp's copies in flight land (bounded) before exiting
      if (lane == 0)
        for (int sl = 0; sl < DR; ++sl) mbar_drain(&full[sl], (phases >> sl) & 1u);
      break;
    }

#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
    __nv_bfloat16* orow = p.out + static_cast<size_t>(row) * p.n_q * D + g * p.grp * D;
    if (nsplit == 1) {
      const float ia = l[0] > 0.f ? 1.f / l[0] : 0.f, ib = l[1] > 0.f ? 1.f / l[1] : 0.f;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const int col = 8 * j + 2 * t4;
        if (oka) *reinterpret_cast<uint32_t*>(orow + ga * D + col) = pack_bf16x2(o[j][0] * ia, o[j][1] * ia);
        if (okb) *reinterpret_cast<uint32_t*>(orow + (ga + 8) * D + col) = pack_bf16x2(o[j][2] * ib, o[j][3] * ib);
      }
      continue;
    }
    // split record (unnormalised O, running max in log2 units, row sum)
    float* rec = p.partials + static_cast<size_t>(u) * REC_FLOATS;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      const int col = 8 * j + 2 * t4;
      if (oka) *reinterpret_cast<float2*>(rec + ga * D + col) = make_float2(o[j][0], o[j][1]);
      if (okb) *reinterpret_cast<float2*>(rec + (ga + 8) * D + col) = make_float2(o[j][2], o[j][3]);
    }
    if (t4 == 0) {
      rec[16 * D + ga] = m[0];
      rec[16 * D + ga + 8] = m[1];
      rec[16 * D + 16 + ga] = l[0];
      rec[16 * D + 16 + ga + 8] = l[1];
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      int* cnt = p.combine_counters + s * p.n_kv + g;
      const int old = atomicAdd(cnt, 1);
      last = old == nsplit - 1;
      if (last) *cnt = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __threadfence();
    // combine the splits of this (row, kv head) in split order: lane r < grp
    // finds row r's max and sum over splits; then each lane owns 4 columns
    // of up to four rows at a time and issues the split loads of all of
    // them before accumulating (one round trip to L2 per group of four
    // rows, not one per row: this combine ends the kernel's longest units)
    const float* rec0 = p.partials + static_cast<size_t>(u - split * p.n_kv) * REC_FLOATS;
    const size_t rstride = static_cast<size_t>(p.n_kv) * REC_FLOATS;
    float Mr = -INFINITY, Lr = 0.f;
    if (lane < p.grp) {
#pragma unroll 4
      for (int sp = 0; sp < nsplit; ++sp) Mr = fmaxf(Mr, __ldcg(rec0 + sp * rstride + 16 * D + lane));
#pragma unroll 4
      for (int sp = 0; sp < nsplit; ++sp) {
        const float* rs = rec0 + sp * rstride;
        Lr += __ldcg(rs + 16 * D + 16 + lane) * exp2f(__ldcg(rs + 16 * D + lane) - Mr);
      }
    }
    for (int r0 = 0; r0 < p.grp; r0 += 4) {
      const int nr = min(4, p.grp - r0);
      float M[4], inv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        M[i] = __shfl_sync(0xffffffffu, Mr, r0 + i);  // r0 + i < 16: rows past grp are never used
        const float L = __shfl_sync(0xffffffffu, Lr, r0 + i);
        inv[i] = L > 0.f ? 1.f / L : 0.f;
      }
      for (int c4 = lane; c4 < D / 4; c4 += 32) {
        float4 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int sp = 0; sp < nsplit; ++sp) {
          const float* rs = rec0 + sp * rstride;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i < nr) {
              const int r = r0 + i;
              const float wgt = exp2f(__ldcg(rs + 16 * D + r) - M[i]);
              const float4 ov = __ldcg(reinterpret_cast<const float4*>(rs + r * D) + c4);
              acc[i].x += wgt * ov.x;
              acc[i].y += wgt * ov.y;
              acc[i].z += wgt * ov.z;
              acc[i].w += wgt * ov.w;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i < nr)
            *reinterpret_cast<uint2*>(orow + (r0 + i) * D + 4 * c4) =
                make_uint2(pack_bf16x2(acc[i].x * inv[i], acc[i].y * inv[i]),
                           pack_bf16x2(acc[i].z * inv[i], acc[i].w * inv[i]));
        }
      }
    }
  }
  if (p.wait_at_end) griddep_wait();
}

// ---------------------------------------------------------------- SM split
// Chunk rows (tensor cores, latency-bound per tile) and decode rows (HBM
// streaming) cannot share an SM (each kernel fills its shared memory), so
// when the plan's hints give both kinds of work the SMs are split and the
// two persistent kernels run at the same time on disjoint SMs, both on the
// caller's stream: the decode kernel is a programmatic dependent of the
// chunk kernel and starts beside it.  Cost model (GB300, measured):
//   chunk : U = 128-row tiles x q heads units of about kUnitUs + (key blocks
//           per tile) x kBlockUs each (key blocks over all tiles ~ pairs /
//           128^2 + rows / 128), taken heaviest first, so on n SMs the
//           makespan is about W / n + half a unit, and at least the heaviest
//           unit;
//   decode: the larger of bytes / min(kDecodeBw, n x kDecodeBwPerSm) and
//           ceil(units / (8 warps x n)) x kSplitUs, with units ~ 1.1 x
//           pairs / SPLIT x n_kv (one warp streams one SPLIT-key unit).
// The split is the middle of the chunk shares within 2% of the best
// max(t_c, t_d) (the decode's one-round boundary is sharp), or none when
// running the two one after the other is estimated faster.  It only moves
// work between SMs: every row's result is the same for any split.
constexpr double kUnitUs = 8.0;             // per chunk unit, d_head 128
constexpr double kBlockUs = 1.5;            // per 128-key block of a chunk unit, d_head 128
constexpr double kSplitUs = 50.0;           // one full decode split on one warp, d_head 128
constexpr double kDecodeBwPerSm = 55000.0;  // bytes per us per SM
constexpr double kDecodeBw = 6.2e6;         // bytes per us, whole GPU

// CTAs for the chunk kernel when both paths run concurrently (the decode
// kernel gets the rest); 0 = run them one after the other on all SMs.
int chunk_sms(const DeviceCtx& ctx, const hb_device_plan& plan, const hb_layer_dims& dm) {
  const int S = ctx.num_sms;
  if (plan.chunk_pairs <= 0 || plan.decode_pairs <= 0 || plan.chunk_rows <= 0 || S < 4) return 0;
  const double dscale = dm.d_head / 128.0;
  const double blk = kBlockUs * (0.5 + 0.5 * dscale);
  const double rows = static_cast<double>(plan.chunk_rows);
  const double tiles = ceil(rows / 128.0);
  const double units_c = tiles * dm.n_q;
  const double blocks = static_cast<double>(plan.chunk_pairs) / 16384.0 + rows / 128.0;
  const double t_unit = kUnitUs + blocks / tiles * blk;
  const double t_max = t_unit + (tiles - 1.0) / 2.0 * blk;
  const double work_c = units_c * t_unit;
  const double bytes_d = static_cast<double>(plan.decode_pairs) * dm.n_kv * dm.d_head * 4.0;
  const double units_d = 1.1 * static_cast<double>(plan.decode_pairs) / SPLIT * dm.n_kv;
  auto t_chunk = [&](int n) {
    if (units_c <= n) return t_max;
    const double t = work_c / n + 0.5 * t_unit;
    return t > t_max ? t : t_max;
  };
  auto t_decode = [&](int n) {
    const double bw = n * kDecodeBwPerSm < kDecodeBw ? n * kDecodeBwPerSm : kDecodeBw;
    const double t_bw = bytes_d / bw;
    const double t_units = ceil(units_d / (kDecWarps * n)) * kSplitUs * dscale;
    return t_bw > t_units ? t_bw : t_units;
  };
  auto t_both = [&](int n) { return t_chunk(n) > t_decode(S - n) ? t_chunk(n) : t_decode(S - n); };
  double best = 1e300;
  for (int n = 1; n < S; ++n)
    if (t_both(n) < best) best = t_both(n);
  if (best >= t_chunk(S) + t_decode(S)) return 0;
  int lo = S, hi = 0;
  for (int n = 1; n < S; ++n)
    if (t_both(n) <= best * 1.02) {
      lo = n < lo ? n : lo;
      hi = n;
    }
  // Decode SMs beyond the number whose streams reach the whole GPU's
  // bandwidth add contention, not speed (64 decodes to 8192 keys beside a
  // 192-row chunk: 193.5 us with 112 decode SMs, 199 us with 130): within
  // the window, give the chunk kernel at least the SMs past that number.
  const int n_sat = static_cast<int>(ceil(kDecodeBw / kDecodeBwPerSm));
  if (lo < S - n_sat && S - n_sat <= hi) lo = S - n_sat;
  return (lo + hi) / 2;
}

template <int D>
hb_status attention_launch_d(const DeviceCtx& ctx, const void* q, const hb_device_plan& plan, const hb_layer_dims& dm,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmK3,
                             const CUtensorMap& tmV3, Params p, cudaStream_t stream) {
  static std::atomic<bool> attr_set[kMaxDevices];
  hb_status st0 = smem_limit_once(attr_set, ctx.device, decode_kernel<D>, DC<D>::SMEM, "cudaFuncSetAttribute(decode)");
  if (st0 != HB_OK) return st0;
  // Chunk rows first, then decode rows, both on `stream` with programmatic
  // serialization: the chunk kernel takes nc SMs (all of them when run one
  // after the other) and the decode kernel starts beside it on the rest as
  // soon as every chunk CTA has passed its wait for the inputs.  Both are
  // launched whatever the hints say (a kernel without work exits at once),
  // so results never depend on the hints.
  const int nc = chunk_sms(ctx, plan, dm);
  hb_status st = chunk_tc_launch(ctx, q, tmK, tmV, plan, dm, p.num_pages, p.max_kv_len, p.out, p.work_counter,
                                 nc > 0 ? nc : ctx.num_sms, stream);
  if (st != HB_OK) return st;
  p.wait_at_end = 1;
  return launch_pdl(decode_kernel<D>, nc > 0 ? ctx.num_sms - nc : ctx.num_sms, kDecWarps * 32, DC<D>::SMEM, stream,
                    "decode_kernel launch", tmK3, tmV3, p);
}

}  // namespace

size_t attention_counter_bytes(const hb_layer_dims& dm, int n_seqs) {
  const size_t c = 256 + static_cast<size_t>(n_seqs) * dm.n_kv * 4;
  return (c + 255) & ~size_t(255);
}

size_t attention_workspace_bytes(const hb_layer_dims& dm, int max_seqs, int max_kv_len) {
  const size_t splits = (static_cast<size_t>(max_kv_len) + SPLIT - 1) / SPLIT;
  const size_t units = static_cast<size_t>(max_seqs) * dm.n_kv * splits;
  return attention_counter_bytes(dm, max_seqs) + units * (16 * static_cast<size_t>(dm.d_head) + 32) * 4;
}

hb_status attention_launch(const DeviceCtx& ctx, const void* q, const void* k_cache, const void* v_cache,
                           int num_pages, const hb_device_plan& plan, const hb_layer_dims& dm, int max_kv_len,
                           void* out, void* ws, size_t ws_bytes, cudaStream_t stream, bool counters_zeroed) {
  HB_REQUIRE(dm.d_head == 128 || dm.d_head == 64, "hb_attention: d_head must be 64 or 128");
  HB_REQUIRE(plan.n_seqs <= MAX_SEQS, "hb_attention: at most %d sequences per iteration", MAX_SEQS);
  HB_REQUIRE(plan.n_seqs >= 0 && plan.n_rows >= 0 && plan.max_pages >= 1, "hb_attention: bad plan sizes");
  HB_REQUIRE(max_kv_len >= 1, "hb_attention: max_kv_len >= 1");
  if (plan.n_seqs == 0 || plan.n_rows == 0) return HB_OK;
  const size_t need = attention_workspace_bytes(dm, plan.n_seqs, max_kv_len);
  HB_REQUIRE(ws != nullptr && ws_bytes >= need, "hb_attention: workspace of %zu bytes needed, %zu given", need,
             ws_bytes);
  HB_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "hb_attention: workspace must be 256-byte aligned");
  CUtensorMap tmK, tmV, tmK3, tmV3;  // 2-D half-page boxes (chunk kernel), 3-D whole pages (decode kernel)
  const uint64_t rows = static_cast<uint64_t>(num_pages) * dm.n_kv * 16;
  hb_status st = encode_tmap_2d(&tmK, k_cache, dm.d_head, rows, dm.d_head * 2, 64, 16, true);
  if (st != HB_OK) return st;
  st = encode_tmap_2d(&tmV, v_cache, dm.d_head, rows, dm.d_head * 2, 64, 16, true);
  if (st != HB_OK) return st;
  st = encode_tmap_kv_pages(&tmK3, k_cache, rows, dm.d_head);
  if (st != HB_OK) return st;
  st = encode_tmap_kv_pages(&tmV3, v_cache, rows, dm.d_head);
  if (st != HB_OK) return st;
  const size_t counters = attention_counter_bytes(dm, plan.n_seqs);
  if (!counters_zeroed) {
    st = cuda_status(cudaMemsetAsync(ws, 0, counters, stream), "cudaMemsetAsync(attention counters)");
    if (st != HB_OK) return st;
  }
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.q_start = plan.seq_q_start;
  p.kv_len = plan.seq_kv_len;
  p.block_table = plan.block_table;
  p.S = plan.n_seqs;
  p.T = plan.n_rows;
  p.max_kv_len = max_kv_len;
  p.max_pages = plan.max_pages;
  p.num_pages = num_pages;
  p.n_q = dm.n_q;
  p.n_kv = dm.n_kv;
  p.grp = dm.n_q / dm.n_kv;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(dm.d_head)));
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  p.work_counter = reinterpret_cast<int*>(w8);  // [0] chunk tiles, [1] decode units
  p.combine_counters = reinterpret_cast<int*>(w8 + 256);
  p.partials = reinterpret_cast<float*>(w8 + counters);
  p.status = ctx.status;
  return dm.d_head == 128 ? attention_launch_d<128>(ctx, q, plan, dm, tmK, tmV, tmK3, tmV3, p, stream)
                          : attention_launch_d<64>(ctx, q, plan, dm, tmK, tmV, tmK3, tmV3, p, stream);
}

}  // namespace hb

extern "C" size_t hb_attention_workspace_bytes(const hb_layer_dims* dims, int32_t max_rows, int32_t max_seqs,
                                               int32_t max_kv_len) {
  (void)max_rows;
  if (!dims || max_seqs < 0 || max_kv_len < 0) return 0;
  return hb::attention_workspace_bytes(*dims, max_seqs, max_kv_len);
}

extern "C" hb_status hb_attention(const void* q, const void* k_cache, const void* v_cache, int32_t num_pages,
                                  const hb_device_plan* plan, const hb_layer_dims* dims, int32_t max_kv_len, void* out,
                                  void* workspace, size_t ws_bytes, void* stream) {
  hb::clear_error();
  hb_status st = hb::check_dims(dims);
  if (st != HB_OK) return st;
  HB_REQUIRE(plan != nullptr, "hb_attention: null plan");
  HB_REQUIRE(q && k_cache && v_cache && out, "hb_attention: null pointer");
  HB_REQUIRE(plan->n_seqs == 0 || (plan->seq_q_start && plan->seq_kv_len && plan->block_table),
             "hb_attention: null plan array");
  HB_REQUIRE(num_pages > 0, "hb_attention: num_pages > 0");
  HB_REQUIRE(hb::aligned16(q) && hb::aligned16(out) && hb::aligned16(k_cache) && hb::aligned16(v_cache),
             "hb_attention: 16-byte alignment");
  hb::DeviceCtx ctx;
  st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  return hb::attention_launch(ctx, q, k_cache, v_cache, num_pages, *plan, *dims, max_kv_len, out, workspace, ws_bytes,
                              static_cast<cudaStream_t>(stream), false);
}
