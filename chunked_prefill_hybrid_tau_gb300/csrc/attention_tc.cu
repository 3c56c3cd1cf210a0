// Chunk-row attention on the 5th-generation tensor cores.
//
// A prompt chunk's query at position p attends to keys 0..p of its request:
// the prefix cached by earlier chunks plus the causal part of its own chunk
// (Sarathi-Serve reading notes, sections 3.1 and 7.5b).  This is the dense,
// tensor-bound half of the hybrid attention; decode rows go to the HBM path.
//
// Work unit: 128 consecutive query rows of one sequence x one q head (GQA: the
// unit's kv head is head / (n_q / n_kv)), keys 0 .. pos_last in 128-key blocks
// read through the block table.  Persistent CTAs take units from a global
// counter, heaviest (latest) tiles first.
//
// Warp roles (352 threads, one CTA per SM):
//   warps 0, 10  TMA producers: warp 0 loads the unit's Q tile (3-D box over
//            [T][n_q][D]) and each block's 8 K pages into a 3-stage K ring,
//            warp 10 the V pages into a 2-stage V ring (16 keys x 64 dims per
//            box, 128-byte swizzle).  A K stage is released when its S block
//            is computed, a V stage when its PV block is.  Block-table entries
//            are read four blocks ahead and checked when used, so the issue
//            cadence is not bound by the latency of those loads;
//   warp 1   MMA issuer (one thread), issuing whichever is ready first:
//            S_j = Q K_j^T into one of two TMEM S buffers (K-major operands),
//            or O += P_j V_j with P read from one of two TMEM P buffers and V
//            as an MN-major shared-memory operand;
//   warps 2-9 softmax, two threads per query row (warps 2-5 take keys 0..63
//            of a block, warps 6-9 keys 64..127; the halves exchange the row
//            maximum once per block): tcgen05.ld of the S half row, causal
//            mask, online softmax in base 2 with a lazily updated maximum (O in
//            TMEM is rescaled only when a row's maximum grows by more than 2^8),
//            P written as bf16 into the block's TMEM P buffer (two buffers, so
//            a block's P waits only for the PV of two blocks back); finally
//            O / l from TMEM to global memory, each thread its half of the
//            head dimension.
// Every wait is bounded; an expired wait sets the status word and unwinds.
#include <cuda_bf16.h>

#include "attention_tc.cuh"

namespace hb {
namespace {

using namespace dev;
using namespace tc;

constexpr int KSTAGE = 3;         // K ring depth: S blocks wait on K loads, so K runs deeper
constexpr int VSTAGE = 2;         // V ring depth

template <int D>
struct TC {
  static constexpr int HALVES = D / 64;
  static constexpr int HALF_TILE = 128 * 128;            // 128 rows x 128 bytes
  static constexpr int Q_BYTES = HALVES * HALF_TILE;     // Q tile
  static constexpr int KV_BYTES = HALVES * HALF_TILE;    // K (or V) block of 128 keys
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;                  // K ring [KSTAGE]
  static constexpr int OFF_V = OFF_K + KSTAGE * KV_BYTES;  // V ring [VSTAGE]
  static constexpr int OFF_BAR = OFF_V + VSTAGE * KV_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int OFF_XCH = OFF_BAR + BAR_BYTES;    // row maxima / sums exchanged by the two halves
  static constexpr int XCH_BYTES = (2 * 2 * 128 + 2 * 128) * 4;
  static constexpr int OFF_PRE = OFF_XCH + XCH_BYTES;
  static constexpr int SMEM = OFF_PRE + (MAX_SEQS + 1) * 4 + 1024;
  static_assert(SMEM <= 232448, "shared memory");
  static constexpr uint32_t TMEM_COLS = 512;             // S0 | S1 | O | P0 | P1
  static constexpr uint32_t COL_O = 256;
  static constexpr uint32_t COL_P = 384;                 // P_b (bf16, 2 keys per column) at COL_P + 64 b
};


struct TcUnit {
  int seq, head, row0, nrows, pos0, nblk, valid;
};


__device__ __forceinline__ TcUnit tc_unit(const TcParams& p, const int* pre, int u) {
  TcUnit w;
  w.valid = u < pre[p.S];
  if (!w.valid) return w;
  const int s = upper_index(pre, p.S, u);
  const int local = u - pre[s];
  const int q0 = p.q_start[s], qlen = p.q_start[s + 1] - q0;
  const int ntiles = (qlen + TQ - 1) / TQ;
  const int t = ntiles - 1 - local / p.n_q;  // heaviest tiles first
  w.seq = s;
  w.head = local % p.n_q;
  w.row0 = q0 + t * TQ;
  w.nrows = min(TQ, qlen - t * TQ);
  w.pos0 = p.kv_len[s] - qlen + t * TQ;
  w.nblk = (w.pos0 + w.nrows + TK - 1) / TK;
  return w;
}



template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, TcParams p) {
  using C = TC<D>;
  // The decode kernel that follows on the stream starts once every CTA here
  // has passed this wait (so the appended K/V and q are complete) and runs
  // beside this kernel on the other SMs.
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bar;                   // [KSTAGE]
  uint64_t* k_empty = bar + 4;              // [KSTAGE]
  uint64_t* v_full = bar + 8;               // [VSTAGE]
  uint64_t* v_empty = bar + 12;             // [VSTAGE]
  uint64_t* q_full = bar + 16;
  uint64_t* q_empty = bar + 17;
  uint64_t* s_full = bar + 18;              // [2]
  uint64_t* s_empty = bar + 20;             // [2]
  uint64_t* o_empty = bar + 22;
  uint64_t* uq_full = bar + 23;             // [2]
  uint64_t* uq_empty = bar + 25;            // [2]
  uint64_t* drain = bar + 27;
  uint64_t* xbar = bar + 28;                // [2] row maxima exchanged (block parity)
  uint64_t* xsbar = bar + 30;               // row sums exchanged (once per unit)
  uint64_t* p_full = bar + 31;              // [2] P_b stored (8 warps), once per use of buffer b
  uint64_t* pv_done = bar + 33;             // [2] the PV that read P_b has completed
  int* uq = reinterpret_cast<int*>(bar + 35);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 36);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xmax = reinterpret_cast<float*>(smem + C::OFF_XCH);  // [2 parity][2 half][128 rows]
  float* xsum = xmax + 2 * 2 * 128;                             // [2 half][128 rows]
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- per-sequence unit counts (chunk sequences: more than one row)
  for (int s = tid; s < p.S; s += kThreads) {
    const int q0 = p.q_start[s], q1 = p.q_start[s + 1];
    const int qlen = q1 - q0, kvl = p.kv_len[s];
    int c = 0;
    if (q0 < 0 || q1 > p.T || qlen < 0 || kvl < qlen || kvl > p.max_kv_len || (kvl + 15) / 16 > p.max_pages)
      flag_error(p.status, kStatusIndex);
    else if (qlen > 1)
      c = p.n_q * ((qlen + TQ - 1) / TQ);
    pre[s + 1] = c;
  }
  if (tid == 0) {
    for (int i = 0; i < KSTAGE; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VSTAGE; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kSoftWarps);
      mbar_init(&uq_full[i], 1);
      mbar_init(&uq_empty[i], 2 + kSoftWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], kSoftWarps);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_empty, kSoftWarps);
    mbar_init(&xbar[0], kSoftWarps);
    mbar_init(&xbar[1], kSoftWarps);
    mbar_init(xsbar, kSoftWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    pre[0] = 0;
    for (int s = 1; s <= p.S; ++s) pre[s] += pre[s - 1];
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    // warp 0: unit queue, Q and the K ring; warp kVWarp: the V ring.  Lane 0
    // arms each stage; the warp's lanes then issue one TMA box each (page
    // lane / HALVES, half lane % HALVES), so a block's 8 pages go out at once.
    const bool kside = warp == 0;
    if (lane == 0) {
      if (kside) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
      } else {
        tma_prefetch_desc(&tmV);
      }
    }
    const CUtensorMap* tm = kside ? &tmK : &tmV;
    uint8_t* ring = kside ? sK : sV;
    uint64_t* full = kside ? k_full : v_full;
    uint64_t* empty = kside ? k_empty : v_empty;
    const int nst = kside ? KSTAGE : VSTAGE;
    int qs = 0, stage = 0, nunit = 0;
    uint32_t qph = 0, kph = 0;
    uint32_t pending = 0, armed = 0;
    bool ok = true;
    while (ok) {
      int u = 0;
      bool got = true;
      if (lane == 0) {
        if (kside) {
          got = mbar_wait(&uq_empty[qs], qph ^ 1u, abort_flag, p.status);
          if (got) {
            u = atomicAdd(p.work_counter, 1);
            uq[qs] = u;
            mbar_arrive(&uq_full[qs]);
          }
        } else {
          got = mbar_wait(&uq_full[qs], qph, abort_flag, p.status);
          if (got) {
            u = uq[qs];
            mbar_arrive(&uq_empty[qs]);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) break;
      u = __shfl_sync(0xffffffffu, u, 0);
      if (++qs == 2) {
        qs = 0;
        qph ^= 1u;
      }
      const TcUnit w = tc_unit(p, pre, u);
      if (!w.valid) break;
      if (kside && lane == 0) {
        // Q tile (the last S block of the previous unit has read it)
        ok = mbar_wait(q_empty, (nunit & 1) ^ 1u, abort_flag, p.status);
        if (ok) {
          mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            tma_load_3d(sQ + hf * C::HALF_TILE, &tmQ, q_full, hf * 64, w.head, w.row0);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      ++nunit;
      const int g = w.head / p.grp;
      const int* bt = p.block_table + static_cast<size_t>(w.seq) * p.max_pages;
      const int key_end = w.pos0 + w.nrows;
      const int my_pg = lane / C::HALVES, my_hf = lane % C::HALVES;
      // this lane's raw page id of block j (0 past the last block), loaded
      // four blocks ahead and checked at use
      auto load_page = [&](int j) {
        const int npg = j < w.nblk ? min(8, (key_end - j * TK + 15) / 16) : 0;
        return my_pg < npg ? __ldg(bt + j * 8 + my_pg) : 0;
      };
      int pf0 = load_page(0), pf1 = load_page(1), pf2 = load_page(2), pf3 = load_page(3);
      for (int j = 0; j < w.nblk; ++j) {
        int cur = pf0;
        pf0 = pf1;
        pf1 = pf2;
        pf2 = pf3;
        pf3 = load_page(j + 4);
        if (cur < 0 || cur >= p.num_pages) {
          flag_error(p.status, kStatusIndex);
          cur = 0;
        }
        const int npg = min(8, (key_end - j * TK + 15) / 16);
        bool eok = true;
        if (lane == 0) {
          eok = mbar_wait(&empty[stage], kph ^ 1u, abort_flag, p.status);
          if (eok) {
            pending |= 1u << stage;
            armed = (armed & ~(1u << stage)) | (kph << stage);
            mbar_arrive_expect_tx(&full[stage], npg * C::HALVES * 2048);
          }
        }
        if (!__shfl_sync(0xffffffffu, eok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (my_pg < npg) {
          uint8_t* dst = ring + stage * C::KV_BYTES + my_hf * C::HALF_TILE + my_pg * 2048;
          tma_load_2d(dst, tm, &full[stage], my_hf * 64, (cur * p.n_kv + g) * 16);
        }
        if (++stage == nst) {
          stage = 0;
          kph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0)
      for (int s = 0; s < nst; ++s)
        if (pending & (1u << s)) mbar_drain(&full[s], (armed >> s) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = lane == 0;
    constexpr uint32_t idS = idesc_bf16_f32(TQ, TK);
    constexpr uint32_t idPV = idesc_bf16_f32(TQ, D) | (1u << 16);  // B (V) is MN-major
    int qs = 0, J = 0, nunit = 0;
    uint32_t qph = 0;
    bool ok = true;
    while (ok) {
      bool got = mbar_wait(&uq_full[qs], qph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int u = uq[qs];
      __syncwarp();
      if (leader) mbar_arrive(&uq_empty[qs]);
      if (++qs == 2) {
        qs = 0;
        qph ^= 1u;
      }
      const TcUnit w = tc_unit(p, pre, u);
      if (!w.valid) break;
      if (leader) {
        ok = mbar_wait(q_full, nunit & 1, abort_flag, p.status);
        const uint32_t q_addr = smem_u32(sQ);
        // S_js and PV_jp are issued in whatever order their inputs arrive
        int js = 0, jp = 0;
        bool o_free = false;
        uint64_t t0 = globaltimer();
        while (ok && jp < w.nblk) {
          bool progressed = false;
          if (js < w.nblk) {
            const int gk = J + js, b = gk & 1, st = gk % KSTAGE;
            if (mbar_test(&k_full[st], (gk / KSTAGE) & 1) && mbar_test(&s_empty[b], ((gk >> 1) & 1) ^ 1u)) {
              tc_fence_after();
              const uint32_t k_addr = smem_u32(sK + st * C::KV_BYTES);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * C::HALF_TILE + (kk & 3) * 32;
                mma_bf16(tmem + b * TK, smem_desc_sw128(q_addr + off), smem_desc_sw128(k_addr + off), idS,
                         kk > 0 ? 1u : 0u);
              }
              mma_commit(&s_full[b]);
              mma_commit(&k_empty[st]);
              if (js == w.nblk - 1) mma_commit(q_empty);
              ++js;
              progressed = true;
            }
          }
          if (jp < js) {
            const int gv = J + jp, st = gv % VSTAGE;
            // O of the previous unit has been read by the epilogue before the first PV
            if (!o_free) o_free = mbar_test(o_empty, (nunit & 1) ^ 1u);
            const int pb = gv & 1;  // P buffer of this block; its use number is gv >> 1
            if (o_free && mbar_test(&p_full[pb], (gv >> 1) & 1) && mbar_test(&v_full[st], (gv / VSTAGE) & 1)) {
              tc_fence_after();
              const uint32_t v_addr = smem_u32(sV + st * C::KV_BYTES);
#pragma unroll
              for (int kk = 0; kk < TK / 16; ++kk) {
                const uint64_t bdesc = smem_desc_sw128_mn(v_addr + kk * 2048, C::HALF_TILE, 1024);
                mma_bf16_ts(tmem + C::COL_O, tmem + C::COL_P + pb * 64 + kk * 8, bdesc, idPV,
                            (jp > 0 || kk > 0) ? 1u : 0u);
              }
              mma_commit(&v_empty[st]);
              mma_commit(&pv_done[pb]);
              ++jp;
              progressed = true;
            }
          }
          if (progressed) {
            t0 = globaltimer();
          } else if (*abort_flag) {
            ok = false;
          } else if (globaltimer() - t0 > kWaitTimeoutNs) {
            flag_error(p.status, kStatusTimeout);
            *abort_flag = 1;
            ok = false;
          }
        }
        J += w.nblk;
        ++nunit;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      J = __shfl_sync(0xffffffffu, J, 0);
      nunit = __shfl_sync(0xffffffffu, nunit, 0);
    }
    if (leader && !ok) {
      mma_commit(drain);
      mbar_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    constexpr int HK = TK / 2;        // keys per thread per block
    constexpr int HD = D / 2;         // head dims per thread in O
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // 0: keys 0..63 / dims 0..D/2-1, 1: the rest
    const int r = quarter * 32 + lane;  // query row of this thread within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int stid = (warp - 2) * 32 + lane;  // 0..255 among the softmax threads
    int qs = 0, J = 0, nunit = 0;
    uint32_t qph = 0;
    while (true) {
      bool got = mbar_wait(&uq_full[qs], qph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int u = uq[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&uq_empty[qs]);
      if (++qs == 2) {
        qs = 0;
        qph ^= 1u;
      }
      const TcUnit w = tc_unit(p, pre, u);
      if (!w.valid) break;
      const int key_end = w.pos0 + w.nrows;
      const int lim = r < w.nrows ? w.pos0 + r : key_end - 1;  // last key this row sees
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < w.nblk; ++j) {
        const int b = (J + j) & 1;
        bool sok = mbar_wait(&s_full[b], ((J + j) >> 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, sok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[HK];
#pragma unroll
        for (int c = 0; c < HK / 32; ++c)
          tmem_ld_32x32b_x32(tmem + lane_base + b * TK + half * HK + c * 32,
                             *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[b]);
        // this half's row maximum of the raw scores (the scale is positive),
        // masked keys set to -inf; only a block crossing this row's last key
        // needs the mask; then the full row's maximum in base-2 units
        const int key0 = j * TK + half * HK;
        float mx = -INFINITY;
        if (key0 + HK - 1 <= lim) {
#pragma unroll
          for (int c = 0; c < HK; ++c) mx = fmaxf(mx, __uint_as_float(sv[c]));
        } else {
#pragma unroll
          for (int c = 0; c < HK; ++c) {
            const float s = key0 + c <= lim ? __uint_as_float(sv[c]) : -INFINITY;
            sv[c] = __float_as_uint(s);
            mx = fmaxf(mx, s);
          }
        }
        mx *= p.scale_log2;
        // exchange with the other half of the row (mbarrier per block parity;
        // a phase cannot run ahead: it needs every softmax warp's arrival)
        float* xm = xmax + ((J + j) & 1) * 256;
        xm[half * 128 + r] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[(J + j) & 1]);
        bool xok = mbar_wait(&xbar[(J + j) & 1], ((J + j) >> 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, xok)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, xm[(half ^ 1) * 128 + r]);
        // lazily raise the maximum; rescale O (in TMEM) and l when it moves
        const bool raise = mx > m_used + kRescale;
        const float m_new = raise ? mx : m_used;
        const float alpha = raise ? ex2_approx(m_used - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          // the previous PV block must be complete before O is touched
          const int gp = J + j - 1;
          bool pok = mbar_wait(&pv_done[gp & 1], (gp >> 1) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, pok)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t ov[32];
            const uint32_t ta = tmem + lane_base + C::COL_O + half * HD + c * 32;
            tmem_ld_32x32b_x32(ta, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st_32x32b_x32(ta, ov);
          }
          tmem_st_wait();
        }
        m_used = m_new;
        l *= alpha;
        // P = 2^(s - m) as bf16: this thread's 64 keys are row r of P half `half`
        // P = 2^(s scale - m) (one rounding for the exponent argument)
        float rs = 0.f;
        uint32_t pk[HK / 2];
        const float neg_m = -m_used;
#pragma unroll
        for (int c = 0; c < HK / 2; ++c) {
          const float a0 = ex2_approx(fmaf(__uint_as_float(sv[2 * c]), p.scale_log2, neg_m));
          const float a1 = ex2_approx(fmaf(__uint_as_float(sv[2 * c + 1]), p.scale_log2, neg_m));
          rs += a0 + a1;
          pk[c] = pack_bf16x2(a0, a1);
        }
        l += rs;
        // P of this block goes to TMEM buffer b = block & 1 once the PV that
        // read the buffer two blocks ago has completed
        const int gb = J + j, pb = gb & 1;
        if (gb >= 2) {
          bool pok = mbar_wait(&pv_done[pb], ((gb >> 1) - 1) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, pok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // row r's keys half * 64 .. + 63 -> columns half * 32 .. + 31 of P_b
        tmem_st_32x32b_x32(tmem + lane_base + C::COL_P + pb * 64 + half * 32, pk);
        if (j * TK + TK > key_end) {
          // keys past key_end may hold uninitialised memory: zero their V rows
          // once the V block has landed (its stage cannot be refilled before
          // this block's PV, which waits for p_full below)
          const int gv = J + j, stage = gv % VSTAGE;
          bool vok = mbar_wait(&v_full[stage], (gv / VSTAGE) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, vok)) {
            ok = false;
            break;
          }
          uint8_t* sv_base = sV + stage * C::KV_BYTES;
          const int first = key_end - j * TK;
          constexpr int per = C::HALVES * 8;
          for (int i = stid; i < (TK - first) * per; i += 32 * kSoftWarps) {
            const int key = first + i / per, rem = i % per, hf = rem >> 3, cc = rem & 7;
            *reinterpret_cast<uint4*>(sv_base + hf * C::HALF_TILE + key * 128 + ((cc ^ (key & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[pb]);
      }
      if (!ok) break;
      J += w.nblk;
      // epilogue: row sum of both halves; the unit's last PV block is complete -> O / l
      xsum[half * 128 + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(xsbar);
      bool xok = mbar_wait(xsbar, nunit & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, xok)) break;
      l += xsum[(half ^ 1) * 128 + r];
      bool pok = mbar_wait(&pv_done[(J - 1) & 1], ((J - 1) >> 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, pok)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + static_cast<size_t>(w.row0 + r) * p.n_q * D + w.head * D + half * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem + lane_base + C::COL_O + half * HD + c * 32, ov);
        tmem_ld_wait();
        if (r < w.nrows) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t q4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              q4[e] = pack_bf16x2(__uint_as_float(ov[8 * i + 2 * e]) * inv, __uint_as_float(ov[8 * i + 2 * e + 1]) * inv);
            dst[i] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      ++nunit;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

hb_status chunk_tc_launch(const DeviceCtx& ctx, const void* q, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const hb_device_plan& plan, const hb_layer_dims& dm, int num_pages, int max_kv_len,
                          void* out, int* work_counter, int grid, cudaStream_t stream) {
  CUtensorMap tmQ;
  hb_status st = encode_tmap_q3d(&tmQ, q, plan.n_rows, dm.n_q, dm.d_head);
  if (st != HB_OK) return st;
  TcParams p;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.q_start = plan.seq_q_start;
  p.kv_len = plan.seq_kv_len;
  p.block_table = plan.block_table;
  p.S = plan.n_seqs;
  p.T = plan.n_rows;
  p.max_pages = plan.max_pages;
  p.num_pages = num_pages;
  p.n_q = dm.n_q;
  p.n_kv = dm.n_kv;
  p.grp = dm.n_q / dm.n_kv;
  p.max_kv_len = max_kv_len;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(dm.d_head)));
  p.work_counter = work_counter;
  p.status = ctx.status;
  if (chunk_pair_eligible(dm)) return chunk_pair_launch(ctx, tmQ, tmK, tmV, p, grid, stream);
  static std::atomic<bool> attr_set[2][kMaxDevices];
  st = dm.d_head == 128
           ? smem_limit_once(attr_set[1], ctx.device, chunk_tc_kernel<128>, TC<128>::SMEM, "cudaFuncSetAttribute(chunk_tc)")
           : smem_limit_once(attr_set[0], ctx.device, chunk_tc_kernel<64>, TC<64>::SMEM, "cudaFuncSetAttribute(chunk_tc)");
  if (st != HB_OK) return st;
  if (dm.d_head == 128)
    return launch_pdl(chunk_tc_kernel<128>, grid, kThreads, TC<128>::SMEM, stream, "chunk_tc_kernel launch", tmQ, tmK,
                      tmV, p);
  return launch_pdl(chunk_tc_kernel<64>, grid, kThreads, TC<64>::SMEM, stream, "chunk_tc_kernel launch", tmQ, tmK, tmV,
                    p);
}

}  // namespace hb
