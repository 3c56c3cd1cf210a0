// Chunk-row attention on CTA pairs (tcgen05 cta_group::2).
//
// The same computation as chunk_tc_kernel (attention_tc.cu): a prompt
// chunk's query at position p attends to keys 0..p of its request
// (Sarathi-Serve reading notes, sections 3.1 and 7.5b).  Here a cluster of
// two CTAs on neighbouring SMs takes two q heads of one kv head for the same
// 128 query rows, so both need the same K and V blocks:
//   * S = Q K^T is one M = 256, N = 128 pair MMA: each CTA holds its head's
//     Q tile and 64 of the block's 128 keys (the even CTA keys 0..63);
//   * O += P V is one M = 256, N = 128 pair MMA with P read from each CTA's
//     tensor memory and V's head dimensions split between the CTAs (the even
//     CTA dims 0..63), each holding all 128 keys of its half;
// so each SM streams 32 KB of K and V per 128-key block instead of 64 KB,
// which is what bounds the one-CTA kernel.  Each CTA runs its own softmax
// over its own rows; the even CTA's MMA thread issues every MMA once both
// CTAs' inputs are ready.
//
// Hand-offs between the two CTAs (every wait bounded):
//   * K and Q boxes of both CTAs complete on the even CTA's k_full / q_full;
//     V boxes complete on each CTA's own v_full, and each CTA's softmax waits
//     for its V block before it declares P ready, so p_full (arrivals from
//     both CTAs' softmax warps, count 16) also means both V halves landed;
//   * s_empty, p_full and o_empty (count 16) live in the even CTA; the MMA
//     commits (stage releases, S ready, PV done, Q consumed) are multicast to
//     both CTAs.
// Units are assigned statically (unit v to cluster v mod clusters), heaviest
// tiles first.  d_head = 128 only; with an odd number of q heads per kv head
// the one-CTA kernel runs instead.
#include <cuda_bf16.h>

#include "attention_tc.cuh"

namespace hb {
namespace {

using namespace dev;
using namespace tc;

constexpr int D = 128;
constexpr int KSTAGE = 4;
constexpr int VSTAGE = 4;

struct PC {
  static constexpr int HALF_TILE = 128 * 128;       // 128 rows x 128 bytes
  static constexpr int Q_BYTES = 2 * HALF_TILE;     // this CTA's Q tile (two 64-dim halves)
  static constexpr int KH = 64 * 128;               // one 64-dim half of this CTA's 64 keys
  static constexpr int K_BYTES = 2 * KH;            // this CTA's 64 keys x 128 dims
  static constexpr int V_BYTES = 128 * 128;         // this CTA's 64 dims x 128 keys
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGE * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + VSTAGE * V_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int OFF_XCH = OFF_BAR + BAR_BYTES;
  static constexpr int XCH_BYTES = (2 * 2 * 128 + 2 * 128) * 4;
  static constexpr int OFF_PRE = OFF_XCH + XCH_BYTES;
  static constexpr int SMEM = OFF_PRE + (MAX_SEQS + 1) * 4 + 1024;
  static_assert(SMEM <= 232448, "shared memory");
  static constexpr uint32_t TMEM_COLS = 512;  // S0 | S1 | O | P0 | P1 (allocated by the pair)
  static constexpr uint32_t COL_O = 256;
  static constexpr uint32_t COL_P = 384;
};

struct PairTcUnit {
  int seq, head, row0, nrows, pos0, nblk, valid;
};

// Pair unit v: sequence, 128-row tile (heaviest first) and head pair; this
// CTA's head is 2 * pair + rank.
__device__ __forceinline__ PairTcUnit pair_tc_unit(const TcParams& p, const int* pre, int v, int rank) {
  PairTcUnit w;
  w.valid = v < pre[p.S];
  if (!w.valid) return w;
  const int s = upper_index(pre, p.S, v);
  const int local = v - pre[s];
  const int pairs = p.n_q / 2;
  const int q0 = p.q_start[s], qlen = p.q_start[s + 1] - q0;
  const int ntiles = (qlen + TQ - 1) / TQ;
  const int t = ntiles - 1 - local / pairs;
  w.seq = s;
  w.head = 2 * (local % pairs) + rank;
  w.row0 = q0 + t * TQ;
  w.nrows = min(TQ, qlen - t * TQ);
  w.pos0 = p.kv_len[s] - qlen + t * TQ;
  w.nblk = (w.pos0 + w.nrows + TK - 1) / TK;
  return w;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    chunk_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, TcParams p) {
  using C = PC;
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
  uint64_t* k_full = bar;              // [KSTAGE] even CTA: both CTAs' K boxes
  uint64_t* k_empty = bar + 4;         // [KSTAGE] multicast
  uint64_t* v_full = bar + 8;          // [VSTAGE] this CTA's V boxes
  uint64_t* v_empty = bar + 12;        // [VSTAGE] multicast
  uint64_t* q_full = bar + 16;         // even CTA: both CTAs' Q tiles
  uint64_t* q_empty = bar + 17;        // multicast
  uint64_t* s_full = bar + 18;         // [2] multicast
  uint64_t* s_empty = bar + 20;        // [2] even CTA, 16 softmax warps
  uint64_t* o_empty = bar + 22;        // even CTA, 16 softmax warps
  uint64_t* drain = bar + 23;
  uint64_t* xbar = bar + 24;           // [2] local: row maxima exchanged
  uint64_t* xsbar = bar + 26;          // local: row sums exchanged
  uint64_t* p_full = bar + 27;         // [2] even CTA, 16 softmax warps
  uint64_t* pv_done = bar + 29;        // [2] multicast
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 31);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xmax = reinterpret_cast<float*>(smem + C::OFF_XCH);
  float* xsum = xmax + 2 * 2 * 128;
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int n_clusters = static_cast<int>(gridDim.x >> 1);

  // ---- per-sequence pair-unit counts (chunk sequences: more than one row)
  for (int s = tid; s < p.S; s += kThreads) {
    const int q0 = p.q_start[s], q1 = p.q_start[s + 1];
    const int qlen = q1 - q0, kvl = p.kv_len[s];
    int c = 0;
    if (q0 < 0 || q1 > p.T || qlen < 0 || kvl < qlen || kvl > p.max_kv_len || (kvl + 15) / 16 > p.max_pages)
      flag_error(p.status, kStatusIndex);
    else if (qlen > 1)
      c = (p.n_q / 2) * ((qlen + TQ - 1) / TQ);
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
      mbar_init(&s_empty[i], 2 * kSoftWarps);
      mbar_init(&p_full[i], 2 * kSoftWarps);
      mbar_init(&pv_done[i], 1);
      mbar_init(&xbar[i], kSoftWarps);
    }
    mbar_init(o_empty, 2 * kSoftWarps);
    mbar_init(xsbar, kSoftWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    pre[0] = 0;
    for (int s = 1; s <= p.S; ++s) pre[s] += pre[s - 1];
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anything arrives on them
  const uint32_t tmem = *tmem_slot;
  const int units = pre[p.S];

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    // warp 0: Q and this CTA's 64 keys of each K block (lanes 0..7: page
    // 4 rank + lane / 2, dim half lane % 2); warp kVWarp: this CTA's 64 dims
    // of each V block (lanes 0..7: page lane).
    const bool kside = warp == 0;
    if (lane == 0) {
      if (kside) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
      } else {
        tma_prefetch_desc(&tmV);
      }
    }
    const int nst = kside ? KSTAGE : VSTAGE;
    uint64_t* empty = kside ? k_empty : v_empty;
    int stage = 0, nunit = 0;
    uint32_t kph = 0;
    uint32_t pending = 0, armed = 0;
    bool ok = true;
    const int my_pg = kside ? 4 * rank + (lane >> 1) : lane;  // page of the block this lane loads
    const int my_hf = kside ? (lane & 1) : rank;              // 64-dim half
    for (int v = cluster; v < units && ok; v += n_clusters) {
      const PairTcUnit w = pair_tc_unit(p, pre, v, rank);
      if (kside && lane == 0) {
        // Q tile (the last S block of the previous unit has read both CTAs' tiles)
        ok = mbar_wait(q_empty, (nunit & 1) ^ 1u, abort_flag, p.status);
        if (ok) {
          if (leader) mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
          const uint32_t qb = cluster_addr(q_full, 0);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) tma_load_3d_pair(sQ + hf * C::HALF_TILE, &tmQ, qb, hf * 64, w.head, w.row0);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      ++nunit;
      const int g = w.head / p.grp;
      const int* bt = p.block_table + static_cast<size_t>(w.seq) * p.max_pages;
      const int key_end = w.pos0 + w.nrows;
      // this lane's raw page id of block j (0 past the last block or page),
      // loaded four blocks ahead and checked at use
      auto load_page = [&](int j) {
        const int npg = j < w.nblk ? min(8, (key_end - j * TK + 15) / 16) : 0;
        return lane < 8 && my_pg < npg ? __ldg(bt + j * 8 + my_pg) : 0;
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
            if (kside) {
              if (leader) mbar_arrive_expect_tx(&k_full[stage], npg * 4096);  // both CTAs: 2 KB per page half
            } else {
              mbar_arrive_expect_tx(&v_full[stage], npg * 2048);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, eok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane < 8 && my_pg < npg) {
          const int y = (cur * p.n_kv + g) * 16;
          if (kside) {
            uint8_t* dst = sK + stage * C::K_BYTES + my_hf * C::KH + (lane >> 1) * 2048;
            tma_load_2d_pair(dst, &tmK, cluster_addr(&k_full[stage], 0), my_hf * 64, y);
          } else {
            tma_load_2d(sV + stage * C::V_BYTES + lane * 2048, &tmV, &v_full[stage], my_hf * 64, y);
          }
        }
        if (++stage == nst) {
          stage = 0;
          kph ^= 1u;
        }
      }
    }
    if (lane == 0 && *abort_flag) raise_peer_abort(abort_flag, static_cast<uint32_t>(rank));
    if (!ok && lane == 0)
      for (int s = 0; s < nst; ++s)
        if (pending & (1u << s)) mbar_drain(&empty[s], (armed >> s) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(2 * TQ, TK);
      constexpr uint32_t idPV = idesc_bf16_f32(2 * TQ, D) | (1u << 16);  // B (V) is MN-major
      int J = 0, nunit = 0;
      bool ok = true;
      for (int v = cluster; v < units && ok; v += n_clusters) {
        const PairTcUnit w = pair_tc_unit(p, pre, v, rank);
        ok = mbar_wait_cluster(q_full, nunit & 1, abort_flag, p.status);
        const uint32_t q_addr = smem_u32(sQ);
        int js = 0, jp = 0;
        bool o_free = false;
        uint64_t t0 = globaltimer();
        while (ok && jp < w.nblk) {
          bool progressed = false;
          if (js < w.nblk) {
            const int gk = J + js, b = gk & 1, st = gk % KSTAGE;
            if (mbar_test_cluster(&k_full[st], (gk / KSTAGE) & 1) &&
                mbar_test_cluster(&s_empty[b], ((gk >> 1) & 1) ^ 1u)) {
              tc_fence_after();
              const uint32_t k_addr = smem_u32(sK + st * C::K_BYTES);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16_pair(tmem + b * TK, smem_desc_sw128(q_addr + (kk >> 2) * C::HALF_TILE + (kk & 3) * 32),
                              smem_desc_sw128(k_addr + (kk >> 2) * C::KH + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
              mma_commit_pair(&s_full[b], 3);
              mma_commit_pair(&k_empty[st], 3);
              if (js == w.nblk - 1) mma_commit_pair(q_empty, 3);
              ++js;
              progressed = true;
            }
          }
          if (jp < js) {
            const int gv = J + jp, st = gv % VSTAGE;
            if (!o_free) o_free = mbar_test_cluster(o_empty, (nunit & 1) ^ 1u);
            const int pb = gv & 1;
            // p_full: both CTAs stored P and saw their V half of this block land
            if (o_free && mbar_test_cluster(&p_full[pb], (gv >> 1) & 1)) {
              tc_fence_after();
              const uint32_t v_addr = smem_u32(sV + st * C::V_BYTES);
#pragma unroll
              for (int kk = 0; kk < TK / 16; ++kk)
                mma_bf16_ts_pair(tmem + C::COL_O, tmem + C::COL_P + pb * 64 + kk * 8,
                                 smem_desc_sw128_mn(v_addr + kk * 2048, C::HALF_TILE, 1024), idPV,
                                 (jp > 0 || kk > 0) ? 1u : 0u);
              mma_commit_pair(&v_empty[st], 3);
              mma_commit_pair(&pv_done[pb], 3);
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
      if (*abort_flag) raise_peer_abort(abort_flag, static_cast<uint32_t>(rank));
      // no pair MMA may still read either CTA's shared memory or write its
      // tensor memory when the CTAs leave
      mma_commit_pair(drain, 1);
      mbar_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue (both CTAs)
    constexpr int HK = TK / 2;
    constexpr int HD = D / 2;
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int stid = (warp - 2) * 32 + lane;
    int J = 0, nunit = 0;
    for (int v = cluster; v < units; v += n_clusters) {
      const PairTcUnit w = pair_tc_unit(p, pre, v, rank);
      const int key_end = w.pos0 + w.nrows;
      const int lim = r < w.nrows ? w.pos0 + r : key_end - 1;
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
        if (lane == 0) mbar_arrive_cluster_relaxed(cluster_addr(&s_empty[b], 0));  // S was read into registers
        // row maximum of the raw scores (the scale is positive), masked keys
        // set to -inf; only a block crossing this row's last key needs the mask
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
        const bool raise = mx > m_used + kRescale;
        const float m_new = raise ? mx : m_used;
        const float alpha = raise ? ex2_approx(m_used - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
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
        const int gb = J + j, pb = gb & 1;
        if (gb >= 2) {
          bool pok = mbar_wait(&pv_done[pb], ((gb >> 1) - 1) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, pok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st_32x32b_x32(tmem + lane_base + C::COL_P + pb * 64 + half * 32, pk);
        // this CTA's V half of the block has landed (the pair MMA reads it once
        // p_full completes); keys past key_end may hold uninitialised memory:
        // zero their rows (the stage cannot be refilled before this block's PV)
        const int gv = J + j, stage = gv % VSTAGE;
        bool vok = mbar_wait(&v_full[stage], (gv / VSTAGE) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, vok)) {
          ok = false;
          break;
        }
        if (j * TK + TK > key_end) {
          uint8_t* sv_base = sV + stage * C::V_BYTES;
          const int first = key_end - j * TK;
          for (int i = stid; i < (TK - first) * 8; i += 32 * kSoftWarps) {
            const int key = first + i / 8, cc = i % 8;
            *reinterpret_cast<uint4*>(sv_base + key * 128 + ((cc ^ (key & 7)) << 4)) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        // P is in tensor memory (tcgen05.wait::st above); zeroed V rows are
        // shared-memory stores the pair MMA must see: release only then
        if (lane == 0) {
          if (j * TK + TK > key_end)
            mbar_arrive_cluster(cluster_addr(&p_full[pb], 0));
          else
            mbar_arrive_cluster_relaxed(cluster_addr(&p_full[pb], 0));
        }
      }
      if (!ok) break;
      J += w.nblk;
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
      if (lane == 0) mbar_arrive_cluster_relaxed(cluster_addr(o_empty, 0));  // O was read into registers
      ++nunit;
    }
    if (lane == 0 && *abort_flag) raise_peer_abort(abort_flag, static_cast<uint32_t>(rank));
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

}  // namespace

bool chunk_pair_eligible(const hb_layer_dims& dm) { return dm.d_head == 128 && (dm.n_q / dm.n_kv) % 2 == 0; }

hb_status chunk_pair_launch(const DeviceCtx& ctx, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const TcParams& p, int grid, cudaStream_t stream) {
  static std::atomic<bool> attr_set[kMaxDevices];
  hb_status st = smem_limit_once(attr_set, ctx.device, chunk_pair_kernel, PC::SMEM, "cudaFuncSetAttribute(chunk_pair)");
  if (st != HB_OK) return st;
  grid &= ~1;
  if (grid < 2) grid = 2;
  return launch_pdl(chunk_pair_kernel, grid, kThreads, PC::SMEM, stream, "chunk_pair_kernel launch", tmQ, tmK, tmV, p);
}

}  // namespace hb
