// Pieces shared by the chunk-row attention kernels (attention_tc.cu: one
// CTA per unit; attention_tc_pair.cu: CTA pairs): the work-unit shape, the
// warp roles' sizes, the kernel parameters and a few tcgen05 helpers.
#pragma once
#include <cuda_bf16.h>

#include "device.cuh"
#include "runtime.h"

namespace hb {
namespace tc {

using namespace dev;

constexpr int TQ = 128;           // query rows per unit (MMA M)
constexpr int TK = 128;           // keys per block (MMA N of S, K of PV)
constexpr int MAX_SEQS = 1024;
constexpr int kSoftWarps = 8;                // two threads per query row (column halves)
constexpr int kVWarp = 2 + kSoftWarps;        // the V producer
constexpr int kThreads = 32 * (kVWarp + 1);
constexpr float kRescale = 8.0f;  // log2 growth of a row maximum that forces an O rescale

struct TcParams {
  __nv_bfloat16* out;
  const int* q_start;
  const int* kv_len;
  const int* block_table;
  int S, T, max_pages, num_pages, n_q, n_kv, grp, max_kv_len;
  float scale_log2;
  int* work_counter;
  int* status;
};

__device__ __forceinline__ int upper_index(const int* pre, int n, int u) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// O (+)= A B^T with A (M x K bf16) read from tensor memory, B a shared-memory
// descriptor; kind::f16, fp32 accumulate.  A: lane = row, column c holds
// elements 2c (low half) and 2c + 1 of the row.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with cta_group::2 (issued by the pair's even CTA; A from each
// CTA's tensor memory at the same address, B's N columns split between the
// two CTAs' shared memory).
__device__ __forceinline__ void mma_bf16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// rows of 64 contiguous MN elements (128 B) along K, 8-row groups `sbo` bytes
// apart (K direction), 64-element MN atoms `lbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

}  // namespace tc

// Chunk-row attention on CTA pairs (attention_tc_pair.cu): d_head = 128 and
// an even number of q heads per kv head; `grid` is rounded down to an even
// number of CTAs (at least 2).
hb_status chunk_pair_launch(const DeviceCtx& ctx, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const tc::TcParams& p, int grid, cudaStream_t stream);
bool chunk_pair_eligible(const hb_layer_dims& dm);

}  // namespace hb
