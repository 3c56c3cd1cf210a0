// Packed-token projections on the 5th-generation tensor cores, bf16
// operands (kind::f16, fp32 accumulate): the host side of hb_gemm, the
// tile-width and split-K rules, and the gate/up interleave of the weights.
// The kernel template is in gemm_kernel.cuh.
#include "gemm_kernel.cuh"

namespace hb {

bool gemm_split_k(int N, int K, int epi) {
  // a function of the shape alone, never of M: a row's result must not
  // depend on how many rows share the launch
  return epi == HB_EPI_RESIDUAL && N % 256 == 0 && N <= 8192 && K >= 4096;
}

size_t gemm_split_part_bytes(int M, int N) {
  const size_t tiles = static_cast<size_t>((M + BM - 1) / BM) * ((N + 255) / 256);
  return tiles * 2 * 256 * BM * 4;
}

int gemm_split_flags(int M, int N) { return ((M + BM - 1) / BM) * ((N + 255) / 256) * 4; }

bool gemm_rope_ok(int N, const hb_layer_dims& dims) {
  // every 128- or 256-column tile holds whole heads
  return N % 256 == 0 && (dims.d_head == 64 || dims.d_head == 128);
}

int gemm_pair_bn(int M, int N, int epi, bool split, int num_sms) {
  // CTA-pair tiles (256 rows) once M spans more than one 128-row tile: a
  // pair streams the same bytes per k-block as a one-CTA 128 x 128 tile for
  // twice the FLOPs, and the k-block time of both is set by the ring's round
  // trip, not by the MMAs (about 280 ns either way on GB300).  SwiGLU and the
  // split-K residual projections take 256-wide tiles; a plain store picks
  // 192 or 256 for the fewest waves of pair tiles over the SM pairs.
  if (M <= BM) return 0;
  if (epi == HB_EPI_SWIGLU || epi == kEpiRope || (epi == HB_EPI_RESIDUAL && split))
    return N % kPairBN == 0 ? kPairBN : 0;
  if (epi != HB_EPI_STORE) return 0;
  const int pm = (M + 2 * BM - 1) / (2 * BM);
  const int pairs = num_sms / 2;
  int best = 0;
  double best_cost = 1e30;
  for (int bn : {256, 192}) {
    if (N % bn != 0) continue;
    const int waves = (pm * (N / bn) + pairs - 1) / pairs;
    const double cost = waves * (bn + 32.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

hb_status gemm_launch(const DeviceCtx& ctx, const void* A, int lda, const void* B, void* C, int ldc, const void* R,
                      int M, int N, int K, int epi, cudaStream_t stream, const GemmNorm* norm, const GemmSplit* split) {
  if (split != nullptr && !gemm_split_k(N, K, epi)) split = nullptr;
  const int pbn = gemm_pair_bn(M, N, epi, split != nullptr, ctx.num_sms);
  if (pbn != 0) {
    if (epi == HB_EPI_SWIGLU)
      return launch_pair<kPairBN, HB_EPI_SWIGLU, false>(ctx, A, lda, nullptr, B, nullptr, C, ldc, R, M, N, K, norm, split,
                                                      stream);
    if (epi == HB_EPI_RESIDUAL)
      return launch_pair<kPairBN, HB_EPI_RESIDUAL, false>(ctx, A, lda, nullptr, B, nullptr, C, ldc, R, M, N, K, norm,
                                                        split, stream);
    if (pbn == 192)
      return launch_pair<192, HB_EPI_STORE, false>(ctx, A, lda, nullptr, B, nullptr, C, ldc, R, M, N, K, norm, split,
                                                   stream);
    return launch_pair<256, HB_EPI_STORE, false>(ctx, A, lda, nullptr, B, nullptr, C, ldc, R, M, N, K, norm, split,
                                                 stream);
  }
  // split-K units use the widest tile (N = 256 MMAs run near the tensor peak)
  const int bn = split ? 256 : choose_bn(M, N, epi, ctx.num_sms);
#define HB_GEMM_CASE(BN_, EPI_)                                                                                \
  if (bn == BN_ && epi == EPI_)                                                                                \
    return launch<BN_, EPI_, false>(ctx, A, lda, nullptr, B, nullptr, C, ldc, R, M, N, K, norm, split, stream);
  HB_GEMM_CASE(256, HB_EPI_STORE)
  HB_GEMM_CASE(192, HB_EPI_STORE)
  HB_GEMM_CASE(128, HB_EPI_STORE)
  HB_GEMM_CASE(256, HB_EPI_RESIDUAL)
  HB_GEMM_CASE(192, HB_EPI_RESIDUAL)
  HB_GEMM_CASE(128, HB_EPI_RESIDUAL)
  HB_GEMM_CASE(256, HB_EPI_SWIGLU)
  HB_GEMM_CASE(128, HB_EPI_SWIGLU)
  HB_GEMM_CASE(256, HB_EPI_F32)
  HB_GEMM_CASE(192, HB_EPI_F32)
  HB_GEMM_CASE(128, HB_EPI_F32)
#undef HB_GEMM_CASE
  set_error("hb_gemm: no kernel for BN=%d epilogue=%d", bn, epi);
  return HB_ERR_UNSUPPORTED;
}

hb_status gemm_check(const void* A, const void* B, void* C, const void* R, int M, int N, int K, int epi) {
  HB_REQUIRE(A && B && C, "hb_gemm: null operand");
  HB_REQUIRE(M >= 1 && N >= 8 && K >= 8, "hb_gemm: bad shape M=%d N=%d K=%d", M, N, K);
  HB_REQUIRE(K % 8 == 0 && N % 8 == 0, "hb_gemm: K and N must be multiples of 8 (K=%d N=%d)", K, N);
  HB_REQUIRE(epi >= HB_EPI_STORE && epi <= HB_EPI_F32, "hb_gemm: unknown epilogue %d", epi);
  HB_REQUIRE(epi != HB_EPI_SWIGLU || N % 128 == 0, "hb_gemm: SWIGLU needs N %% 128 == 0");
  HB_REQUIRE(epi != HB_EPI_RESIDUAL || R != nullptr, "hb_gemm: RESIDUAL needs R");
  HB_REQUIRE(aligned16(A) && aligned16(B) && aligned16(C) && (R == nullptr || aligned16(R)),
             "hb_gemm: operands must be 16-byte aligned");
  return HB_OK;
}

namespace {
// ---------------------------------------------------------------- weight prep
// w_gu row 128*b + e holds gate row 64*b + e (e < 64) or up row 64*b + e - 64;
// rows past F (when F % 64 != 0) are zero.
__global__ void interleave_gate_up_kernel(const uint4* __restrict__ wg, const uint4* __restrict__ wu,
                                          uint4* __restrict__ out, int F, int F_pad, int d8) {
  const size_t total = static_cast<size_t>(2 * F_pad) * d8;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(i / d8);
    const int c = static_cast<int>(i % d8);
    const int blk = row / 128, e = row % 128;
    const int src = blk * 64 + (e & 63);
    out[i] = src < F ? (e < 64 ? wg : wu)[static_cast<size_t>(src) * d8 + c] : make_uint4(0, 0, 0, 0);
  }
}
}  // namespace

}  // namespace hb

extern "C" hb_status hb_gemm(const void* A, const void* B, void* C, const void* R, int32_t M, int32_t N, int32_t K,
                             int32_t epilogue, void* stream) {
  hb::clear_error();
  hb_status st = hb::gemm_check(A, B, C, R, M, N, K, epilogue);
  if (st != HB_OK) return st;
  hb::DeviceCtx ctx;
  st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  const int ldc = epilogue == HB_EPI_SWIGLU ? N / 2 : N;
  return hb::gemm_launch(ctx, A, K, B, C, ldc, R, M, N, K, epilogue, static_cast<cudaStream_t>(stream));
}

extern "C" hb_status hb_interleave_gate_up(const void* w_gate, const void* w_up, void* w_gu, int32_t F, int32_t d,
                                           void* stream) {
  hb::clear_error();
  HB_REQUIRE(w_gate && w_up && w_gu, "hb_interleave_gate_up: null pointer");
  HB_REQUIRE(F > 0 && F % 8 == 0 && d > 0 && d % 8 == 0, "hb_interleave_gate_up: F %% 8 and d %% 8 required");
  HB_REQUIRE(hb::aligned16(w_gate) && hb::aligned16(w_up) && hb::aligned16(w_gu),
             "hb_interleave_gate_up: pointers must be 16-byte aligned");
  hb::DeviceCtx ctx;
  hb_status st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  hb::interleave_gate_up_kernel<<<ctx.num_sms * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(w_gate), static_cast<const uint4*>(w_up), static_cast<uint4*>(w_gu), F,
      (F + 63) / 64 * 64, d / 8);
  return hb::launch_status("interleave_gate_up_kernel launch");
}
