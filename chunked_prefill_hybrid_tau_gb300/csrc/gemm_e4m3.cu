// Packed-token projections with E4M3 operands (kind::f8f6f4, fp32
// accumulate): the host side of hb_gemm_e4m3 and of the layer's FP8 path.
//
// FP8 doubles the FLOPs per byte of the linear layers and moves their knee
// to the right (Sarathi-Serve reading notes, section 7.7).  Operands are
// E4M3 codes with one fp32 scale per row of A (token) and of B (output
// channel); the epilogue applies sa[m] sb[n] to the fp32 accumulator and
// then runs the bf16 path's STORE / RESIDUAL / SWIGLU / F32 arithmetic.
// The kernel is the bf16 one (gemm_kernel.cuh) with 128 K elements per
// 128-byte k-block, so tiles, rings, split-K and tile-width rules are the
// same.
#include "gemm_kernel.cuh"

namespace hb {

hb_status gemm_e4m3_launch(const DeviceCtx& ctx, const void* A, int lda, const float* sa, const void* B,
                           const float* sb, void* C, int ldc, const void* R, int M, int N, int K, int epi,
                           cudaStream_t stream, const GemmNorm* norm, const GemmSplit* split, const GemmRope* rope) {
  if (split != nullptr && !gemm_split_k(N, K, epi)) split = nullptr;
  const int pbn = gemm_pair_bn(M, N, epi, split != nullptr, ctx.num_sms);
  if (epi == kEpiRope) {
    if (rope == nullptr || N % 256 != 0) {
      set_error("gemm_e4m3: the fused RoPE epilogue needs its destinations and N %% 256 == 0");
      return HB_ERR_UNSUPPORTED;
    }
    if (pbn != 0)
      return launch_pair<kPairBN, kEpiRope, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split, stream,
                                                  rope);
    if (choose_bn(M, N, epi, ctx.num_sms) == 256)
      return launch<256, kEpiRope, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split, stream, rope);
    return launch<128, kEpiRope, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split, stream, rope);
  }
  if (pbn != 0) {
    if (epi == HB_EPI_SWIGLU)
      return launch_pair<kPairBN, HB_EPI_SWIGLU, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split,
                                                      stream);
    if (epi == HB_EPI_RESIDUAL)
      return launch_pair<kPairBN, HB_EPI_RESIDUAL, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split,
                                                        stream);
    if (pbn == 192)
      return launch_pair<192, HB_EPI_STORE, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split, stream);
    return launch_pair<256, HB_EPI_STORE, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split, stream);
  }
  const int bn = split ? 256 : choose_bn(M, N, epi, ctx.num_sms);
#define HB_GEMM_CASE(BN_, EPI_) \
  if (bn == BN_ && epi == EPI_) \
    return launch<BN_, EPI_, true>(ctx, A, lda, sa, B, sb, C, ldc, R, M, N, K, norm, split, stream);
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
  set_error("hb_gemm_e4m3: no kernel for BN=%d epilogue=%d", bn, epi);
  return HB_ERR_UNSUPPORTED;
}

hb_status gemm_e4m3_check(const void* A, const float* sa, const void* B, const float* sb, void* C, const void* R,
                          int M, int N, int K, int epi) {
  HB_REQUIRE(A && sa && B && sb && C, "hb_gemm_e4m3: null operand");
  HB_REQUIRE(M >= 1 && N >= 8 && K >= 16, "hb_gemm_e4m3: bad shape M=%d N=%d K=%d", M, N, K);
  HB_REQUIRE(K % 16 == 0 && N % 8 == 0, "hb_gemm_e4m3: K %% 16 and N %% 8 required (K=%d N=%d)", K, N);
  HB_REQUIRE(epi >= HB_EPI_STORE && epi <= HB_EPI_F32, "hb_gemm_e4m3: unknown epilogue %d", epi);
  HB_REQUIRE(epi != HB_EPI_SWIGLU || N % 128 == 0, "hb_gemm_e4m3: SWIGLU needs N %% 128 == 0");
  HB_REQUIRE(epi != HB_EPI_RESIDUAL || R != nullptr, "hb_gemm_e4m3: RESIDUAL needs R");
  HB_REQUIRE(aligned16(A) && aligned16(B) && aligned16(C) && aligned16(sb) && (R == nullptr || aligned16(R)),
             "hb_gemm_e4m3: operands and sb must be 16-byte aligned");
  return HB_OK;
}

}  // namespace hb

extern "C" hb_status hb_gemm_e4m3(const void* A, const float* s_a, const void* B, const float* s_b, void* C,
                                  const void* R, int32_t M, int32_t N, int32_t K, int32_t epilogue, void* stream) {
  hb::clear_error();
  hb_status st = hb::gemm_e4m3_check(A, s_a, B, s_b, C, R, M, N, K, epilogue);
  if (st != HB_OK) return st;
  hb::DeviceCtx ctx;
  st = hb::device_context(&ctx);
  if (st != HB_OK) return st;
  const int ldc = epilogue == HB_EPI_SWIGLU ? N / 2 : N;
  return hb::gemm_e4m3_launch(ctx, A, K, s_a, B, s_b, C, ldc, R, M, N, K, epilogue,
                              static_cast<cudaStream_t>(stream));
}
