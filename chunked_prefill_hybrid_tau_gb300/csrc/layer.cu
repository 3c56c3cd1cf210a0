// One decoder layer over a packed hybrid batch, and the final norm + LM head.
//
// The forward of a hybrid iteration ("run_iteration(B)" of the scheduling
// loop, Sarathi-Serve reading notes section 3.4) for one pre-norm layer:
//   rmsnorm1 -> qkv projection -> RoPE + paged KV append -> hybrid attention
//   -> o projection + residual -> rmsnorm2 -> gate/up projection + SwiGLU
//   -> down projection + residual.
// Both RMSNorms are folded into the projections that consume them: the
// gains are folded into W_qkv and W_gu at weight preparation, a row's
// 1/rms factor scales its accumulators in the QKV and gate/up epilogues, and
// the statistics come from a row pass over x (rmsnorm1) and from the o
// projection's epilogue (rmsnorm2, no separate pass).  Every stage is one
// kernel launch on the caller's stream (attention: two, see attention.cu);
// the workspace is carved into 256-byte aligned regions.
//
// E4M3 weights (FP8 projections, reading notes section 7.7): each
// projection's input is quantized per token right before it (x together
// with its row statistics, then o, h and the SwiGLU output), and the
// projections run on the tensor cores' FP8 path with the per-row scales of
// both operands applied in the epilogue; the 1/rms factors still come from
// the bf16 rows.
#include <cuda_runtime.h>

#include "runtime.h"

namespace hb {
namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// SwiGLU width rounded up to the 64-row interleave blocks of w_gu.
inline int ffn_pad(const hb_layer_dims& dm) { return (dm.d_ff + 63) / 64 * 64; }

struct LayerWs {
  size_t ss_x, ss_h, qkv, q, o, h, a, part_o, part_d, flags, q8_x, q8_o, q8_h, q8_a, s8, attn, total;
};

LayerWs layer_ws(const hb_layer_dims& dm, int T, int S, int max_kv_len) {
  LayerWs w;
  const size_t t = static_cast<size_t>(T);
  size_t off = 0;
  w.ss_x = off; off += align256(t * (dm.d_model / 32) * 4);
  w.ss_h = off; off += align256(t * (dm.d_model / 32) * 4);
  w.qkv = off;  off += align256(t * (dm.n_q + 2 * dm.n_kv) * dm.d_head * 2);
  w.q = off;    off += align256(t * dm.n_q * dm.d_head * 2);
  w.o = off;    off += align256(t * dm.n_q * dm.d_head * 2);
  w.h = off;    off += align256(t * dm.d_model * 2);
  w.a = off;    off += align256(t * ffn_pad(dm) * 2);
  w.part_o = off; off += align256(gemm_split_part_bytes(T, dm.d_model));
  w.part_d = off; off += align256(gemm_split_part_bytes(T, dm.d_model));
  // E4M3 operands of the four projections and their per-token scales
  w.q8_x = off; off += align256(t * dm.d_model);
  w.q8_o = off; off += align256(t * dm.n_q * dm.d_head);
  w.q8_h = off; off += align256(t * dm.d_model);
  w.q8_a = off; off += align256(t * ffn_pad(dm));
  w.s8 = off;   off += 4 * align256(t * 4);
  // split-K counters right before the attention workspace, whose counters
  // come first: one kernel of the layer zeroes both in one range
  w.flags = off;  off += align256(static_cast<size_t>(2) * gemm_split_flags(T, dm.d_model) * 4);
  w.attn = off; off += align256(attention_workspace_bytes(dm, S, max_kv_len));
  w.total = off;
  return w;
}

}  // namespace
}  // namespace hb

extern "C" size_t hb_layer_workspace_bytes(const hb_layer_dims* dims, int32_t max_rows, int32_t max_seqs,
                                           int32_t max_kv_len) {
  if (!dims || max_rows < 0 || max_seqs < 0 || max_kv_len < 0) return 0;
  return hb::layer_ws(*dims, max_rows, max_seqs, max_kv_len).total;
}

extern "C" hb_status hb_layer_kernel_count(const hb_layer_dims* dims, int32_t n_rows, int32_t format,
                                           int32_t* count) {
  using namespace hb;
  clear_error();
  hb_status st = check_dims(dims);
  if (st != HB_OK) return st;
  HB_REQUIRE(count && n_rows >= 0, "hb_layer_kernel_count: bad arguments");
  HB_REQUIRE(format == HB_WEIGHTS_BF16 || format == HB_WEIGHTS_E4M3, "hb_layer_kernel_count: unknown format %d",
             format);
  // the same rules as hb_layer_forward: row statistics, QKV, RoPE/KV
  // append, chunk and decode attention, O, gate/up, down; E4M3: three more
  // quantization kernels, RoPE/KV append inside the QKV projection when
  // its tiles hold whole heads
  const int qkv_cols = (dims->n_q + 2 * dims->n_kv) * dims->d_head;
  if (n_rows == 0)
    *count = 0;
  else if (format == HB_WEIGHTS_E4M3)
    *count = gemm_rope_ok(qkv_cols, *dims) ? 10 : 11;
  else
    *count = 8;
  return HB_OK;
}

namespace hb {
namespace {

// Argument checks of one layer's weights.
hb_status check_weights(const hb_layer_weights* w, const hb_layer_dims* dims) {
  HB_REQUIRE(w, "layer forward: null weights");
  HB_REQUIRE(w->w_qkv && w->w_o && w->w_gu && w->w_d, "layer forward: null weight");
  HB_REQUIRE(w->format == HB_WEIGHTS_BF16 || w->format == HB_WEIGHTS_E4M3, "layer forward: unknown format %d",
             w->format);
  const bool f8 = w->format == HB_WEIGHTS_E4M3;
  HB_REQUIRE(!f8 || (w->s_qkv && w->s_o && w->s_gu && w->s_d), "layer forward: E4M3 weights need scales");
  HB_REQUIRE(!f8 || (aligned16(w->s_qkv) && aligned16(w->s_o) && aligned16(w->s_gu) && aligned16(w->s_d)),
             "layer forward: E4M3 scales must be 16-byte aligned");
  HB_REQUIRE(!f8 || dims->d_ff % 16 == 0, "layer forward: E4M3 weights need d_ff %% 16 == 0");
  return HB_OK;
}

// Argument checks shared by every layer of a call (dims already checked).
hb_status check_call(const hb_layer_dims* dims, const hb_device_plan* plan, const void* rope, int max_pos,
                     const void* x_in, const void* x_out, int num_pages, int max_kv_len, const void* workspace,
                     size_t ws_bytes) {
  HB_REQUIRE(plan, "layer forward: null plan");
  HB_REQUIRE(x_in && x_out && rope, "layer forward: null pointer");
  HB_REQUIRE(plan->n_rows >= 0 && plan->n_seqs >= 0, "layer forward: bad plan sizes");
  HB_REQUIRE(plan->n_rows == 0 || (plan->row_pos && plan->slot_mapping && plan->seq_q_start && plan->seq_kv_len &&
                                   plan->block_table),
             "layer forward: null plan array");
  HB_REQUIRE(num_pages > 0 && max_pos > 0 && max_kv_len > 0, "layer forward: bad sizes");
  HB_REQUIRE(aligned16(x_in) && aligned16(x_out) && aligned16(rope), "layer forward: 16-byte alignment");
  if (plan->n_rows == 0) return HB_OK;
  const size_t need = layer_ws(*dims, plan->n_rows, plan->n_seqs, max_kv_len).total;
  HB_REQUIRE(workspace && ws_bytes >= need, "layer forward: workspace of %zu bytes needed, %zu given", need, ws_bytes);
  HB_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "layer forward: workspace 256-byte alignment");
  return HB_OK;
}

// One layer (arguments checked, T > 0).  x_stats: the row statistics of
// x_in are already in the workspace (the previous layer's down projection
// wrote them), so the statistics kernel is left out; stats_next: the down
// projection also writes the statistics of x_out, for the next layer.
// Both are formed in the same order, so the results do not depend on which
// kernel produced them.
hb_status run_layer(const DeviceCtx& ctx, const hb_layer_weights* w, const hb_layer_dims* dims,
                    const hb_device_plan* plan, const void* rope, int max_pos, const void* x_in, void* x_out,
                    void* k_cache, void* v_cache, int num_pages, int max_kv_len, void* workspace, cudaStream_t s,
                    const hb_profile* prof, bool x_stats, bool stats_next) {
  hb_status st = HB_OK;
  const bool f8 = w->format == HB_WEIGHTS_E4M3;
  const int T = plan->n_rows;
  const hb_layer_dims& dm = *dims;
  const LayerWs lw = layer_ws(dm, T, plan->n_seqs, max_kv_len);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* ss_x = reinterpret_cast<float*>(ws + lw.ss_x);
  float* ss_h = reinterpret_cast<float*>(ws + lw.ss_h);
  void* qkv = ws + lw.qkv;
  void* q = ws + lw.q;
  void* o = ws + lw.o;
  void* h = ws + lw.h;
  void* a = ws + lw.a;
  void* aws = ws + lw.attn;
  const int d = dm.d_model, hd = dm.n_q * dm.d_head, qkv_cols = (dm.n_q + 2 * dm.n_kv) * dm.d_head;
  const int fp = ffn_pad(dm);

  auto mark = [&](int k) -> hb_status {
    if (!prof) return HB_OK;
    return cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(prof->events[k]), s), "cudaEventRecord");
  };
#define HB_STEP(k, call)         \
  do {                           \
    st = mark(k);                \
    if (st != HB_OK) return st;  \
    st = (call);                 \
    if (st != HB_OK) return st;  \
  } while (0)

  // RoPE and the KV append in the QKV projection's epilogue (E4M3 weights,
  // when every projection tile holds whole heads); else a separate
  // kv_append kernel.  Both give the same bits.  With bf16 weights the
  // fused path is slower at the benchmark shapes: it needs 256-wide tiles
  // (48 CTA pairs) where the plain projection runs 192-wide ones on 64
  // pairs, which costs more than the saved launch.
  const bool fuse_rope = f8 && gemm_rope_ok(qkv_cols, dm);
  GemmRope rope_qkv;
  rope_qkv.rope = static_cast<const float2*>(rope);
  rope_qkv.row_pos = plan->row_pos;
  rope_qkv.slots = plan->slot_mapping;
  rope_qkv.q_out = q;
  rope_qkv.k_cache = k_cache;
  rope_qkv.v_cache = v_cache;
  rope_qkv.n_q = dm.n_q;
  rope_qkv.n_kv = dm.n_kv;
  rope_qkv.d_head = dm.d_head;
  rope_qkv.max_pos = max_pos;
  rope_qkv.num_slots = static_cast<long long>(num_pages) * 16;
  const int qkv_epi = fuse_rope ? kEpiRope : HB_EPI_STORE;
  GemmNorm norm_x, norm_h_out, norm_h_in, norm_x_next;
  norm_x.ss_in = ss_x;
  norm_h_out.ss_out = ss_h;
  norm_h_in.ss_in = ss_h;
  norm_x_next.ss_out = ss_x;  // the next layer's input statistics (read by this layer's QKV long before)
  for (GemmNorm* nm : {&norm_x, &norm_h_out, &norm_h_in, &norm_x_next}) {
    nm->parts = d / 32;
    nm->inv_d = 1.0f / d;
    nm->eps = dm.rms_eps;
  }
  // split-K workspaces of the o and down projections: fp32 partial tiles
  // and arrival counters, and the attention counters after them: zeroed by
  // the quantization of x (E4M3) or by the RoPE/KV append (bf16), both
  // ahead of every kernel that uses them and behind every kernel of the
  // previous layer
  const int n_flags = gemm_split_flags(T, d);
  const int n_zero = static_cast<int>((lw.attn - lw.flags + attention_counter_bytes(dm, plan->n_seqs)) / 4);
  GemmSplit split_o, split_d;
  split_o.part = reinterpret_cast<float*>(ws + lw.part_o);
  split_d.part = reinterpret_cast<float*>(ws + lw.part_d);
  split_o.flags = reinterpret_cast<int*>(ws + lw.flags);
  split_d.flags = split_o.flags + n_flags;
  if (f8) {
    uint8_t* xq = ws + lw.q8_x;
    uint8_t* oq = ws + lw.q8_o;
    uint8_t* hq = ws + lw.q8_h;
    uint8_t* aq = ws + lw.q8_a;
    float* sx = reinterpret_cast<float*>(ws + lw.s8);
    float* so = sx + align256(static_cast<size_t>(T) * 4) / 4;
    float* sh = so + align256(static_cast<size_t>(T) * 4) / 4;
    float* sa = sh + align256(static_cast<size_t>(T) * 4) / 4;
    HB_STEP(0, quant_rows_launch(ctx, x_in, xq, sx, T, d, ss_x, split_o.flags, n_zero, s));
    HB_STEP(1, gemm_e4m3_launch(ctx, xq, d, sx, w->w_qkv, w->s_qkv, qkv, qkv_cols, nullptr, T, qkv_cols, d, qkv_epi,
                                s, &norm_x, nullptr, &rope_qkv));
    HB_STEP(2, fuse_rope ? HB_OK
                         : kv_append_launch(ctx, qkv, T, plan->row_pos, plan->slot_mapping, rope, max_pos, dm, q,
                                            k_cache, v_cache, num_pages, s));
    HB_STEP(3, attention_launch(ctx, q, k_cache, v_cache, num_pages, *plan, dm, max_kv_len, o, aws,
                                lw.total - lw.attn, s, true));
    HB_STEP(4, quant_rows_launch(ctx, o, oq, so, T, hd, nullptr, nullptr, 0, s));
    st = gemm_e4m3_launch(ctx, oq, hd, so, w->w_o, w->s_o, h, d, x_in, T, d, hd, HB_EPI_RESIDUAL, s, &norm_h_out,
                          &split_o);
    if (st != HB_OK) return st;
    HB_STEP(5, HB_OK);
    HB_STEP(6, quant_rows_launch(ctx, h, hq, sh, T, d, nullptr, nullptr, 0, s));
    st = gemm_e4m3_launch(ctx, hq, d, sh, w->w_gu, w->s_gu, a, fp, nullptr, T, 2 * fp, d, HB_EPI_SWIGLU, s,
                          &norm_h_in);
    if (st != HB_OK) return st;
    HB_STEP(7, quant_rows_launch(ctx, a, aq, sa, T, fp, nullptr, nullptr, 0, s));
    st = gemm_e4m3_launch(ctx, aq, fp, sa, w->w_d, w->s_d, x_out, d, h, T, d, dm.d_ff, HB_EPI_RESIDUAL, s,
                          stats_next ? &norm_x_next : nullptr, &split_d);
    if (st != HB_OK) return st;
    return mark(HB_LAYER_STAGES);
  }
  HB_STEP(0, x_stats ? HB_OK : row_sumsq_launch(ctx, x_in, ss_x, T, d, nullptr, 0, s));
  HB_STEP(1, gemm_launch(ctx, x_in, d, w->w_qkv, qkv, qkv_cols, nullptr, T, qkv_cols, d, HB_EPI_STORE, s, &norm_x));
  HB_STEP(2, kv_append_launch(ctx, qkv, T, plan->row_pos, plan->slot_mapping, rope, max_pos, dm, q, k_cache, v_cache,
                              num_pages, s, split_o.flags, n_zero));
  HB_STEP(3, attention_launch(ctx, q, k_cache, v_cache, num_pages, *plan, dm, max_kv_len, o, aws,
                              lw.total - lw.attn, s, true));
  HB_STEP(4, gemm_launch(ctx, o, hd, w->w_o, h, d, x_in, T, d, hd, HB_EPI_RESIDUAL, s, &norm_h_out, &split_o));
  HB_STEP(5, HB_OK);  // rmsnorm2: statistics came from the o projection, scaling goes to gate/up
  HB_STEP(6, gemm_launch(ctx, h, d, w->w_gu, a, fp, nullptr, T, 2 * fp, d, HB_EPI_SWIGLU, s, &norm_h_in));
  HB_STEP(7, gemm_launch(ctx, a, fp, w->w_d, x_out, d, h, T, d, dm.d_ff, HB_EPI_RESIDUAL, s,
                         stats_next ? &norm_x_next : nullptr, &split_d));
#undef HB_STEP
  return mark(HB_LAYER_STAGES);
}


}  // namespace
}  // namespace hb

extern "C" hb_status hb_layer_forward(const hb_layer_weights* w, const hb_layer_dims* dims, const hb_device_plan* plan,
                                      const void* rope, int32_t max_pos, const void* x_in, void* x_out, void* k_cache,
                                      void* v_cache, int32_t num_pages, int32_t max_kv_len, void* workspace,
                                      size_t ws_bytes, void* stream, const hb_profile* prof) {
  using namespace hb;
  clear_error();
  hb_status st = check_dims(dims);
  if (st != HB_OK) return st;
  st = check_weights(w, dims);
  if (st != HB_OK) return st;
  st = check_call(dims, plan, rope, max_pos, x_in, x_out, num_pages, max_kv_len, workspace, ws_bytes);
  if (st != HB_OK) return st;
  HB_REQUIRE(k_cache && v_cache, "hb_layer_forward: null KV cache");
  HB_REQUIRE(prof == nullptr || (prof->events && prof->n_events >= HB_LAYER_STAGES + 1),
             "hb_layer_forward: profile needs %d events", HB_LAYER_STAGES + 1);
  if (plan->n_rows == 0) return HB_OK;
  DeviceCtx ctx;
  st = device_context(&ctx);
  if (st != HB_OK) return st;
  return run_layer(ctx, w, dims, plan, rope, max_pos, x_in, x_out, k_cache, v_cache, num_pages, max_kv_len, workspace,
                   static_cast<cudaStream_t>(stream), prof, false, false);
}

extern "C" hb_status hb_layers_forward(const hb_layer_weights* w, int32_t n_layers, const hb_layer_dims* dims,
                                       const hb_device_plan* plan, const void* rope, int32_t max_pos, const void* x_in,
                                       void* x_out, void* const* k_caches, void* const* v_caches, int32_t num_pages,
                                       int32_t max_kv_len, void* workspace, size_t ws_bytes, void* stream) {
  using namespace hb;
  clear_error();
  hb_status st = check_dims(dims);
  if (st != HB_OK) return st;
  HB_REQUIRE(w && k_caches && v_caches && n_layers >= 0, "hb_layers_forward: null array or negative layer count");
  for (int l = 0; l < n_layers; ++l) {
    st = check_weights(w + l, dims);
    if (st != HB_OK) return st;
    HB_REQUIRE(k_caches[l] && v_caches[l], "hb_layers_forward: null KV cache of layer %d", l);
  }
  st = check_call(dims, plan, rope, max_pos, x_in, x_out, num_pages, max_kv_len, workspace, ws_bytes);
  if (st != HB_OK) return st;
  if (plan->n_rows == 0 || n_layers == 0) return HB_OK;
  DeviceCtx ctx;
  st = device_context(&ctx);
  if (st != HB_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int l = 0; l < n_layers; ++l) {
    // a bf16 layer takes its input statistics from the layer before it
    const bool next_bf16 = l + 1 < n_layers && w[l + 1].format == HB_WEIGHTS_BF16;
    const bool x_stats = l > 0 && w[l].format == HB_WEIGHTS_BF16;
    st = run_layer(ctx, w + l, dims, plan, rope, max_pos, l == 0 ? x_in : x_out, x_out, k_caches[l], v_caches[l],
                   num_pages, max_kv_len, workspace, s, nullptr, x_stats, next_bf16);
    if (st != HB_OK) return st;
  }
  return HB_OK;
}

extern "C" hb_status hb_final_logits(const void* x, int32_t T, const int32_t* rows, int32_t n_sel, const void* g_f,
                                     const void* w_lm, int32_t vocab, int32_t d, float eps, void* logits,
                                     void* workspace, size_t ws_bytes, void* stream) {
  using namespace hb;
  clear_error();
  HB_REQUIRE(x && rows && g_f && w_lm && logits && workspace, "hb_final_logits: null pointer");
  HB_REQUIRE(T >= 0 && n_sel >= 0 && vocab > 0 && vocab % 64 == 0 && d > 0 && d % 64 == 0,
             "hb_final_logits: vocab and d must be multiples of 64");
  HB_REQUIRE(ws_bytes >= static_cast<size_t>(n_sel) * d * 2, "hb_final_logits: workspace too small");
  HB_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "hb_final_logits: workspace 256-byte alignment");
  if (n_sel == 0) return HB_OK;
  hb_status st = gemm_check(workspace, w_lm, logits, nullptr, n_sel, vocab, d, HB_EPI_F32);
  if (st != HB_OK) return st;
  DeviceCtx ctx;
  st = device_context(&ctx);
  if (st != HB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = rmsnorm_launch(ctx, x, rows, g_f, workspace, n_sel, d, eps, T, s);
  if (st != HB_OK) return st;
  return gemm_launch(ctx, workspace, d, w_lm, logits, vocab, nullptr, n_sel, vocab, d, HB_EPI_F32, s);
}
