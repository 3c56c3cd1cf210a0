/*
 * hb.h - C ABI of the hybrid-iteration forward (chunked prefill + decodes
 * under a token budget tau) for NVIDIA GB300 (sm_103a).
 *
 * One hybrid iteration packs every active decode (one token each) with
 * prompt chunks until the token count reaches the budget tau, then runs one
 * decoder-layer forward over the packed rows against a 16-token paged KV
 * cache (Sarathi-Serve reading notes, section 3.1 "chunked prefills",
 * 3.2 "stall-free hybrid batching", 3.4 "the scheduling algorithm";
 * "Chunked Prefill" knowledge page, mechanism section: chunks keep
 * appending to paged KV).
 *
 * Conventions for every call:
 *   - The caller owns every buffer.  No call allocates device memory; device
 *     scratch is a caller-provided workspace whose size a *_workspace_bytes
 *     call reports.
 *   - "device" pointers are CUDA device memory of the current device;
 *     "host" pointers are ordinary host memory.  bf16 is IEEE bfloat16
 *     stored as 16-bit words.  All matrices are row-major.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Their return value covers
 *     argument checks and launch errors only.  Errors detected inside a kernel
 *     (a bounded wait that expired, an index out of range) set a device
 *     status word that hb_check_status() reads.
 *   - On any status other than HB_OK, hb_last_error() returns a message for
 *     the calling thread.
 */
#ifndef HB_H_
#define HB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hb_status {
  HB_OK = 0,
  HB_ERR_INVALID_ARG = 1,   /* a null pointer, a negative size, a shape the kernels do not support */
  HB_ERR_CAPACITY = 2,      /* a caller-sized output is too small; required sizes are reported */
  HB_ERR_OUT_OF_PAGES = 3,  /* the free-page pool cannot hold the iteration's new tokens */
  HB_ERR_CUDA = 4,          /* a CUDA runtime call or a kernel launch failed */
  HB_ERR_TIMEOUT = 5,       /* a bounded device-side wait expired (reported by hb_check_status) */
  HB_ERR_UNSUPPORTED = 6,   /* the device is not sm_103 / a feature is missing */
  HB_ERR_DEVICE = 7         /* a device-side index check failed (reported by hb_check_status) */
} hb_status;

/* Text of a status code (static storage). */
const char* hb_status_string(int status);
/* Message of the last failing call on this thread ("" if none). */
const char* hb_last_error(void);
/* Library version as 10000*major + 100*minor + patch. */
int32_t hb_version(void);

/* ------------------------------------------------------------------------
 * Shapes of one decoder layer (Llama/Mistral pre-norm block: RMSNorm, GQA
 * attention with rotate-half RoPE, SwiGLU MLP; the pages name the models but
 * not their layer arithmetic).
 * ---------------------------------------------------------------------- */
typedef struct hb_layer_dims {
  int32_t d_model;     /* hidden size d (multiple of 64) */
  int32_t n_q;         /* query heads */
  int32_t n_kv;        /* key/value heads; n_q % n_kv == 0 (GQA: q head h reads kv head h / (n_q / n_kv)) */
  int32_t d_head;      /* head dimension; 64 or 128 */
  int32_t d_ff;        /* SwiGLU inner size (multiple of 8) */
  int32_t page_size;   /* tokens per KV page; must be 16 */
  float rms_eps;       /* RMSNorm epsilon, inside the square root */
  float rope_theta;    /* RoPE base, used by hb_rope_table */
} hb_layer_dims;

/* ------------------------------------------------------------------------
 * hb_plan_batch - token-budget packing of one hybrid iteration (host).
 *
 * Follows the scheduling loop of the Sarathi-Serve reading notes (section
 * 3.4) and stall-free batching (section 3.2): all decodes first (one token
 * each, in the order given), then, while fewer than tau tokens are packed,
 * walk the prefill FIFO in order and take
 *     take = min(prompt_len - done, chunk, tau - n)
 * tokens from each request (at most one chunk per request per iteration; a
 * partial chunk only where the budget ends).  If there are more decodes than
 * tau, all decodes are admitted, no prefill is added and over_budget = 1.
 *
 * Paged KV (PagedAttention pages of `page_size` tokens): a row at position p
 * of a request needs page index p / page_size of that request's page list;
 * missing pages are popped from the FRONT of the free pool, decode rows
 * first, then chunk rows in position order.  slot = page_id*page_size +
 * p % page_size.
 *
 * Inputs/outputs (all host memory, caller-owned):
 *   decodes[n_dec], prefills[n_pf]: request state.  On HB_OK each request's
 *     pages[]/n_pages gains the pages allocated for it; `done` is NOT
 *     advanced (the KV of the new rows exists only after the forward runs).
 *   pool: FIFO free list; on HB_OK pool->head advances by plan->pages_used.
 *   plan: caller-sized output arrays (capacities row_cap, seq_cap, pf_cap,
 *     max_pages) and scalar results.
 * Rows are ordered: decode rows (one sequence each), then each prefill
 * chunk's rows in position order (one sequence per chunk).
 *
 * Errors: HB_ERR_INVALID_ARG (null pointers, tau/chunk/page_size < 1,
 * done > prompt_len, a negative page id in a request); HB_ERR_CAPACITY (an
 * output array or a request's page_cap is too small: need_* fields report
 * the sizes); HB_ERR_OUT_OF_PAGES (need_pages reports how many).  On any
 * error nothing is modified except the plan's result fields.
 * ---------------------------------------------------------------------- */
typedef struct hb_request {
  int32_t prompt_len;  /* prompt length (prefills); ignored for decodes */
  int32_t done;        /* tokens already in the KV cache (decode: context length) */
  int32_t n_pages;     /* pages held (in/out) */
  int32_t page_cap;    /* capacity of pages[] */
  int32_t* pages;      /* page ids held, in position order (in/out) */
} hb_request;

typedef struct hb_page_pool {
  const int32_t* pages; /* free page ids, FIFO order */
  int32_t count;        /* entries in pages[] */
  int32_t head;         /* index of the next page to pop (in/out) */
} hb_page_pool;

typedef struct hb_plan {
  /* caller-owned output arrays and their capacities */
  int32_t row_cap;
  int32_t* row_seq;       /* [row_cap] sequence index of each row */
  int32_t* row_pos;       /* [row_cap] absolute position of each row */
  int32_t* slot_mapping;  /* [row_cap] KV slot of each row */
  int32_t seq_cap;
  int32_t* seq_q_start;   /* [seq_cap + 1] first row of each sequence (CSR) */
  int32_t* seq_pos0;      /* [seq_cap] position of the sequence's first row */
  int32_t* seq_kv_len;    /* [seq_cap] keys visible to its last row (= pos0 + rows) */
  int32_t* seq_kind;      /* [seq_cap] 0 = decode, 1 = prefill chunk */
  int32_t* seq_req;       /* [seq_cap] index into decodes[] or prefills[] */
  int32_t max_pages;      /* row stride of block_table */
  int32_t* block_table;   /* [seq_cap][max_pages] page ids, -1 padded */
  int32_t pf_cap;
  int32_t* pf_take;       /* [pf_cap] tokens taken from each prefill (0 if none) */
  int32_t* pf_finished;   /* [pf_cap] 1 if the take completes the prompt */
  /* results */
  int32_t n_rows;         /* packed tokens T */
  int32_t n_seqs;
  int32_t n_decode_seqs;
  int32_t pages_used;     /* pages popped from the pool */
  int32_t over_budget;    /* 1 if n_dec > tau */
  int32_t need_rows, need_seqs, need_max_pages, need_pages; /* sizes required (always written) */
  /* scheduling hints for the attention launch: query-key pairs the
   * iteration's attention visits (a row at position p sees p + 1 keys),
   * split by path -- sequences of one row (the HBM-bound path: every decode,
   * and a one-token chunk) and sequences of several rows (the tensor-core
   * path: prompt chunks).  Their sum is the method's attention cost.
   * chunk_rows: rows of the several-row sequences. */
  int64_t decode_pairs;
  int64_t chunk_pairs;
  int64_t chunk_rows;
} hb_plan;

hb_status hb_plan_batch(hb_request* decodes, int32_t n_dec, hb_request* prefills, int32_t n_pf,
                        hb_page_pool* pool, int32_t tau, int32_t chunk, int32_t page_size,
                        hb_plan* plan);

/* ------------------------------------------------------------------------
 * hb_sched - the iteration driver: the scheduling loop of the Sarathi-Serve
 * reading notes (section 3.4) around hb_plan_batch.  Host only, opaque
 * state, not thread-safe.
 *   hb_sched_create : budget tau, chunk size, page size and the free page
 *                     ids (FIFO) the scheduler owns from then on.
 *   hb_sched_add    : a request of prompt_len tokens that generates max_new
 *                     tokens; queued behind the other waiting prompts.
 *                     Refused between hb_sched_plan and hb_sched_commit.
 *   hb_sched_plan   : packs the next iteration into `plan` exactly as
 *                     hb_plan_batch does (all running decodes in the order
 *                     their prompts completed, then one chunk per waiting
 *                     prompt in FIFO order under tau), and writes the request
 *                     id of every row to row_req[row_cap] (may be NULL).
 *                     plan->n_rows == 0 when nothing is active.  Errors as
 *                     hb_plan_batch (CAPACITY reports sizes; OUT_OF_PAGES:
 *                     there is no preemption); on error the state is
 *                     unchanged.
 *   hb_sched_commit : after the iteration's forward: each decode has one
 *                     more cached token and one more new token; each chunk
 *                     advanced its prompt; a completed prompt has produced
 *                     its first new token and starts decoding; a request
 *                     with max_new tokens is finished and its pages go to
 *                     the back of the free pool in page order.
 *   hb_sched_info   : state (0 prefilling, 1 decoding, 2 finished), cached
 *                     tokens, new tokens so far and pages held (any output
 *                     may be NULL).
 *   hb_sched_active : requests not finished.  hb_sched_free_pages: pool size.
 * A request holds at most ceil((prompt_len + max_new - 1) / page_size) pages.
 * ---------------------------------------------------------------------- */
typedef struct hb_sched hb_sched;
hb_status hb_sched_create(int32_t tau, int32_t chunk, int32_t page_size, const int32_t* pages, int32_t n_pages,
                          hb_sched** out);
void hb_sched_destroy(hb_sched* s);
hb_status hb_sched_add(hb_sched* s, int32_t prompt_len, int32_t max_new, int32_t* id);
hb_status hb_sched_plan(hb_sched* s, hb_plan* plan, int32_t* row_req);
hb_status hb_sched_commit(hb_sched* s);
hb_status hb_sched_info(const hb_sched* s, int32_t id, int32_t* state, int32_t* cached, int32_t* generated,
                        int32_t* n_pages);
int32_t hb_sched_active(const hb_sched* s);
int32_t hb_sched_free_pages(const hb_sched* s);

/* ------------------------------------------------------------------------
 * Device view of a plan (device pointers; copies of the hb_plan arrays).
 * ---------------------------------------------------------------------- */
typedef struct hb_device_plan {
  int32_t n_rows;              /* T */
  int32_t n_seqs;              /* S */
  int32_t max_pages;           /* row stride of block_table */
  const int32_t* row_pos;      /* [T] */
  const int32_t* slot_mapping; /* [T] */
  const int32_t* seq_q_start;  /* [S + 1] */
  const int32_t* seq_kv_len;   /* [S] */
  const int32_t* block_table;  /* [S][max_pages] */
  /* hb_plan's scheduling hints (host values).  hb_attention splits the SMs
   * between chunk and decode rows by their estimated cost; with zeros
   * (unknown) the two paths run one after the other on all SMs.  Results
   * never depend on them. */
  int64_t decode_pairs;
  int64_t chunk_pairs;
  int64_t chunk_rows;
} hb_device_plan;

/* ------------------------------------------------------------------------
 * hb_rope_table - fill the rotary table (device, one-off set-up).
 * table[p][i] = (cos(p * theta^(-2i/d_head)), sin(...)) for p < max_pos,
 * i < d_head/2, computed in double precision and rounded to float.
 * table: device float2 [max_pos][d_head/2], caller-owned.
 * ---------------------------------------------------------------------- */
hb_status hb_rope_table(void* table, int32_t max_pos, int32_t d_head, double theta, void* stream);

/* ------------------------------------------------------------------------
 * hb_rmsnorm - y[r] = x[r] / sqrt(mean(x[r]^2) + eps) * gamma, fp32 math.
 * x, y: device bf16 [rows][d]; gamma: device bf16 [d]; d % 8 == 0.
 * y may not alias x.
 * ---------------------------------------------------------------------- */
hb_status hb_rmsnorm(const void* x, const void* gamma, void* y, int32_t rows, int32_t d, float eps,
                     void* stream);

/* ------------------------------------------------------------------------
 * hb_kv_append - fused RoPE + paged KV write (the chunk "writes its KV",
 * Sarathi-Serve reading notes section 3.1; chunks continue writing paged
 * KV, Chunked Prefill page, mechanism section).
 *   qkv     : device bf16 [T][(n_q + 2 n_kv) d_head]: q heads, k heads, v heads
 *   row_pos : device int32 [T]; slot_mapping: device int32 [T]
 *   rope    : device float2 [max_pos][d_head/2] from hb_rope_table; row_pos < max_pos
 *   q_out   : device bf16 [T][n_q][d_head], rotated q
 *   k_cache, v_cache: device bf16 [num_pages][n_kv][page_size][d_head];
 *     rotated k and raw v of row r are written at slot_mapping[r].
 * Rows with slot < 0 are skipped (padding).  A slot >= num_pages*page_size
 * or a position >= max_pos sets HB_ERR_DEVICE and skips the row.
 * ---------------------------------------------------------------------- */
hb_status hb_kv_append(const void* qkv, int32_t T, const int32_t* row_pos, const int32_t* slot_mapping,
                       const void* rope, int32_t max_pos, const hb_layer_dims* dims, void* q_out,
                       void* k_cache, void* v_cache, int32_t num_pages, void* stream);

/* ------------------------------------------------------------------------
 * hb_attention - varlen paged hybrid attention.  Row r of sequence s at
 * position p attends to keys 0..p of s, read through its block table: a
 * chunk row sees the request's cached prefix plus the causal part of its own
 * chunk; a decode row sees its whole context (Sarathi-Serve reading notes,
 * section 3.1 and 7.5b).  Softmax scale 1/sqrt(d_head), fp32 online softmax.
 *   q      : device bf16 [T][n_q][d_head] (rotated)
 *   caches : as in hb_kv_append (after the append of this iteration)
 *   plan   : device plan (row_pos, seq_q_start, seq_kv_len, block_table)
 *   out    : device bf16 [T][n_q * d_head]
 *   workspace: device scratch of hb_attention_workspace_bytes(...) bytes,
 *     256-byte aligned; contents need not be initialised.
 * Requires d_head == 64 or 128 and page_size == 16.
 * ---------------------------------------------------------------------- */
size_t hb_attention_workspace_bytes(const hb_layer_dims* dims, int32_t max_rows, int32_t max_seqs,
                                    int32_t max_kv_len);
hb_status hb_attention(const void* q, const void* k_cache, const void* v_cache, int32_t num_pages,
                       const hb_device_plan* plan, const hb_layer_dims* dims, int32_t max_kv_len,
                       void* out, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * hb_attention_noalloc - hb_attention for callers that cannot allocate
 * device memory (no counterpart on the pages: an interface addition).
 *
 * Some callers cannot pass a workspace: a plug-in running inside another
 * engine's execution step, where that engine owns every device allocation
 * and cudaMalloc is not allowed (it can also synchronise the device), or a
 * host runtime with no spare device buffer.  This call takes only the inputs
 * and the output (same meaning and layout as hb_attention) and uses a fixed
 * 32 MiB scratch array that the library places in device memory of every GPU
 * that loads it, held until the process exits.  It allocates nothing.
 *   - Its first call on a device looks up that array's device address (once
 *     per device, with the device current); make that first call before any
 *     stream capture.
 *   - Plans needing more scratch than 32 MiB (hb_attention_workspace_bytes
 *     of n_seqs and max_kv_len above 32 MiB) are rejected with
 *     HB_ERR_CAPACITY and a message; use hb_attention with a workspace then.
 *   - Every call on a device shares the one array; the counters that must
 *     start at zero are cleared by each call on `stream`.  Calls that can
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on the array and give wrong results: order them.
 * ---------------------------------------------------------------------- */
hb_status hb_attention_noalloc(const void* q, const void* k_cache, const void* v_cache, int32_t num_pages,
                               const hb_device_plan* plan, const hb_layer_dims* dims, int32_t max_kv_len,
                               void* out, void* stream);

/* ------------------------------------------------------------------------
 * hb_gemm - C = epilogue(A B^T) on the tensor cores (bf16 in, fp32
 * accumulate): the packed-token projections whose roofline the pages use
 * (Sarathi-Serve reading notes, section 1.6: T = max(T_math, T_mem)).
 *   A: device bf16 [M][K]; B: device bf16 [N][K] (weights, row-major)
 *   HB_EPI_STORE   : C bf16 [M][N] = AB^T
 *   HB_EPI_RESIDUAL: C bf16 [M][N] = R + AB^T  (R bf16 [M][N], may alias C)
 *   HB_EPI_SWIGLU  : B holds gate/up rows interleaved in blocks of 64
 *                    (hb_interleave_gate_up); C bf16 [M][N/2] =
 *                    silu(A Bg^T) * (A Bu^T)
 *   HB_EPI_F32     : C fp32 [M][N] = AB^T
 * Requires K % 8 == 0 and N % 8 == 0 (N % 128 for SWIGLU), 16-byte aligned
 * pointers.
 * ---------------------------------------------------------------------- */
typedef enum hb_epilogue {
  HB_EPI_STORE = 0,
  HB_EPI_RESIDUAL = 1,
  HB_EPI_SWIGLU = 2,
  HB_EPI_F32 = 3
} hb_epilogue;

hb_status hb_gemm(const void* A, const void* B, void* C, const void* R, int32_t M, int32_t N, int32_t K,
                  int32_t epilogue, void* stream);

/* ------------------------------------------------------------------------
 * hb_quantize_e4m3 - per-row FP8 quantization, the operand preparation of
 * the E4M3 projections (FP8 doubles the FLOPs per byte of the linear layers
 * and moves their knee to the right: Sarathi-Serve reading notes, section
 * 7.7).  Format: OCP E4M3 (largest finite magnitude 448).  For each row r of
 * x [rows][cols] (device bf16):
 *   amax = max_c |x[r][c]|, inv = 448 / amax, scale[r] = amax / 448
 *   (correctly rounded fp32 divisions),
 *   q[r][c] = E4M3(fp32(x[r][c] * inv)), nearest-even, saturating to +-448;
 * an all-zero row gets scale 0 and zero codes.  q: device bytes
 * [rows][cols]; scale: device fp32 [rows].  cols % 16 == 0 and cols <= 32768,
 * x and q 16-byte aligned.  Asynchronous on stream.  Used for weights (rows =
 * output channels) and for activations (rows = tokens).
 * ---------------------------------------------------------------------- */
hb_status hb_quantize_e4m3(const void* x, void* q, float* scale, int32_t rows, int32_t cols, void* stream);

/* ------------------------------------------------------------------------
 * hb_gemm_e4m3 - C = epilogue(s_a[m] s_b[n] (A B^T)) with E4M3 operands on
 * the tensor cores (kind::f8f6f4, fp32 accumulate): A [M][K] codes with
 * per-row scales s_a [M], B [N][K] codes with per-row scales s_b [N] (both
 * from hb_quantize_e4m3).  The epilogues are hb_gemm's, applied to the
 * scaled accumulator (SWIGLU: s_b holds the scales of the interleaved rows).
 * K % 16 == 0, N % 8 == 0 (N % 128 for SWIGLU); A, B, C, R and s_b 16-byte
 * aligned.
 * ---------------------------------------------------------------------- */
hb_status hb_gemm_e4m3(const void* A, const float* s_a, const void* B, const float* s_b, void* C, const void* R,
                       int32_t M, int32_t N, int32_t K, int32_t epilogue, void* stream);

/* Weight preparation: w_gu[2 Fp][d], Fp = F rounded up to a multiple of 64,
 * from w_gate[F][d] and w_up[F][d] (device bf16): rows interleaved in blocks
 * of 64 ([gate 0..63, up 0..63, gate 64..127, ...]); rows of the padding
 * (gate/up index >= F) are zero.  F % 8 == 0, d % 8 == 0. */
hb_status hb_interleave_gate_up(const void* w_gate, const void* w_up, void* w_gu, int32_t F, int32_t d,
                                void* stream);

/* ------------------------------------------------------------------------
 * hb_fold_gamma - weight preparation for the folded RMSNorm:
 * out[r][c] = bf16(w[r][c] * gamma[c]) for a weight w [rows][cols] that
 * consumes RMSNorm(x; gamma) rows (cols = d_model).  Device bf16 buffers,
 * cols % 8 == 0, 16-byte aligned; out may alias w.  Asynchronous on stream.
 * ---------------------------------------------------------------------- */
hb_status hb_fold_gamma(const void* w, const void* gamma, void* out, int32_t rows, int32_t cols, void* stream);

/* ------------------------------------------------------------------------
 * hb_layer_forward - one decoder layer over a packed hybrid batch:
 *   xn = RMSNorm(x; g1); qkv = xn W_qkv^T; RoPE + KV append;
 *   o = attention; h = x + o W_o^T; hn = RMSNorm(h; g2);
 *   x_out = h + (silu(hn W_g^T) * hn W_u^T) W_d^T
 * the "run_iteration(B)" step of the scheduling loop (Sarathi-Serve reading
 * notes, section 3.4) for one layer.
 *   w      : device weights, prepared once (see hb_layer_weights): both
 *            RMSNorm gains folded in, gate/up interleaved.  The norms run
 *            inside the projections: (x * r * g) W^T = r * x (W diag g)^T
 *            with r = 1/sqrt(mean(x^2) + eps) applied per row in fp32 to the
 *            accumulators of the QKV and gate/up GEMMs.  HB_WEIGHTS_E4M3:
 *            x, o, h and the SwiGLU output are quantized per token
 *            (hb_quantize_e4m3's rule, r still from the bf16 rows) and the
 *            projections run as hb_gemm_e4m3; d_ff % 16 == 0 required.  With
 *            E4M3 weights and (n_q + 2 n_kv) d_head % 256 == 0 the RoPE and
 *            KV append run inside the QKV projection (same results; the
 *            rope+kv stage is then empty).
 *   plan   : device plan; rope: table from hb_rope_table with max_pos rows
 *   x_in   : device bf16 [T][d_model]; x_out may alias x_in
 *   caches : updated in place with this iteration's K/V
 *   workspace: hb_layer_workspace_bytes(dims, max_rows, max_seqs, max_kv_len)
 *   prof   : optional (NULL): when set, events[k] (cudaEvent_t) is recorded
 *            on `stream` before stage k and events[HB_LAYER_STAGES] after the
 *            last, stages = rmsnorm1 (row statistics of x), qkv, rope+kv,
 *            attention, o+residual (+ statistics of h), rmsnorm2 (no launch:
 *            folded), gate/up+swiglu, down+residual.  HB_WEIGHTS_E4M3: the
 *            quantization of a projection's input is part of the stage of
 *            that projection (rmsnorm1 quantizes x).
 * ---------------------------------------------------------------------- */
typedef enum hb_weight_format {
  HB_WEIGHTS_BF16 = 0, /* bf16 matrices */
  HB_WEIGHTS_E4M3 = 1  /* each matrix as E4M3 codes of its bf16 form (hb_quantize_e4m3) with per-row scales;
                          the four projection inputs are quantized per token inside the layer */
} hb_weight_format;

typedef struct hb_layer_weights {
  const void* w_qkv;  /* [(n_q + 2 n_kv) d_head][d_model] = W_qkv diag(g1) (hb_fold_gamma) */
  const void* w_o;    /* [d_model][n_q d_head] */
  const void* w_gu;   /* [2 Fp][d_model]: hb_interleave_gate_up of W_g, W_u (Fp = d_ff rounded up to
                         64), then hb_fold_gamma with g2 */
  const void* w_d;    /* [d_model][d_ff] */
  const float* s_qkv; /* HB_WEIGHTS_E4M3: per-row scales of the four matrices (16-byte aligned); */
  const float* s_o;   /* NULL for HB_WEIGHTS_BF16 */
  const float* s_gu;
  const float* s_d;
  int32_t format;     /* hb_weight_format */
} hb_layer_weights;

#define HB_LAYER_STAGES 8
typedef struct hb_profile {
  void** events;      /* cudaEvent_t[n_events] */
  int32_t n_events;   /* >= HB_LAYER_STAGES + 1 */
} hb_profile;

size_t hb_layer_workspace_bytes(const hb_layer_dims* dims, int32_t max_rows, int32_t max_seqs,
                                int32_t max_kv_len);
hb_status hb_layer_forward(const hb_layer_weights* w, const hb_layer_dims* dims, const hb_device_plan* plan,
                           const void* rope, int32_t max_pos, const void* x_in, void* x_out,
                           void* k_cache, void* v_cache, int32_t num_pages, int32_t max_kv_len,
                           void* workspace, size_t ws_bytes, void* stream, const hb_profile* prof);

/* ------------------------------------------------------------------------
 * hb_layers_forward - the layer stack of one hybrid iteration: n_layers
 * decoder layers back to back over the same packed batch, each layer's
 * output the next one's input (the per-layer "run_iteration(B)" step of the
 * scheduling loop, Sarathi-Serve reading notes section 3.4, repeated down
 * the model).  Layer l uses w[l] and the KV pools k_caches[l], v_caches[l]
 * (host arrays of n_layers device pointers); layer 0 reads x_in, every
 * layer writes x_out (x_out may alias x_in); one workspace serves all
 * layers (hb_layer_workspace_bytes).  The results are those of n_layers
 * hb_layer_forward calls, bit for bit: a bf16 layer after the first takes
 * the row statistics of its input from the previous layer's down
 * projection, which writes them in the same order as the statistics
 * kernel, and that kernel is left out (one launch less per layer).
 * Errors as hb_layer_forward; nothing is launched when any layer's
 * arguments are invalid.
 * ---------------------------------------------------------------------- */
hb_status hb_layers_forward(const hb_layer_weights* w, int32_t n_layers, const hb_layer_dims* dims,
                            const hb_device_plan* plan, const void* rope, int32_t max_pos, const void* x_in,
                            void* x_out, void* const* k_caches, void* const* v_caches, int32_t num_pages,
                            int32_t max_kv_len, void* workspace, size_t ws_bytes, void* stream);

/* hb_layer_kernel_count - how many kernels one hb_layer_forward call launches
 * for n_rows packed rows with weights in `format` (host logic only, no
 * device call; the chunk and decode attention kernels
 * count whatever the batch holds, n_rows == 0 launches nothing).  bf16: 8;
 * E4M3: 11, or 10 when the RoPE and KV append run inside the QKV
 * projection.  *count written on HB_OK; HB_ERR_INVALID_ARG for a null
 * pointer, bad dims, n_rows < 0 or an unknown format. */
hb_status hb_layer_kernel_count(const hb_layer_dims* dims, int32_t n_rows, int32_t format, int32_t* count);

/* ------------------------------------------------------------------------
 * hb_final_logits - final RMSNorm + untied LM head for selected rows (the
 * decode rows and the last chunk row of a model-level iteration):
 *   logits[i] = RMSNorm(x[rows[i]]; g_f) W_lm^T  (fp32 out)
 * x: device bf16 [T][d]; rows: device int32 [n_sel], each in [0, T) (a row
 * outside sets HB_ERR_DEVICE and is skipped); g_f bf16 [d]; w_lm bf16
 * [vocab][d]; logits fp32 [n_sel][vocab]; workspace of n_sel*d*2 bytes
 * (256-byte aligned).  vocab % 64 == 0, d % 64 == 0.
 * ---------------------------------------------------------------------- */
hb_status hb_final_logits(const void* x, int32_t T, const int32_t* rows, int32_t n_sel, const void* g_f,
                          const void* w_lm, int32_t vocab, int32_t d, float eps, void* logits, void* workspace,
                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * hb_check_status - synchronise `stream`, then read and clear the device
 * status word of the current device: HB_OK, HB_ERR_TIMEOUT (a bounded wait
 * inside a kernel expired) or HB_ERR_DEVICE (an index check failed).
 * ---------------------------------------------------------------------- */
hb_status hb_check_status(void* stream);

/* Number of SMs of the current device and whether it is sm_103 (1/0). */
hb_status hb_device_info(int32_t* num_sms, int32_t* is_sm103);

/* Kernels this library has launched in this process so far, over every
 * device and host thread (a launch counts once the CUDA runtime accepts
 * it).  Read it before and after a region to count that region's kernels;
 * needs no device. */
uint64_t hb_kernel_launches(void);

/* ------------------------------------------------------------------------
 * hb_selftest_wait_timeout - exercise the failure path of the bounded
 * device waits without faulting the GPU.  The pages define no such
 * operation: it checks this library's own error reporting.  One thread of
 * one CTA waits on a shared-memory barrier that nothing completes; after
 * timeout_us microseconds (1 .. 1 000 000) the wait gives up, records a
 * timeout in the device status word and the kernel returns.  The next
 * hb_check_status on `stream` returns HB_ERR_TIMEOUT and clears the word;
 * the context stays usable.  Argument errors return HB_ERR_INVALID_ARG
 * before any device work.
 * ---------------------------------------------------------------------- */
hb_status hb_selftest_wait_timeout(int32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* HB_H_ */
