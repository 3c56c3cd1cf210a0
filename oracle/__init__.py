"""CPU oracle for the hybrid-iteration forward: TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct NumPy restatement of what one hybrid
iteration computes (token-budget packing with paged KV slots, then one
decoder-layer forward over the packed rows).  Only the test-suite,
`__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
it.  It shares no code with the CUDA library and neither imports the other.

Sources (three web pages on chunked prefill):
  * "Sarathi-Serve ... reading notes" (zhongzhuzhou.org), section 3.1
    (chunked prefills), 3.2 (stall-free hybrid batching), 3.4 (scheduling
    loop), 7.5b (FLOP arithmetic of chunked attention), 7.6 (worked Yi-34B
    iteration);
  * "Chunked Prefill" (bowenzhou.top), mechanism section (chunks continue
    writing paged KV) and the derivation of the hybrid-iteration arithmetic
    intensity I and the optimal chunk c*.
The decoder-layer arithmetic (RMSNorm, GQA, rotate-half RoPE, SwiGLU) is not
on the pages; the oracle takes the standard Llama/Mistral pre-norm block.

Precision: float32 by default (the oracle precision the workload contract
fixes); every function takes a `dtype` so the pins can also run in float64.

Parity status per function (what pins it, in tests/test_oracle_pins.py):
  plan.plan_batch        worked example of section 7.6; invariants of the
                         greedy rule; brute-force enumeration on tiny queues
  layer.attention        brute-force dense masked softmax in float64
  layer.rmsnorm          unit RMS at gain 1, scale invariance
  layer.rope             identity at position 0, pair-norm preservation,
                         relative-position property
  layer.silu             logistic-function identity (scipy.special.expit)
  layer.layer_forward    closed forms of a hand-wired layer (single routes
                         through each projection: q/k/v order and head
                         layout, GQA groups, W_o orientation, residual
                         sources, the gains of the two norms, gate versus
                         up); chunked == unchunked; decode batch
                         independence; identity when the output
                         projections are zero
  costs.*                chunked-attention pair-count identity (section
                         7.5b); closed form of I and c* against counters
  sched.SchedLoop        closed form of one request's iterations; token and
                         page conservation; a step-by-step replay on tiny
                         streams
  fp8.* (E4M3 projections, reading notes section 7.7; tests/test_oracle_fp8.py)
                         the 256-code table and round-to-nearest-even
                         against torch's float8_e4m3fn conversion;
                         saturation; per-row scaling bounds and invariances;
                         the projection against exact rational sums; the
                         layer's QKV exact on representable inputs, chunked
                         == unchunked, within E4M3's error of the bf16
                         layer, and within E4M3's error of the hand-wired
                         layer's closed forms
"""
