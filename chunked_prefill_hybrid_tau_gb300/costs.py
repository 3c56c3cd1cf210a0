"""Algorithmic FLOPs and bytes of a hybrid iteration, per kernel stage.

These are the work the method itself requires (no re-reads, no padding):
  * a projection of T packed rows with a [N][K] weight: 2*T*N*K FLOPs and
    N*K*2 weight bytes (read once) + T*K*2 input + T*N*2 output bytes;
  * attention: 4*n_q*d_head*(p+1) FLOPs for a row at position p (QK^T and
    PV over keys 0..p); bytes = every visible key's K and V once per
    sequence and kv head (n_kv*d_head*2*2 per key) + q and o;
  * RMSNorm / RoPE+append: their reads and writes.
The per-iteration roofline is t_roof = max(FLOPs / peak FLOP/s, bytes / peak
B/s) of the whole layer (linear-layer roofline of the Sarathi-Serve reading
notes, section 1.6, extended with the attention's KV reads as in the hybrid-
iteration intensity of the Chunked Prefill page).

E4M3 weights (weight_bytes=1): a weight matrix is read at one byte per
parameter and the projections' FLOPs run at the FP8 tensor rate, twice the
bf16 one (section 7.7 of the reading notes: FP8 doubles FLOPs per byte);
activations stay bf16 in the algorithmic count.
"""
from __future__ import annotations

import numpy as np

STAGES = ["rmsnorm1", "qkv", "rope_kv", "attention", "o_proj", "rmsnorm2", "gate_up", "down"]


def stage_costs(dims, row_pos, seq_q_start, seq_kv_len, weight_bytes=2):
    """{stage: (flops, bytes, bound)} for one layer over the packed rows."""
    T = len(row_pos)
    d, dh, nq, nkv, F = dims.d_model, dims.d_head, dims.n_q, dims.n_kv, dims.d_ff
    qkv_cols = (nq + 2 * nkv) * dh
    hd = nq * dh
    b = 2  # bf16
    sw = weight_bytes

    def gemm(N, K):
        return 2.0 * T * N * K, float(N * K * sw + T * K * b + T * N * b)

    kv_len = np.asarray(seq_kv_len, np.int64)
    pos = np.asarray(row_pos, np.int64)
    attn_flops = 4.0 * nq * dh * float(np.sum(pos + 1))
    attn_bytes = float(np.sum(kv_len)) * nkv * dh * b * 2 + T * hd * b * 2
    c = {
        "rmsnorm1": (3.0 * T * d, float(2 * T * d * b + d * b), "hbm"),
        "qkv": gemm(qkv_cols, d) + ("tensor",),
        "rope_kv": (6.0 * T * (nq + nkv) * dh, float(T * qkv_cols * b * 2 + T * dh // 2 * 8), "hbm"),
        "attention": (attn_flops, attn_bytes, "hbm"),
        "o_proj": (gemm(d, hd)[0], gemm(d, hd)[1] + T * d * b, "tensor"),
        "rmsnorm2": (3.0 * T * d, float(2 * T * d * b + d * b), "hbm"),
        "gate_up": (2.0 * T * 2 * F * d, float(2 * F * d * sw + T * d * b + T * F * b), "tensor"),
        "down": (gemm(d, F)[0], gemm(d, F)[1] + T * d * b, "tensor"),
    }
    return c


def roofline_time(costs: dict, tflops_bf16: float, hbm_gbs: float, f8: bool = False) -> float:
    """t_roof = max(sum of FLOPs over their tensor rates, bytes / HBM B/s); with
    f8 the projections (the "tensor" stages other than attention) run at twice
    the bf16 rate."""
    t_math = 0.0
    for name, (fl, _, bound) in costs.items():
        rate = tflops_bf16 * (2.0 if (f8 and bound == "tensor") else 1.0)
        t_math += fl / (rate * 1e12)
    byts = sum(v[1] for v in costs.values())
    return max(t_math, byts / (hbm_gbs * 1e9))


def iteration_totals(costs: dict):
    flops = sum(v[0] for v in costs.values())
    byts = sum(v[1] for v in costs.values())
    return flops, byts


def page_intensity(c, b, psi, s_psi, n_layers, n_kv, d_head, s_bar):
    """Hybrid-iteration arithmetic intensity as the Chunked Prefill page
    writes it: 2(c+b)Psi / (s_Psi Psi + 2 L n_kv d_head s_bar b)."""
    return 2.0 * (c + b) * psi / (s_psi * psi + 2.0 * n_layers * n_kv * d_head * s_bar * b)
