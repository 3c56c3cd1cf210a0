"""Oracle of the FP8 (E4M3) projections (test infrastructure only).

What it computes.  The Sarathi-Serve reading notes (section 7.7, what changes
on Hopper-class GPUs) say that FP8 moves the knee of the linear layers to
the right because it doubles the FLOPs per byte.  They fix neither the FP8
format nor how values are scaled into it, so this module takes the plain
reading (listed with the other readings in the design notes):

  * format: the 8-bit floating-point format E4M3 of the OCP FP8
    specification: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
    subnormals when the exponent field is 0; the pattern S.1111.111 is NaN,
    so there is no infinity and the largest finite magnitude is 448;
  * scaling: one fp32 scale per row of each operand (per output channel of a
    weight, per token of an activation), chosen from the row's largest
    magnitude: inv = 448 / amax and scale = amax / 448, both divisions
    correctly rounded in fp32, and code = E4M3(fp32(v * inv)) rounded to
    nearest with ties to even, magnitudes above 448 clamped to 448
    ("saturating" conversion); an all-zero row gets scale 0 and zero codes;
  * projection: C[m][n] = s_a[m] * s_b[n] * sum_k qa[m][k] * qb[n][k].  The
    codes' values are small dyadic rationals (4 significant bits, exponents
    2^-9 .. 2^8), so the sum of their products is exact in float64 for any
    K used here and the oracle computes it there.

Which quantities are quantized in the layer: the four projection inputs
(x, the attention output o, h, and the SwiGLU output a) and the four prepared
weight matrices.  The weights are the bf16 matrices the bf16 layer uses
(W_qkv diag(g1) and W_{g,u} diag(g2) each rounded once to bf16), quantized
row by row.  Everything else (norm factors, RoPE, attention, SwiGLU,
residuals) is the bf16 layer's arithmetic (oracle.layer).

Parity notes.  A code is an integer decided by floating point; this module
takes each decision in fp32, as the device does, so that codes computed from
the same fp32 inputs agree bit for bit.  Inside the layer the device
quantizes its bf16-stored activations; the oracle's storage="bf16" variant
rounds the same tensors to bf16 before quantizing them.
"""
from __future__ import annotations

import numpy as np

from . import layer as ol

E4M3_MAX = 448.0


def e4m3_table():
    """Value of each of the 256 E4M3 codes (float64; NaN for S.1111.111):
    normal (1 + M/8) 2^(E-7) = (8 + M) 2^(E-10) for E >= 1, subnormal
    (M/8) 2^-6 = M 2^-9 for E == 0."""
    c = np.arange(256)
    sign = np.where(c >> 7, -1.0, 1.0)
    E = (c >> 3) & 15
    M = (c & 7).astype(np.float64)
    mag = np.where(E == 0, M * 2.0 ** -9, (8.0 + M) * np.exp2(E.astype(np.float64) - 10.0))
    v = sign * mag
    v[(E == 15) & ((c & 7) == 7)] = np.nan
    return v


def e4m3_round(v):
    """Round to the nearest E4M3 value, ties to even, magnitudes above 448
    (and infinities) clamped to 448, NaN kept; returned as float64.

    The value is held in a binade [2^e, 2^(e+1)), e >= -6 (the subnormals
    share the spacing of the lowest binade), where E4M3 values are the
    multiples of 2^(e-3); rounding to a multiple is exact division by a power
    of two followed by round-half-even.  A value that rounds up to 2^(e+1)
    lands on the next binade's first value, which is the correct result."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    finite = np.isfinite(a)
    _, ex = np.frexp(np.where(finite, a, 1.0))     # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)
    step = np.ldexp(1.0, e - 3)
    r = np.rint(np.where(finite, a, 0.0) / step) * step
    r = np.where(finite, np.minimum(r, E4M3_MAX), E4M3_MAX)
    out = np.copysign(r, v)
    return np.where(np.isnan(v), np.nan, out)


_POS = e4m3_table()[:127]  # codes 0x00 .. 0x7E, strictly increasing


def e4m3_encode(v):
    """Codes (uint8) of e4m3_round(v): the sign bit of v (so -0 -> 0x80),
    then the position of the rounded magnitude among the positive values;
    NaN -> 0x7F with v's sign."""
    v = np.asarray(v, np.float64)
    r = e4m3_round(v)
    nan = np.isnan(r)
    idx = np.searchsorted(_POS, np.where(nan, 0.0, np.abs(r)))
    assert np.all(nan | (_POS[np.minimum(idx, 126)] == np.abs(np.where(nan, 0.0, r)))), "not an E4M3 value"
    code = np.where(nan, 0x7F, idx).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << 7)


def e4m3_decode(codes):
    return e4m3_table()[np.asarray(codes, np.uint8)]


def quantize_rows(x):
    """Per-row E4M3 quantization of x [rows][cols] (fp32 values):
    -> (codes uint8 [rows][cols], scale float32 [rows]) with
    x[r][c] ~ scale[r] * value(codes[r][c])."""
    x = np.asarray(x, np.float32)
    amax = np.max(np.abs(x), axis=-1)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1))
    inv = np.where(nz, np.float32(E4M3_MAX) / safe, np.float32(0)).astype(np.float32)
    scale = np.where(nz, amax / np.float32(E4M3_MAX), np.float32(0)).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)  # one fp32 product per element
    return e4m3_encode(y), scale


def dequantize_rows(codes, scale):
    return e4m3_decode(codes) * np.asarray(scale, np.float64)[..., None]


def gemm(qa, sa, qb, sb):
    """C = s_a[m] s_b[n] sum_k qa[m][k] qb[n][k] (float64; the code sum is exact)."""
    acc = e4m3_decode(qa) @ e4m3_decode(qb).T
    return acc * np.asarray(sa, np.float64)[:, None] * np.asarray(sb, np.float64)[None, :]


def prepare_weights(w):
    """The prepared bf16 weights (gains folded, rounded once to bf16), then
    per-row codes and scales: dict name -> (codes, scale) for qkv, o, g, u, d."""
    f32 = np.float32
    fold = {
        "qkv": ol.round_bf16(np.asarray(w["w_qkv"], f32) * np.asarray(w["g1"], f32)[None, :]),
        "o": np.asarray(w["w_o"], f32),
        "g": ol.round_bf16(np.asarray(w["w_g"], f32) * np.asarray(w["g2"], f32)[None, :]),
        "u": ol.round_bf16(np.asarray(w["w_u"], f32) * np.asarray(w["g2"], f32)[None, :]),
        "d": np.asarray(w["w_d"], f32),
    }
    def by_rows(m, block=2048):  # rows are independent; blocks only bound the memory in use
        parts = [quantize_rows(m[i:i + block]) for i in range(0, m.shape[0], block)]
        return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])

    return {k: by_rows(v) for k, v in fold.items()}


def layer_forward(wq, dims, plan, x, k_pool, v_pool, cos, sin, storage=None, dtype=np.float32,
                  return_parts=False):
    """One decoder layer with E4M3 projections (module docstring); wq from
    prepare_weights.  RMSNorm stays in the projections that consume it:
    RMSNorm(v; g) W^T = r (v (W diag g)^T), r = 1/sqrt(mean(v^2) + eps) per row,
    with v's quantized codes standing in for v.  storage="bf16" rounds the
    tensors that a bf16 implementation stores, as in oracle.layer."""
    T = len(plan.row_seq)
    nq, nkv, dh = dims.n_q, dims.n_kv, dims.d_head
    st = ol.round_bf16 if storage == "bf16" else (lambda t: t)

    def inv_rms(v):
        v = np.asarray(v, dtype)
        return 1.0 / np.sqrt(np.mean(v * v, axis=-1) + dtype(dims.eps))

    def proj(v, name):
        qa, sa = quantize_rows(v)
        qb, sb = wq[name]
        return gemm(qa, sa, qb, sb).astype(dtype)

    x = np.asarray(x, dtype)
    qkv = st(inv_rms(x)[:, None] * proj(x, "qkv"))
    q = qkv[:, :nq * dh].reshape(T, nq, dh)
    k = qkv[:, nq * dh:(nq + nkv) * dh].reshape(T, nkv, dh)
    v = qkv[:, (nq + nkv) * dh:].reshape(T, nkv, dh)
    pos = np.asarray(plan.row_pos)
    q = st(ol.rope(q, pos, cos, sin, dtype))
    k = st(ol.rope(k, pos, cos, sin, dtype))
    ol.kv_append(k, v, plan.slot_mapping, k_pool, v_pool, dims.page)
    o = st(ol.attention(q, k_pool, v_pool, plan, nq, nkv, dims.page, dtype,
                        round_p=ol.round_bf16 if storage == "bf16" else None))
    h = st(x + proj(o.reshape(T, nq * dh), "o"))
    r = inv_rms(h)[:, None]
    a = st(ol.silu(r * proj(h, "g")) * (r * proj(h, "u")))
    out = st(h + proj(a, "d"))
    if return_parts:
        return out, dict(qkv=qkv, o=o, h=h, a=a)
    return out
