"""Oracle of one decoder-layer forward over a packed hybrid batch (test
infrastructure only).

What the hybrid iteration computes (chunked prefill, Sarathi-Serve reading
notes section 3.1; chunked prefill knowledge page, mechanism section): chunk i
of a prompt covers positions [(i-1)C, iC), writes their KV into the paged
cache, and its queries attend to every key written by earlier chunks plus the
causal part of their own chunk; a decode row attends to its full context.
Chunking only re-partitions the work, so the result is the plain causal
attention of every row over keys 0..pos.

The layer arithmetic (absent from the pages) is the Llama/Mistral pre-norm
block without biases:
    xn = RMSNorm(x; g1)                y = x / sqrt(mean(x^2) + eps) * g
    q, k, v = split(xn W_qkv^T)
    q, k = RoPE(q, k; pos)             rotate-half, inv_freq_i = theta^(-2i/d_head)
    k, v -> paged cache at slot        (k stored after rotation)
    o = softmax(q k^T / sqrt(d_head)) v     per q head h on kv head h*n_kv//n_q
    h = x + o W_o^T
    out = h + (silu(hn W_g^T) * (hn W_u^T)) W_d^T,  hn = RMSNorm(h; g2)

Everything is computed in `dtype` (float32 by default), with no intermediate
rounding; inputs are the bf16-representable values the GPU also sees.

Precision variant (storage="bf16"): the same arithmetic in fp32 but with every
tensor that a bf16 implementation stores rounded to bf16 (round to nearest
even) where it is stored: qkv, the rotated q and k, the softmax weights P
fed to the P V product, o, h, the SwiGLU output a and the layer output.  The
normalised rows xn and hn are never stored: each RMSNorm is applied as
    RMSNorm(v; g) W^T = (v (W diag g)^T) / sqrt(mean(v^2) + eps),
the algebraic identity of a per-row scale, with W diag g rounded once to
bf16 (the prepared weights) and the 1/rms factor applied to the fp32 product.
It quantifies how far bf16 storage alone moves a result from the fp32 one;
the default path never rounds.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x):
    """Round float32 values to bf16 (nearest, ties to even), kept in float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(x.shape)


def rmsnorm(x, g, eps, dtype=np.float32):
    x = np.asarray(x, dtype)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + dtype(eps)) * np.asarray(g, dtype)


def rope_tables(max_pos, d_head, theta):
    """cos/sin of pos * theta^(-2i/d_head), i < d_head/2, computed in float64 and
    rounded to float32 (shape [max_pos, d_head/2])."""
    i = np.arange(d_head // 2, dtype=np.float64)
    inv_freq = np.power(np.float64(theta), -2.0 * i / d_head)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def rope(x, pos, cos, sin, dtype=np.float32):
    """Rotate-half RoPE. x [rows, heads, d_head], pos [rows]."""
    x = np.asarray(x, dtype)
    half = x.shape[-1] // 2
    c = np.asarray(cos, dtype)[pos][:, None, :]
    s = np.asarray(sin, dtype)[pos][:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1 + np.exp(-x))


def kv_append(k, v, slots, k_pool, v_pool, page):
    """Write rows' K [rows, n_kv, d_head] and V into the paged pools at slots."""
    for r, sl in enumerate(slots):
        k_pool[sl // page, :, sl % page, :] = k[r]
        v_pool[sl // page, :, sl % page, :] = v[r]


def gather_keys(pool, table_row, n_keys, page):
    """Keys 0..n_keys-1 of one sequence through its block table -> [n_keys, n_kv, d]."""
    j = np.arange(n_keys)
    pages = np.asarray(table_row)[j // page]
    return pool[pages, :, j % page, :]


def attention(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype=np.float32, round_p=None):
    """q [T, n_q, d_head] -> o [T, n_q, d_head]; row r of sequence s at
    position p attends to keys 0..p of s (its block table).  round_p, if
    given, is applied to the softmax weights before the P V product."""
    T, _, d_head = q.shape
    scale = dtype(1.0 / np.sqrt(d_head))
    grp = n_q // n_kv
    o = np.zeros((T, n_q, d_head), dtype)
    for s in range(len(plan.seq_pos0)):
        K = gather_keys(k_pool, plan.block_table[s], plan.seq_kv_len[s], page).astype(dtype)
        V = gather_keys(v_pool, plan.block_table[s], plan.seq_kv_len[s], page).astype(dtype)
        for r in range(plan.seq_q_start[s], plan.seq_q_start[s + 1]):
            n_keys = plan.row_pos[r] + 1
            for g in range(n_kv):
                qg = q[r, g * grp:(g + 1) * grp, :].astype(dtype)      # [grp, d]
                sc = (qg @ K[:n_keys, g, :].T) * scale                  # [grp, n_keys]
                sc = sc - sc.max(axis=1, keepdims=True)
                w = np.exp(sc)
                if round_p is None:
                    w = w / w.sum(axis=1, keepdims=True)
                    o[r, g * grp:(g + 1) * grp, :] = w @ V[:n_keys, g, :]
                else:
                    o[r, g * grp:(g + 1) * grp, :] = (round_p(w) @ V[:n_keys, g, :]) / w.sum(axis=1, keepdims=True)
    return o


def layer_forward(w, dims, plan, x, k_pool, v_pool, cos, sin, dtype=np.float32,
                  return_parts=False, storage=None):
    """One decoder layer over the packed rows of `plan`.  k_pool / v_pool are
    updated in place with the rows' rotated K and raw V.  storage="bf16"
    selects the bf16-storage precision variant (module docstring)."""
    T = len(plan.row_seq)
    nq, nkv, dh = dims.n_q, dims.n_kv, dims.d_head
    st = round_bf16 if storage == "bf16" else (lambda t: t)
    x = np.asarray(x, dtype)

    def inv_rms(v):
        return 1.0 / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + dtype(dims.eps))

    def normed_proj(v, g, w_):
        """RMSNorm(v; g) W^T: plainly in fp32; with bf16 storage the gain is
        folded into W (rounded once) and 1/rms scales the product."""
        if storage == "bf16":
            wf = round_bf16(np.asarray(w_, np.float32) * np.asarray(g, np.float32)[None, :]).astype(dtype)
            return (v @ wf.T) * inv_rms(v)
        return rmsnorm(v, g, dims.eps, dtype) @ np.asarray(w_, dtype).T

    xn = rmsnorm(x, w["g1"], dims.eps, dtype)
    qkv = st(normed_proj(x, w["g1"], w["w_qkv"]))
    q = qkv[:, :nq * dh].reshape(T, nq, dh)
    k = qkv[:, nq * dh:(nq + nkv) * dh].reshape(T, nkv, dh)
    v = qkv[:, (nq + nkv) * dh:].reshape(T, nkv, dh)
    pos = np.asarray(plan.row_pos)
    q = st(rope(q, pos, cos, sin, dtype))
    k = st(rope(k, pos, cos, sin, dtype))
    kv_append(k, v, plan.slot_mapping, k_pool, v_pool, dims.page)
    o = st(attention(q, k_pool, v_pool, plan, nq, nkv, dims.page, dtype,
                     round_p=round_bf16 if storage == "bf16" else None))
    h = st(x + o.reshape(T, nq * dh) @ np.asarray(w["w_o"], dtype).T)
    hn = rmsnorm(h, w["g2"], dims.eps, dtype)
    a = st(silu(normed_proj(h, w["g2"], w["w_g"])) * normed_proj(h, w["g2"], w["w_u"]))
    out = st(h + a @ np.asarray(w["w_d"], dtype).T)
    if return_parts:
        return out, dict(xn=xn, qkv=qkv, q=q, k=k, v=v, o=o, h=h, hn=hn, a=a)
    return out


def lm_head(x_rows, g_f, w_lm, eps, dtype=np.float32):
    """Final RMSNorm then the untied LM head -> logits [rows, vocab]."""
    return rmsnorm(x_rows, g_f, eps, dtype) @ np.asarray(w_lm, dtype).T
