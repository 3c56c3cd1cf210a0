"""Oracle cost model of a hybrid iteration (test infrastructure only).

* Chunked-attention pair counts (Sarathi-Serve reading notes, section 7.5b):
  a query at position i of a prompt looks at i+1 keys, so a prompt of length
  L costs sum_i (i+1) = L(L+1)/2 (query, key) pairs whether it is prefilled
  at once or in chunks; chunk k (1-based, size C) alone costs
  (k-1) C^2 + C(C+1)/2.
* Hybrid-iteration arithmetic intensity (chunked prefill knowledge page,
  "hybrid iteration roofline and prefill budget"): with c chunk tokens and b
  decodes, FLOPs 2(c+b)Psi, weight bytes s_Psi * Psi (read once), KV reads
  2 L n_kv d_head s_bar b, so
      I = 2(c+b)Psi / (s_Psi Psi + 2 L n_kv d_head s_bar b),
  and the chunk that brings I to I* is
      c* = I*/(2 Psi) (s_Psi Psi + 2 L n_kv d_head s_bar b) - b.
  The KV term is taken literally as printed (an element count, no bytes per
  element); s_bar is the decodes' mean prior context.
"""
from __future__ import annotations


def intensity_closed_form(c, b, psi, s_psi, n_layers, n_kv, d_head, s_bar):
    return 2.0 * (c + b) * psi / (s_psi * psi + 2.0 * n_layers * n_kv * d_head * s_bar * b)


def c_star(i_star, b, psi, s_psi, n_layers, n_kv, d_head, s_bar):
    return i_star / (2.0 * psi) * (s_psi * psi + 2.0 * n_layers * n_kv * d_head * s_bar * b) - b


def chunk_pairs_closed_form(k, C):
    """(query, key) pairs of the k-th full chunk (1-based) of size C."""
    return (k - 1) * C * C + C * (C + 1) // 2


def prompt_pairs_closed_form(L):
    return L * (L + 1) // 2


def count_pairs(row_pos):
    """Brute-force (query, key) pair count of rows at the given positions."""
    return sum(p + 1 for p in row_pos)


def count_iteration(plan, psi, s_psi, n_layers, n_kv, d_head):
    """Walk a plan's rows and keys: linear FLOPs and the bytes of the page's
    intensity model (weights once + prior KV elements of every decode row)."""
    flops = 0
    kv_elems = 0
    for s in range(len(plan.seq_pos0)):
        for r in range(plan.seq_q_start[s], plan.seq_q_start[s + 1]):
            flops += 2 * psi
            if plan.seq_kind[s] == 0:
                for _ in range(plan.row_pos[r]):          # prior keys of this decode
                    kv_elems += 2 * n_layers * n_kv * d_head
    return flops, s_psi * psi + kv_elems
