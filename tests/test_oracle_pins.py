"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each pin is a function of the oracle module(s) so that the planted-mistake
tests at the bottom can run it against a mutated oracle and check that it
fails.  Nothing here touches the CUDA library.
"""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle.costs as oc
import oracle.layer as ol
import oracle.plan as op
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# helpers: tiny problems
# ----------------------------------------------------------------------------
def tiny_dims(**kw):
    base = dict(d_model=32, n_q=4, n_kv=2, d_head=8, d_ff=48, theta=1e4)
    base.update(kw)
    return wl.Dims(**base)


def tiny_state(rng, dims, dec_ctx, prefills, slack=64):
    return wl.make_state(rng, dims, dec_ctx, prefills, slack_pages=slack)


def plan_from_state(st, tau, chunk, page=16):
    return op.plan_batch([r.done for r in st.decodes], [r.pages for r in st.decodes],
                         [r.prompt_len for r in st.prefills], [r.done for r in st.prefills],
                         [r.pages for r in st.prefills], st.free_pool, tau, chunk, page)


# ----------------------------------------------------------------------------
# planner
# ----------------------------------------------------------------------------
def pin_worked_example(plan_mod=op):
    g = json.load(open(os.path.join(GOLDEN, "yi34b_worked_iteration.json")))
    ctx = g["decode_ctx"]
    pfs = g["prefills"]
    dec_pages = [list(range(1000 * (i + 1), 1000 * (i + 1) + wl.pages_for(c))) for i, c in enumerate(ctx)]
    pf_pages = [list(range(50000, 50000 + wl.pages_for(pfs[0]["done"]))), []]
    pool = list(range(100000, 100400))
    p = plan_mod.plan_batch(ctx, dec_pages, [r["prompt_len"] for r in pfs], [r["done"] for r in pfs],
                            pf_pages, pool, g["tau"], g["chunk"])
    e = g["expect"]
    n_dec = sum(1 for k in p.seq_kind if k == 0)
    assert n_dec == e["decode_tokens"]
    assert g["tau"] - n_dec == e["prefill_budget"]
    assert p.pf_take == e["take"]
    assert e["prefill_budget"] - p.pf_take[0] == e["budget_after_R_A"]
    assert p.n_rows == e["batch_tokens"]
    assert g["tau"] - p.n_rows == e["budget_left"]
    assert p.pf_finished == e["finished"]
    rem = [r["prompt_len"] - r["done"] - t for r, t in zip(pfs, p.pf_take)]
    assert rem == e["remaining_after"]
    assert [p.seq_kv_len[s] for s in range(n_dec, p.n_seqs)] == e["kv_positions_attended_by_last_row"]


def test_plan_worked_example():
    pin_worked_example()


def check_plan_invariants(p, dec_ctx, pf_len, pf_done, dec_pages0, pf_pages0, pool, tau, chunk, page=16):
    b = len(dec_ctx)
    # decodes first, one row each, at their context position
    assert p.seq_kind[:b] == [0] * b
    assert [p.row_pos[p.seq_q_start[s]] for s in range(b)] == list(dec_ctx)
    # budget respected (decodes always admitted)
    assert p.n_rows <= max(tau, b)
    assert p.over_budget == (1 if b > tau else 0)
    # FIFO prefix of prefills, one chunk each, chunk <= C, partial only when budget ends
    takes = p.pf_take
    seen_zero = False
    for j, t in enumerate(takes):
        full = min(chunk, pf_len[j] - pf_done[j])
        assert 0 <= t <= full
        if seen_zero:
            assert t == 0
        if t < full:
            seen_zero = True
            if t > 0 or full > 0:
                assert p.n_rows == tau or b >= tau
        assert p.pf_finished[j] == (1 if t > 0 and pf_done[j] + t == pf_len[j] else 0)
    assert p.n_rows == b + sum(takes)
    # rows of each sequence are consecutive positions starting at pos0
    for s in range(p.n_seqs):
        rows = range(p.seq_q_start[s], p.seq_q_start[s + 1])
        assert [p.row_pos[r] for r in rows] == list(range(p.seq_pos0[s], p.seq_kv_len[s]))
        assert all(p.row_seq[r] == s for r in rows)
    # slots: page table lookup, unique
    for r in range(p.n_rows):
        s, pos = p.row_seq[r], p.row_pos[r]
        assert p.slot_mapping[r] == p.block_table[s][pos // page] * page + pos % page
    assert len(set(p.slot_mapping)) == p.n_rows
    # pages popped from the front of the pool, in row order
    new_pages = []
    for s in range(p.n_seqs):
        held = (dec_pages0 if p.seq_kind[s] == 0 else pf_pages0)[p.seq_req[s]]
        for pg in p.block_table[s][len(held):]:
            if pg >= 0:
                new_pages.append(pg)
    assert new_pages == list(pool[:p.pages_used])
    assert p.free_pool == list(pool[p.pages_used:])


def brute_force_takes(dec_n, pf_rem, tau, chunk):
    """Enumerate every vector of takes (each 0..min(rem, C)) and keep the one
    that the greedy rule of the pages selects: maximal lexicographically in
    FIFO order subject to the budget (a request is only skipped when the
    budget is gone)."""
    import itertools
    budget = tau - dec_n
    best = None
    for takes in itertools.product(*[range(min(r, chunk) + 1) for r in pf_rem]):
        if sum(takes) > max(budget, 0):
            continue
        if best is None or list(takes) > list(best):
            best = takes
    return list(best)


def test_plan_brute_force_tiny():
    rng = np.random.default_rng(1)
    for _ in range(300):
        b = int(rng.integers(0, 5))
        n_pf = int(rng.integers(0, 4))
        tau = int(rng.integers(1, 40))
        chunk = int(rng.integers(1, 20))
        ctx = [int(v) for v in rng.integers(0, 50, b)]
        pf_len = [int(v) for v in rng.integers(1, 30, n_pf)]
        pf_done = [int(rng.integers(0, L)) for L in pf_len]
        dec_pages = [list(range(100 * i, 100 * i + wl.pages_for(c))) for i, c in enumerate(ctx)]
        pf_pages = [list(range(5000 + 100 * j, 5000 + 100 * j + wl.pages_for(d))) for j, d in enumerate(pf_done)]
        pool = [int(v) for v in rng.permutation(np.arange(9000, 9100))]
        p = op.plan_batch(ctx, dec_pages, pf_len, pf_done, pf_pages, pool, tau, chunk)
        exp = brute_force_takes(b, [L - d for L, d in zip(pf_len, pf_done)], tau, chunk)
        assert p.pf_take == exp, (b, tau, chunk, pf_len, pf_done)
        check_plan_invariants(p, ctx, pf_len, pf_done, dec_pages, pf_pages, pool, tau, chunk)


def test_plan_page_boundaries_and_out_of_pages():
    # ctx = 15 (last slot of a page), 16 (needs a new page), 0 (fresh)
    p = op.plan_batch([15, 16, 0], [[7], [8], []], [], [], [], [40, 41, 42], 8, 8)
    assert p.slot_mapping == [7 * 16 + 15, 40 * 16 + 0, 41 * 16 + 0]
    assert p.pages_used == 2 and p.free_pool == [42]
    with pytest.raises(op.OutOfPages):
        op.plan_batch([16, 32], [[1], [2, 3]], [], [], [], [9], 8, 8)


def test_plan_configs_packing():
    # every configuration reproduces b + c = tau with C = tau
    for tau, b, L, off in [(512, 32, 4096, 1024), (2048, 64, 8192, 0), (1024, 128, 16384, 0)]:
        ctx = [600] * b
        dp = [list(range(100 * i, 100 * i + wl.pages_for(600))) for i in range(b)]
        p = op.plan_batch(ctx, dp, [L], [off], [list(range(900000, 900000 + wl.pages_for(off)))],
                          list(range(10**6, 10**6 + 4000)), tau, tau)
        assert p.n_rows == tau and p.pf_take == [tau - b]
        assert p.row_pos[b] == off and p.row_pos[-1] == off + tau - b - 1


# ----------------------------------------------------------------------------
# chunked attention pair counts (section 7.5b)
# ----------------------------------------------------------------------------
def pin_pair_identity(plan_mod=op, costs_mod=oc):
    for L in [1, 2, 7, 64, 100, 513]:
        for C in [1, 3, 16, 64, 512, L]:
            done, rows, k = 0, [], 0
            pages = []
            pool = list(range(10**5))
            while done < L:
                p = plan_mod.plan_batch([], [], [L], [done], [pages], pool, C, C)
                pages = p.pf_pages[0]
                pool = p.free_pool
                chunk_rows = p.row_pos
                k += 1
                if len(chunk_rows) == C:
                    assert costs_mod.count_pairs(chunk_rows) == costs_mod.chunk_pairs_closed_form(k, C)
                rows += chunk_rows
                done += p.pf_take[0]
            assert rows == list(range(L))
            assert costs_mod.count_pairs(rows) == costs_mod.prompt_pairs_closed_form(L)
            if L % C == 0:
                K = L // C
                assert 2 * sum(costs_mod.chunk_pairs_closed_form(i, C) for i in range(1, K + 1)) == L * L + L


def test_pair_identity():
    pin_pair_identity()


def test_pair_identity_symbolic():
    # the page's algebra: C^2 (K-1)K/2 + K C(C+1)/2 = L^2/2 + L/2 with L = KC
    for K in range(1, 40):
        for C in range(1, 40):
            L = K * C
            lhs = sum(oc.chunk_pairs_closed_form(k, C) for k in range(1, K + 1))
            assert 2 * lhs == L * L + L


# ----------------------------------------------------------------------------
# arithmetic intensity I and c*
# ----------------------------------------------------------------------------
def pin_intensity(costs_mod=oc):
    rng = np.random.default_rng(3)
    dims = tiny_dims()
    psi = dims.params_per_layer
    for _ in range(20):
        b = int(rng.integers(1, 6))
        c = int(rng.integers(1, 40))
        ctx = [int(v) for v in rng.integers(1, 90, b)]
        dp = [list(range(100 * i, 100 * i + wl.pages_for(x))) for i, x in enumerate(ctx)]
        p = op.plan_batch(ctx, dp, [500], [0], [[]], list(range(10**4, 10**4 + 100)), b + c, c)
        flops, byts = costs_mod.count_iteration(p, psi, 2, 1, dims.n_kv, dims.d_head)
        closed = costs_mod.intensity_closed_form(c, b, psi, 2, 1, dims.n_kv, dims.d_head, float(np.mean(ctx)))
        assert math.isclose(flops / byts, closed, rel_tol=1e-12)
        # c* brings I exactly to the target
        i_star = closed * 1.7
        cs = costs_mod.c_star(i_star, b, psi, 2, 1, dims.n_kv, dims.d_head, float(np.mean(ctx)))
        i_at = costs_mod.intensity_closed_form(cs, b, psi, 2, 1, dims.n_kv, dims.d_head, float(np.mean(ctx)))
        assert math.isclose(i_at, i_star, rel_tol=1e-12)
    # pure decode (c = 0) has the lowest intensity; it rises monotonically with c
    vals = [costs_mod.intensity_closed_form(c, 32, 218e6, 2, 1, 8, 128, 2300) for c in range(0, 2000, 100)]
    assert all(a < b for a, b in zip(vals, vals[1:]))


def test_intensity():
    pin_intensity()


# ----------------------------------------------------------------------------
# RMSNorm, RoPE, SiLU
# ----------------------------------------------------------------------------
def pin_rmsnorm(layer=ol):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((16, 64))
    y = layer.rmsnorm(x, np.ones(64), 1e-6, np.float64)
    # RMS(y) = sqrt(m / (m + eps)) with m = mean(x^2)
    m = np.mean(x * x, axis=1)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(m / (m + 1e-6)), rtol=1e-12)
    # mean square equal to eps -> RMS 1/sqrt(2)
    z = np.full((1, 64), math.sqrt(1e-6))
    assert np.allclose(np.sqrt(np.mean(layer.rmsnorm(z, np.ones(64), 1e-6, np.float64) ** 2)),
                       1 / math.sqrt(2), rtol=1e-12)
    # scale invariance (eps negligible at this scale), gain multiplies
    g = rng.standard_normal(64)
    assert np.allclose(layer.rmsnorm(1000 * x, g, 1e-6, np.float64), layer.rmsnorm(x, g, 0.0, np.float64),
                       rtol=1e-9, atol=1e-12)


def test_rmsnorm():
    pin_rmsnorm()


def pin_rope(layer=ol):
    d = 16
    cos, sin = layer.rope_tables(64, d, 1e4)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 2, d))
    # position 0 is the identity
    assert np.array_equal(layer.rope(x, np.zeros(3, int), cos, sin, np.float64), x)
    # basis vector e_i at position p -> cos(p f_i) e_i + sin(p f_i) e_{i+d/2}
    for i in range(d // 2):
        for p in [1, 5, 63]:
            e = np.zeros((1, 1, d))
            e[0, 0, i] = 1
            r = layer.rope(e, np.array([p]), cos, sin, np.float64)[0, 0]
            ang = p * 1e4 ** (-2 * i / d)
            assert abs(r[i] - math.cos(ang)) < 1e-6 and abs(r[i + d // 2] - math.sin(ang)) < 1e-6
            assert np.count_nonzero(np.abs(r) > 1e-7) <= 2
    # per-pair norm preservation
    pos = np.array([3, 17, 40])
    r = layer.rope(x, pos, cos, sin, np.float64)
    h = d // 2
    assert np.allclose(r[..., :h] ** 2 + r[..., h:] ** 2, x[..., :h] ** 2 + x[..., h:] ** 2, rtol=1e-6)
    # relative position: <R_m q, R_n k> = <R_{m+t} q, R_{n+t} k>
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    dots = []
    for t in [0, 7, 20]:
        qm = layer.rope(q, np.array([10 + t]), cos, sin, np.float64)
        kn = layer.rope(k, np.array([4 + t]), cos, sin, np.float64)
        dots.append(float(np.sum(qm * kn)))
    assert np.allclose(dots, dots[0], rtol=1e-5)


def test_rope():
    pin_rope()


def test_rope_table_float64_source():
    cos, sin = ol.rope_tables(4096, 128, 1e6)
    assert cos.dtype == np.float32 and cos.shape == (4096, 64)
    ang = 4095 * 1e6 ** (-2 * 3 / 128)
    assert cos[4095, 3] == np.float32(math.cos(ang)) and sin[4095, 3] == np.float32(math.sin(ang))


def test_silu():
    from scipy.special import expit
    x = np.linspace(-30, 30, 1001)
    assert np.allclose(ol.silu(x), x * expit(x), rtol=1e-12, atol=1e-300)
    assert ol.silu(np.array([0.0]))[0] == 0.0
    assert abs(ol.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(ol.silu(np.array([-40.0]))[0]) < 1e-15


# ----------------------------------------------------------------------------
# attention: brute-force dense masked softmax (float64)
# ----------------------------------------------------------------------------
def pin_attention_dense(layer=ol, plan_mod=op):
    rng = np.random.default_rng(6)
    for (n_q, n_kv, d) in [(4, 2, 8), (4, 4, 16), (8, 1, 8)]:
        page = 16
        # two decodes with contexts 5 and 37, one prompt with 21 cached + chunk of 19
        seqs = {"d0": 5, "d1": 37, "p": 21}
        kv = {s: (rng.standard_normal((n + 20, n_kv, d)), rng.standard_normal((n + 20, n_kv, d)))
              for s, n in seqs.items()}
        num_pages = 64
        k_pool = np.zeros((num_pages, n_kv, page, d))
        v_pool = np.zeros_like(k_pool)
        perm = [int(v) for v in rng.permutation(num_pages)]
        pages = {}
        head = 0
        for s, n in seqs.items():
            m = wl.pages_for(n)
            pages[s] = perm[head:head + m]
            head += m
            for t in range(n):
                k_pool[pages[s][t // page], :, t % page] = kv[s][0][t]
                v_pool[pages[s][t // page], :, t % page] = kv[s][1][t]
        p = plan_mod.plan_batch([5, 37], [pages["d0"], pages["d1"]], [60], [21], [pages["p"]],
                                perm[head:], 2 + 19, 19)
        # write the new rows' K/V (positions ctx..) where the plan put them
        names = ["d0", "d1", "p"]
        for r in range(p.n_rows):
            s = names[p.row_seq[r]]
            pos = p.row_pos[r]
            sl = p.slot_mapping[r]
            k_pool[sl // page, :, sl % page] = kv[s][0][pos]
            v_pool[sl // page, :, sl % page] = kv[s][1][pos]
        q = rng.standard_normal((p.n_rows, n_q, d))
        got = layer.attention(q, k_pool, v_pool, p, n_q, n_kv, page, np.float64)
        # dense reference: full score matrix per sequence with an explicit mask
        for si, s in enumerate(names):
            rows = list(range(p.seq_q_start[si], p.seq_q_start[si + 1]))
            nk = p.seq_kv_len[si]
            Kd, Vd = kv[s][0][:nk], kv[s][1][:nk]
            for h in range(n_q):
                g = h // (n_q // n_kv)
                S = q[rows, h, :] @ Kd[:, g, :].T / math.sqrt(d)
                mask = np.array([[j <= p.row_pos[r] for j in range(nk)] for r in rows])
                S = np.where(mask, S, -np.inf)
                P = np.exp(S - S.max(axis=1, keepdims=True))
                P /= P.sum(axis=1, keepdims=True)
                exp = P @ Vd[:, g, :]
                assert np.allclose(got[rows, h, :], exp, rtol=1e-10, atol=1e-12), (n_q, n_kv, s, h)


def test_attention_dense():
    pin_attention_dense()


def test_attention_special_cases():
    # one key -> the output is that key's V; identical keys -> mean of V
    p = op.plan_batch([0], [[]], [], [], [], [3], 1, 1)
    k_pool = np.zeros((4, 1, 16, 8))
    v_pool = np.zeros_like(k_pool)
    v_pool[3, 0, 0] = np.arange(8)
    o = ol.attention(np.ones((1, 2, 8)), k_pool, v_pool, p, 2, 1, 16, np.float64)
    assert np.array_equal(o[0, 0], np.arange(8)) and np.array_equal(o[0, 1], np.arange(8))
    p = op.plan_batch([9], [[2]], [], [], [], [], 1, 1)
    k_pool[2, 0, :10] = 1.0
    v_pool[2, 0, :10] = np.arange(10)[:, None] * np.ones(8)
    o = ol.attention(np.ones((1, 1, 8)), k_pool, v_pool, p, 1, 1, 16, np.float64)
    assert np.allclose(o[0, 0], 4.5)


# ----------------------------------------------------------------------------
# layer: chunked == unchunked, decode batch independence, zero projections
# ----------------------------------------------------------------------------
def run_prompt_chunked(layer, dims, w, x_prompt, C, dtype, pool_pages=64, seed=0):
    L = x_prompt.shape[0]
    cos, sin = layer.rope_tables(L + 1, dims.d_head, dims.theta)
    shape = (pool_pages, dims.n_kv, dims.page, dims.d_head)
    k_pool, v_pool = np.zeros(shape, dtype), np.zeros(shape, dtype)
    pool = [int(v) for v in np.random.default_rng(seed).permutation(pool_pages)]
    done, pages, outs = 0, [], []
    while done < L:
        p = op.plan_batch([], [], [L], [done], [pages], pool, C, C, dims.page)
        pages, pool = p.pf_pages[0], p.free_pool
        xr = x_prompt[np.asarray(p.row_pos)]
        outs.append(layer.layer_forward(w, dims, p, xr, k_pool, v_pool, cos, sin, dtype))
        done += p.pf_take[0]
    return np.concatenate(outs), k_pool, v_pool


def pin_chunked_equals_unchunked(layer=ol, dtype=np.float32, tol=1e-5):
    rng = np.random.default_rng(7)
    dims = tiny_dims(d_model=64, d_ff=96)
    w = wl.layer_weights(rng, dims, gamma_jitter=0.1)
    L = 48
    x = wl.bf16_round(rng.standard_normal((L, dims.d_model), dtype=np.float32))
    ref, k_ref, v_ref = run_prompt_chunked(layer, dims, w, x, L, dtype)
    for C in [1, 7, 16, 48]:
        out, k, v = run_prompt_chunked(layer, dims, w, x, C, dtype)
        assert np.max(np.abs(out - ref)) <= tol, C
        assert np.max(np.abs(k - k_ref)) <= tol and np.max(np.abs(v - v_ref)) <= tol, C


def test_chunked_equals_unchunked_fp32():
    pin_chunked_equals_unchunked(dtype=np.float32, tol=1e-5)


def test_chunked_equals_unchunked_fp64():
    pin_chunked_equals_unchunked(dtype=np.float64, tol=1e-12)


def pin_decode_independence(layer=ol, dtype=np.float64, tol=1e-12):
    rng = np.random.default_rng(8)
    dims = tiny_dims()
    w = wl.layer_weights(rng, dims, gamma_jitter=0.1)
    st = tiny_state(rng, dims, [3, 16, 40, 70], [(60, 20)])
    cos, sin = layer.rope_tables(128, dims.d_head, dims.theta)
    xdec = rng.standard_normal((4, dims.d_model)).astype(np.float32)
    xch = rng.standard_normal((40, dims.d_model)).astype(np.float32)

    def run(order, with_chunk):
        dec = [st.decodes[i] for i in order]
        pfs = st.prefills if with_chunk else []
        p = op.plan_batch([r.done for r in dec], [r.pages for r in dec], [r.prompt_len for r in pfs],
                          [r.done for r in pfs], [r.pages for r in pfs], st.free_pool, 64, 64)
        x = np.concatenate([xdec[order], xch[:p.n_rows - len(order)]])
        k, v = st.k_pool.astype(dtype), st.v_pool.astype(dtype)
        out = layer.layer_forward(w, dims, p, x, k, v, cos, sin, dtype)
        return {i: out[j] for j, i in enumerate(order)}

    base = run([0, 1, 2, 3], True)
    for order, ch in [([2], False), ([3, 2, 1, 0], True), ([2, 0], False), ([1, 2], True)]:
        got = run(order, ch)
        for i in order:
            assert np.max(np.abs(got[i] - base[i])) <= tol, (order, ch, i)


def test_decode_independence():
    pin_decode_independence()


def test_zero_projections_identity():
    rng = np.random.default_rng(9)
    dims = tiny_dims()
    w = wl.layer_weights(rng, dims)
    w["w_o"] = np.zeros_like(w["w_o"])
    w["w_d"] = np.zeros_like(w["w_d"])
    st = tiny_state(rng, dims, [5, 9], [(30, 0)])
    p = plan_from_state(st, 20, 20)
    cos, sin = ol.rope_tables(64, dims.d_head, dims.theta)
    x = rng.standard_normal((p.n_rows, dims.d_model)).astype(np.float32)
    out = ol.layer_forward(w, dims, p, x, st.k_pool, st.v_pool, cos, sin)
    assert np.array_equal(out, x)


# ----------------------------------------------------------------------------
# the layer's assembly: which projection feeds which, in closed form
# ----------------------------------------------------------------------------
def assembly_case():
    """A hand-wired layer whose output and KV writes have closed forms.

    Tiny shapes (d 32, 4 q / 2 kv heads of 8 dims, d_ff 48); two decodes with
    contexts 1 and 3 over random cached K/V, plus the first 3 tokens of a
    fresh prompt.  Inputs are +-1, so every row of x has mean square 1.  The
    weights are zero except for single routes:
      * q head 3, dim 0     <- cq * xn[:, jq]      (the only non-zero query)
      * k head 0, dim 1     <- xn[:, jk]
      * v head 1, dim 2     <- xn[:, jv]
      * W_o a non-symmetric permutation (h[:, i] = x[:, i] + o[:, pi(i)])
      * gate row i0 <- alpha * hn[:, jg], up row i0 <- beta * hn[:, ju],
        down column i0 -> output column m with weight delta.
    The rows of W_qkv are ordered q heads, k heads, v heads, each head's
    d_head rows contiguous (the layout the weights are generated in)."""
    dims = tiny_dims()
    d, dh, nq, nkv, f = dims.d_model, dims.d_head, dims.n_q, dims.n_kv, dims.d_ff
    rng = np.random.default_rng(31)
    st = tiny_state(rng, dims, [1, 3], [(3, 0)], slack=8)
    p = plan_from_state(st, 8, 8)
    x = rng.choice([-1.0, 1.0], (p.n_rows, d)).astype(np.float32)
    g1 = (1 + 0.25 * rng.standard_normal(d)).astype(np.float32)
    g2 = (1 + 0.25 * rng.standard_normal(d)).astype(np.float32)
    c = dict(cq=2.0, jq=3, jk=11, jv=17, alpha=1.5, beta=-0.75, delta=2.0, jg=5, ju=23, i0=7, m=29, shift=5)
    w = dict(w_qkv=np.zeros((dims.qkv_cols, d), np.float32), w_o=np.zeros((d, nq * dh), np.float32),
             w_g=np.zeros((f, d), np.float32), w_u=np.zeros((f, d), np.float32),
             w_d=np.zeros((d, f), np.float32), g1=g1, g2=g2)
    w["w_qkv"][3 * dh + 0, c["jq"]] = c["cq"]
    w["w_qkv"][nq * dh + 0 * dh + 1, c["jk"]] = 1.0
    w["w_qkv"][(nq + nkv) * dh + 1 * dh + 2, c["jv"]] = 1.0
    for i in range(d):
        w["w_o"][i, (i + c["shift"]) % d] = 1.0
    w["w_g"][c["i0"], c["jg"]] = c["alpha"]
    w["w_u"][c["i0"], c["ju"]] = c["beta"]
    w["w_d"][c["m"], c["i0"]] = c["delta"]
    return dims, st, p, x, w, c


def assembly_expected(dims, st, p, x, w, c):
    """Closed forms of assembly_case, in float64, by scalar reasoning on the
    routes: the RMSNorm of a +-1 row is x g / sqrt(1 + eps); RoPE moves a
    lone component at dim e < d_head/2 to (e, e + d_head/2) with factors
    cos(pos theta^(-2e/d_head)), sin(...) (float64, held in float32); a zero query weights its keys
    uniformly; the only scored head is q head 3 over kv head 1."""
    dh, half, nq, nkv, eps = dims.d_head, dims.d_head // 2, dims.n_q, dims.n_kv, dims.eps
    T, d = x.shape
    x = x.astype(np.float64)
    xn = x / math.sqrt(1.0 + eps) * w["g1"].astype(np.float64)
    ang = lambda pos, e: pos * dims.theta ** (-2.0 * e / dh)
    # the rotation factors are computed in float64 and held in float32
    cosf = lambda a: np.cos(a).astype(np.float32).astype(np.float64)
    sinf = lambda a: np.sin(a).astype(np.float32).astype(np.float64)
    pos = np.asarray(p.row_pos)
    # new K/V rows of this iteration (rotated K), each [n_kv, d_head]
    k_new = np.zeros((T, nkv, dh))
    v_new = np.zeros((T, nkv, dh))
    k_new[:, 0, 1] = xn[:, c["jk"]] * cosf(ang(pos, 1))
    k_new[:, 0, 1 + half] = xn[:, c["jk"]] * sinf(ang(pos, 1))
    v_new[:, 1, 2] = xn[:, c["jv"]]
    q3 = np.zeros((T, dh))
    q3[:, 0] = c["cq"] * xn[:, c["jq"]] * cosf(ang(pos, 0))
    q3[:, half] = c["cq"] * xn[:, c["jq"]] * sinf(ang(pos, 0))
    o = np.zeros((T, nq, dh))
    for s in range(len(p.seq_pos0)):
        rows = list(range(p.seq_q_start[s], p.seq_q_start[s + 1]))
        n_cached = p.seq_pos0[s]
        Kc = ol.gather_keys(st.k_pool, p.block_table[s], n_cached, dims.page).astype(np.float64)
        Vc = ol.gather_keys(st.v_pool, p.block_table[s], n_cached, dims.page).astype(np.float64)
        Ks = np.concatenate([Kc, k_new[rows]])
        Vs = np.concatenate([Vc, v_new[rows]])
        for r in rows:
            n = pos[r] + 1
            for hq in range(nq):
                g = hq * nkv // nq
                if hq == 3:
                    sc = Ks[:n, g, :] @ q3[r] / math.sqrt(dh)
                    wts = np.exp(sc - sc.max())
                    wts /= wts.sum()
                else:
                    wts = np.full(n, 1.0 / n)
                o[r, hq] = wts @ Vs[:n, g, :]
    of_ = o.reshape(T, nq * dh)
    h = x + of_[:, (np.arange(d) + c["shift"]) % d]
    hn = h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps) * w["g2"].astype(np.float64)
    gate = c["alpha"] * hn[:, c["jg"]]
    up = c["beta"] * hn[:, c["ju"]]
    out = h.copy()
    out[:, c["m"]] += c["delta"] * gate * scipy_expit(gate) * up
    return out, k_new, v_new


def scipy_expit(z):
    from scipy.special import expit
    return expit(z)


def pin_layer_assembly(layer=ol):
    """The layer's wiring against closed forms: q/k/v column order and head
    layout, GQA groups, RoPE placement, the new token among a decode's keys,
    causal chunk rows, W_o orientation, residual sources, which gain feeds
    which norm, and gate versus up in the SwiGLU."""
    dims, st, p, x, w, c = assembly_case()
    cos, sin = layer.rope_tables(64, dims.d_head, dims.theta)
    k_pool, v_pool = st.k_pool.astype(np.float64), st.v_pool.astype(np.float64)
    got = layer.layer_forward(w, dims, p, x, k_pool, v_pool, cos, sin, np.float64)
    exp, k_new, v_new = assembly_expected(dims, st, p, x, w, c)
    np.testing.assert_allclose(got, exp, rtol=1e-12, atol=1e-12)
    # the decode rows see cached values, so the attention term is non-zero
    assert np.max(np.abs(exp - x)[: 2]) > 0.1
    page = dims.page
    for r, sl in enumerate(p.slot_mapping):
        np.testing.assert_allclose(k_pool[sl // page, :, sl % page, :], k_new[r], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(v_pool[sl // page, :, sl % page, :], v_new[r], rtol=1e-12, atol=1e-12)


def test_layer_assembly_closed_form():
    pin_layer_assembly()


# ----------------------------------------------------------------------------
# paged K/V store and the LM head
# ----------------------------------------------------------------------------
def pin_paged_store(mod=ol):
    """Tokens written through a scattered block table come back in order,
    bit for bit, and no other slot changes (16-token pages; the page and
    offset of a slot are slot // 16 and slot % 16)."""
    rng = np.random.default_rng(21)
    page, n_pages, n_kv, d = 16, 40, 2, 8
    k_pool = rng.standard_normal((n_pages, n_kv, page, d)).astype(np.float32)
    v_pool = rng.standard_normal((n_pages, n_kv, page, d)).astype(np.float32)
    k0, v0 = k_pool.copy(), v_pool.copy()
    for n in (1, 15, 16, 17, 100):
        table = rng.permutation(n_pages)[: (n + page - 1) // page]
        slots = np.array([table[t // page] * page + t % page for t in range(n)])
        k = rng.standard_normal((n, n_kv, d)).astype(np.float32)
        v = rng.standard_normal((n, n_kv, d)).astype(np.float32)
        kp, vp = k0.copy(), v0.copy()
        mod.kv_append(k, v, slots, kp, vp, page)
        assert np.array_equal(mod.gather_keys(kp, table, n, page), k)
        assert np.array_equal(mod.gather_keys(vp, table, n, page), v)
        touched = np.zeros(n_pages * page, bool)
        touched[slots] = True
        flat = lambda pool: pool.transpose(0, 2, 1, 3).reshape(n_pages * page, n_kv, d)
        assert np.array_equal(flat(kp)[~touched], flat(k0)[~touched])
        assert np.array_equal(flat(vp)[~touched], flat(v0)[~touched])


def pin_lm_head(mod=ol):
    """Closed forms of the final norm + untied head.  A one-hot row a e_j has
    mean square a^2/d, so its logits are a / sqrt(a^2/d + eps) g_j W[:, j];
    with W = I the head returns the normalised rows."""
    rng = np.random.default_rng(22)
    d, vocab, eps = 16, 24, 1e-6
    g = (1 + 0.1 * rng.standard_normal(d)).astype(np.float64)
    w = rng.standard_normal((vocab, d)).astype(np.float64)
    for j, a in [(0, 3.0), (5, -0.5), (15, 1e-2)]:
        x = np.zeros((1, d))
        x[0, j] = a
        got = mod.lm_head(x, g, w, eps, dtype=np.float64)
        exp = a / math.sqrt(a * a / d + eps) * g[j] * w[:, j]
        assert np.allclose(got[0], exp, rtol=1e-12, atol=0)
    x = rng.standard_normal((5, d))
    sq = rng.standard_normal((d, d))
    assert np.allclose(mod.lm_head(x, g, np.eye(d), eps, dtype=np.float64),
                       mod.rmsnorm(x, g, eps, dtype=np.float64), rtol=1e-13, atol=0)
    # a square, non-symmetric head tells W from its transpose
    exp = mod.rmsnorm(x, g, eps, dtype=np.float64) @ sq.T
    assert np.allclose(mod.lm_head(x, g, sq, eps, dtype=np.float64), exp, rtol=1e-12, atol=1e-12)
    assert not np.allclose(exp, mod.rmsnorm(x, g, eps, dtype=np.float64) @ sq, rtol=1e-3)


def test_paged_store():
    pin_paged_store()


def test_lm_head():
    pin_lm_head()


# ----------------------------------------------------------------------------
# planted mistakes: each pin must fail on a plausible wrong oracle
# ----------------------------------------------------------------------------
_ORIG_ATTENTION = ol.attention
_ORIG_ROPE = ol.rope


def _attention_variant(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype, kv_head, n_keys, round_p=None):
    """The oracle's attention loop with the head map and key count as parameters."""
    T, _, d_head = q.shape
    o = np.zeros((T, n_q, d_head), dtype)
    for s in range(len(plan.seq_pos0)):
        K = ol.gather_keys(k_pool, plan.block_table[s], plan.seq_kv_len[s], page).astype(dtype)
        V = ol.gather_keys(v_pool, plan.block_table[s], plan.seq_kv_len[s], page).astype(dtype)
        for r in range(plan.seq_q_start[s], plan.seq_q_start[s + 1]):
            nk = n_keys(plan, s, r)
            for h in range(n_q):
                g = kv_head(h, n_q, n_kv)
                sc = K[:nk, g, :] @ q[r, h, :] / np.sqrt(d_head)
                w = np.exp(sc - sc.max())
                o[r, h, :] = (w / w.sum()) @ V[:nk, g, :]
    return o


def _attn_gqa_modulo(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype=np.float32, round_p=None):
    return _attention_variant(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype,
                              lambda h, nq, nkv: h % nkv, lambda p, s, r: p.row_pos[r] + 1)


def _attn_excludes_self(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype=np.float32, round_p=None):
    return _attention_variant(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype,
                              lambda h, nq, nkv: h // (nq // nkv), lambda p, s, r: max(p.row_pos[r], 1))


def _attn_noncausal_chunk(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype=np.float32, round_p=None):
    return _attention_variant(q, k_pool, v_pool, plan, n_q, n_kv, page, dtype,
                              lambda h, nq, nkv: h // (nq // nkv), lambda p, s, r: p.seq_kv_len[s])


def _rope_wrong_sign(x, pos, cos, sin, dtype=np.float32):
    return _ORIG_ROPE(x, pos, cos, -np.asarray(sin), dtype)


def _rms_eps_outside(x, g, eps, dtype=np.float32):
    x = np.asarray(x, dtype)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * np.asarray(g, dtype)


def _gather_off_by_one(pool, table_row, n_keys, page):
    j = np.arange(n_keys)
    return pool[np.asarray(table_row)[j // page], :, (j + 1) % page, :]


def _lm_head_transposed(x_rows, g_f, w_lm, eps, dtype=np.float32):
    """The head applied as W instead of W^T wherever the shapes allow it."""
    w = np.asarray(w_lm, dtype)
    return ol.rmsnorm(x_rows, g_f, eps, dtype) @ (w if w.shape[0] == w.shape[1] else w.T)


@pytest.mark.parametrize("pin,name,mutant", [
    (pin_paged_store, "gather_keys", _gather_off_by_one),
    (pin_lm_head, "lm_head", _lm_head_transposed),
    (pin_attention_dense, "attention", _attn_gqa_modulo),
    (pin_attention_dense, "attention", _attn_excludes_self),
    (pin_attention_dense, "attention", _attn_noncausal_chunk),
    (pin_chunked_equals_unchunked, "attention", _attn_noncausal_chunk),
    (pin_rope, "rope", _rope_wrong_sign),
    (pin_rmsnorm, "rmsnorm", _rms_eps_outside),
])
def test_planted_mistakes_fail(monkeypatch, pin, name, mutant):
    monkeypatch.setattr(ol, name, mutant)
    with pytest.raises(AssertionError):
        pin()


def _layer_variant(mutation):
    """The oracle's layer assembly with one plausible wiring mistake."""
    def forward(w, dims, plan, x, k_pool, v_pool, cos, sin, dtype=np.float32, return_parts=False, storage=None):
        T = len(plan.row_seq)
        nq, nkv, dh = dims.n_q, dims.n_kv, dims.d_head
        x = np.asarray(x, dtype)
        xn = ol.rmsnorm(x, w["g1"], dims.eps, dtype)
        qkv = xn @ np.asarray(w["w_qkv"], dtype).T
        a0, a1 = nq * dh, (nq + nkv) * dh
        if mutation == "qkv order q, v, k":
            q, v, k = qkv[:, :a0], qkv[:, a0:a1], qkv[:, a1:]
        else:
            q, k, v = qkv[:, :a0], qkv[:, a0:a1], qkv[:, a1:]
        if mutation == "q heads interleaved by dim":
            q = q.reshape(T, dh, nq).transpose(0, 2, 1)
        q, k, v = q.reshape(T, nq, dh), k.reshape(T, nkv, dh), v.reshape(T, nkv, dh)
        pos = np.asarray(plan.row_pos)
        q, k = ol.rope(q, pos, cos, sin, dtype), ol.rope(k, pos, cos, sin, dtype)
        ol.kv_append(k, v, plan.slot_mapping, k_pool, v_pool, dims.page)
        o = ol.attention(q, k_pool, v_pool, plan, nq, nkv, dims.page, dtype).reshape(T, nq * dh)
        wo = np.asarray(w["w_o"], dtype)
        h = x + (o @ wo if mutation == "W_o transposed" else o @ wo.T)
        g2 = w["g1"] if mutation == "second norm with g1" else w["g2"]
        hn = ol.rmsnorm(x if mutation == "MLP norm of x" else h, g2, dims.eps, dtype)
        gate, up = hn @ np.asarray(w["w_g"], dtype).T, hn @ np.asarray(w["w_u"], dtype).T
        if mutation == "gate and up swapped":
            gate, up = up, gate
        a = ol.silu(gate) * up
        return (x if mutation == "final residual from x" else h) + a @ np.asarray(w["w_d"], dtype).T
    return forward


LAYER_MUTATIONS = ["gate and up swapped", "final residual from x", "qkv order q, v, k",
                   "q heads interleaved by dim", "W_o transposed", "second norm with g1", "MLP norm of x"]


def test_layer_variant_without_mutation_passes(monkeypatch):
    # the mutants differ from the oracle only in their named mistake
    monkeypatch.setattr(ol, "layer_forward", _layer_variant(None))
    pin_layer_assembly()


@pytest.mark.parametrize("mutation", LAYER_MUTATIONS)
def test_planted_layer_wiring_mistake_fails(monkeypatch, mutation):
    monkeypatch.setattr(ol, "layer_forward", _layer_variant(mutation))
    with pytest.raises(AssertionError):
        pin_layer_assembly()


def test_planted_planner_mistake_fails():
    # the pseudo-code read literally keeps peeking the head request, taking a
    # second chunk of R_A instead of moving on to R_B
    m = types.ModuleType("mutant_plan")

    def literal_peek(dec_ctx, dec_pages, pf_len, pf_done, pf_pages, free_pool, tau, chunk, page=16,
                     max_pages=None):
        return op.plan_batch(dec_ctx, dec_pages, pf_len, pf_done, pf_pages, free_pool, tau, tau, page,
                             max_pages)

    m.plan_batch = literal_peek
    with pytest.raises(AssertionError):
        pin_worked_example(plan_mod=m)


def test_planted_residual_mistake_fails(monkeypatch):
    orig = ol.layer_forward

    def no_residual(w, dims, plan, x, k_pool, v_pool, cos, sin, dtype=np.float32, return_parts=False):
        return orig(w, dims, plan, x, k_pool, v_pool, cos, sin, dtype) - 0.5 * np.asarray(x, dtype)

    monkeypatch.setattr(ol, "layer_forward", no_residual)
    with pytest.raises(AssertionError):
        test_zero_projections_identity()


# ----------------------------------------------------------------------------
# bf16-storage precision variant
# ----------------------------------------------------------------------------
def test_round_bf16_against_bit_definition():
    # bf16 keeps 7 mantissa bits: the grid spacing at 1.0 is 2^-7, ties go to
    # the even neighbour
    h = 2.0 ** -7
    x = np.array([1.0, 1 + h / 2, 1 + 3 * h / 2, 1 + h / 4, 1 + 3 * h / 4, -2.5, 65504.0, 0.0], np.float32)
    exp = np.array([1.0, 1.0, 1 + 2 * h, 1.0, 1 + h, -2.5, 65536.0, 0.0], np.float32)
    assert np.array_equal(ol.round_bf16(x), exp)
    # every output is representable (low 16 bits zero) and within half a spacing
    v = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    r = ol.round_bf16(v)
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
    assert np.all(np.abs(r - v) <= np.abs(v) * 2.0 ** -8)


def test_bf16_storage_variant_is_close_to_fp32_and_not_equal():
    rng = np.random.default_rng(10)
    dims = tiny_dims(d_model=64, d_ff=96)
    w = wl.layer_weights(rng, dims)
    st = tiny_state(rng, dims, [9, 30], [(40, 5)])
    p = plan_from_state(st, 30, 30)
    cos, sin = ol.rope_tables(64, dims.d_head, dims.theta)
    x = wl.bf16_round(rng.standard_normal((p.n_rows, dims.d_model), dtype=np.float32))
    a = ol.layer_forward(w, dims, p, x, st.k_pool.copy(), st.v_pool.copy(), cos, sin)
    b = ol.layer_forward(w, dims, p, x, st.k_pool.copy(), st.v_pool.copy(), cos, sin, storage="bf16")
    rl2 = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rl2 < 1e-2
    assert np.all((b.view(np.uint32) & 0xFFFF) == 0)


def test_bf16_storage_variant_without_rounding_is_the_layer(monkeypatch):
    """With rounding turned into the identity, the variant computes the same
    function as the plain layer: its folded norms are the identity
    RMSNorm(v; g) W^T = (v (W diag g)^T) / rms(v), so only the order of
    float64 operations differs."""
    rng = np.random.default_rng(12)
    dims = tiny_dims(d_model=64, d_ff=96)
    w = wl.layer_weights(rng, dims, gamma_jitter=0.2)
    st = tiny_state(rng, dims, [9, 30], [(40, 5)])
    p = plan_from_state(st, 30, 30)
    cos, sin = ol.rope_tables(64, dims.d_head, dims.theta)
    x = rng.standard_normal((p.n_rows, dims.d_model))
    f64 = np.float64
    a = ol.layer_forward(w, dims, p, x, st.k_pool.astype(f64), st.v_pool.astype(f64), cos, sin, f64)
    monkeypatch.setattr(ol, "round_bf16", lambda t: np.asarray(t, f64))
    b = ol.layer_forward(w, dims, p, x, st.k_pool.astype(f64), st.v_pool.astype(f64), cos, sin, f64,
                         storage="bf16")
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- iteration driver
def _run_loop(loop, arrivals, max_iters=10_000):
    """arrivals: {iteration: [(prompt_len, max_new), ...]}; returns per-iteration (plan, row_req)."""
    hist = []
    it = 0
    while it < max_iters:
        for pl, mn in arrivals.get(it, []):
            loop.add(pl, mn)
        if loop.active() == 0 and it > max(arrivals, default=0):
            break
        p, rr = loop.plan()
        hist.append((p, rr))
        loop.commit()
        it += 1
    return hist


def test_sched_loop_single_request_closed_form():
    """A lone request: ceil(L / C) prefill iterations (C <= tau), then one
    decode iteration per further token; positions 0..L + max_new - 2 each
    processed once, in order."""
    import oracle.sched as osch
    for L, mn, C, tau in [(100, 3, 48, 64), (16, 1, 16, 16), (33, 5, 8, 8), (200, 10, 64, 512)]:
        loop = osch.SchedLoop(tau, C, list(range(100)))
        hist = _run_loop(loop, {0: [(L, mn)]})
        assert len(hist) == -(-L // min(C, tau)) + mn - 1
        pos = [q for p, rr in hist for q in p.row_pos]
        assert pos == list(range(L + mn - 1))
        r = loop.reqs[0]
        assert r["state"] == osch.FINISHED and r["generated"] == mn and r["cached"] == L + mn - 1
        assert sorted(loop.pool) == list(range(100))


def test_sched_loop_conservation_and_pages():
    """Random streams: every request is finished with max_new tokens, each
    cached position is processed exactly once, no page is ever held twice,
    and every page returns to the pool."""
    import oracle.sched as osch
    rng = np.random.default_rng(11)
    for trial in range(25):
        tau = int(rng.integers(8, 200))
        C = int(rng.integers(4, 2 * tau))
        n_pages = 400
        loop = osch.SchedLoop(tau, C, list(rng.permutation(n_pages)))
        arrivals = {}
        for _ in range(int(rng.integers(1, 9))):
            arrivals.setdefault(int(rng.integers(0, 12)), []).append((int(rng.integers(1, 120)),
                                                                      int(rng.integers(1, 9))))
        seen = {}
        it = 0
        while True:
            for pl, mn in arrivals.get(it, []):
                loop.add(pl, mn)
            if loop.active() == 0 and it > max(arrivals):
                break
            p, rr = loop.plan()
            assert p.n_rows <= tau or p.over_budget
            for q, req in zip(p.row_pos, rr):
                assert (req, q) not in seen
                seen[(req, q)] = it
            loop.commit()
            held = [pg for r in loop.reqs for pg in r["pages"]]
            assert len(set(held)) == len(held) and not set(held) & set(loop.pool)
            assert len(held) + len(loop.pool) == n_pages
            it += 1
        for i, r in enumerate(loop.reqs):
            assert r["state"] == osch.FINISHED and r["generated"] == r["max_new"]
            assert sorted(q for (req, q) in seen if req == i) == list(range(r["prompt_len"] + r["max_new"] - 1))
            # a position is processed only after all earlier positions of its request
            its = [seen[(i, q)] for q in range(r["prompt_len"] + r["max_new"] - 1)]
            assert its == sorted(its)
        assert len(loop.pool) == n_pages


def test_sched_loop_matches_replay_on_tiny_streams():
    """Brute force on tiny streams: replaying the definition by hand --
    decodes first in completion order, then FIFO chunks of min(C, rest,
    budget left) -- gives the same row sets per iteration."""
    import oracle.sched as osch
    rng = np.random.default_rng(12)
    for trial in range(60):
        tau, C = int(rng.integers(2, 12)), int(rng.integers(1, 12))
        reqs = [(int(rng.integers(1, 14)), int(rng.integers(1, 5))) for _ in range(int(rng.integers(1, 5)))]
        loop = osch.SchedLoop(tau, C, list(range(64)))
        for pl, mn in reqs:
            loop.add(pl, mn)
        # replay
        state = [dict(pl=pl, mn=mn, cached=0, gen=0) for pl, mn in reqs]
        waiting = list(range(len(reqs)))
        running = []
        while waiting or running:
            p, rr = loop.plan()
            want = [(i, state[i]["cached"]) for i in running]
            n = len(running)
            takes = {}
            for i in waiting:
                t = max(0, min(C, state[i]["pl"] - state[i]["cached"], tau - n))
                if t:
                    takes[i] = t
                    want += [(i, state[i]["cached"] + k) for k in range(t)]
                    n += t
            assert list(zip(rr, p.row_pos)) == want
            loop.commit()
            nrun = []
            for i in running:
                state[i]["cached"] += 1
                state[i]["gen"] += 1
                if state[i]["gen"] < state[i]["mn"]:
                    nrun.append(i)
            nwait = []
            for i in waiting:
                state[i]["cached"] += takes.get(i, 0)
                if state[i]["cached"] < state[i]["pl"]:
                    nwait.append(i)
                elif state[i]["mn"] > 1:
                    state[i]["gen"] = 1
                    nrun.append(i)
            running, waiting = nrun, nwait
