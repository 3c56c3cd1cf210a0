"""Pins of the FP8 (E4M3) oracle against the format's definition, a library
conversion, exact rational arithmetic and properties of per-row scaling.

Each pin takes the oracle module so that the planted-mistake tests at the
bottom can run it against a mutated copy and check that it fails.  Nothing
here touches the CUDA library.
"""
import types
from fractions import Fraction

import numpy as np
import pytest

import oracle.fp8 as of
import oracle.layer as ol
import oracle.plan as op
import workloads as wl

torch = pytest.importorskip("torch")


def torch_e4m3(v):
    """torch's float8_e4m3fn conversion (round to nearest even; no saturation,
    so only |v| <= 464 is compared): -> (codes, values)."""
    t = torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy(), t.float().numpy().astype(np.float64)


# ----------------------------------------------------------------------------
# the format
# ----------------------------------------------------------------------------
def pin_table(m=of):
    t = m.e4m3_table()
    assert t[0x00] == 0 and not np.signbit(t[0x00])
    assert t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9  # subnormals
    assert t[0x08] == 2.0 ** -6                                # smallest normal
    assert t[0x38] == 1.0 and t[0x39] == 1.125 and t[0x40] == 2.0
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.sum(np.isfinite(t)) == 254
    pos = t[:127]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(t[128:255], -pos)
    # every value is a multiple of 2^-9 with at most 4 significant bits
    k = pos * 2 ** 9
    assert np.all(k == np.round(k))
    # the library's decoding of the 256 bit patterns
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    fin = np.isfinite(t)
    assert np.array_equal(np.isnan(lib), ~fin) and np.array_equal(lib[fin], t[fin])


def pin_round_against_library(m=of):
    t = m.e4m3_table()[:127]
    mids = (t[1:] + t[:-1]) / 2                       # ties: decided by the even code
    f32 = np.float32
    near = np.concatenate([np.nextafter(mids.astype(f32), f32(0)), np.nextafter(mids.astype(f32), f32(1e9))])
    rng = np.random.default_rng(5)
    rnd = np.exp2(rng.uniform(-14, np.log2(464), 20000)) * rng.choice([-1, 1], 20000)
    v = np.concatenate([t, mids, near, rnd, -t, -mids, [464.0, -464.0, 2.0 ** -10, -(2.0 ** -10)]]).astype(f32)
    v = v[np.abs(v) <= 464]
    codes, vals = torch_e4m3(v)
    assert np.array_equal(m.e4m3_round(v), vals)
    assert np.array_equal(m.e4m3_encode(v), codes)


def pin_saturation(m=of):
    v = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    r = m.e4m3_round(v)
    assert np.array_equal(r, [448, 448, 448, 448, 448, 448, 448, -448, -448])
    c = m.e4m3_encode(np.array([np.nan, -0.0, 0.0, -1e-9], np.float32))
    assert c[0] & 0x7F == 0x7F and c[1] == 0x80 and c[2] == 0x00 and c[3] == 0x80


# ----------------------------------------------------------------------------
# per-row scaling
# ----------------------------------------------------------------------------
def pin_quantize_rows(m=of):
    rng = np.random.default_rng(7)
    x = wl.bf16_round(rng.standard_normal((64, 300)).astype(np.float32) * np.exp2(rng.uniform(-6, 6, (64, 1))))
    x[5] = 0.0
    x[9, :] = 0.0
    x[9, 17] = -3.0                                   # a row with one nonzero
    q, s = m.quantize_rows(x)
    assert q.dtype == np.uint8 and s.dtype == np.float32
    amax = np.max(np.abs(x), axis=1)
    # the row maximum lands on +-448 exactly; the scale is amax / 448 in fp32
    arg = np.argmax(np.abs(x), axis=1)
    nz = amax > 0
    assert np.all(np.abs(m.e4m3_decode(q[np.arange(64), arg]))[nz] == 448.0)
    assert np.array_equal(s, np.where(nz, amax / np.float32(448), 0).astype(np.float32))
    assert s[5] == 0 and np.all(q[5] == 0)
    assert np.count_nonzero(q[9] & 0x7F) == 1 and q[9, 17] == 0xFE
    # the error bound of round-to-nearest with 3 mantissa bits: half a step,
    # 2^-4 of the value for normals, 2^-10 for subnormals (times the scale)
    err = np.abs(m.dequantize_rows(q, s) - x)
    bound = (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)
    # scaling a row by a power of two keeps its codes and scales its scale
    q2, s2 = m.quantize_rows(x * np.float32(2.0 ** 5))
    assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(2.0 ** 5))
    # rows are independent: a row's codes do not depend on the other rows
    q3, s3 = m.quantize_rows(x[10:11])
    assert np.array_equal(q3[0], q[10]) and s3[0] == s[10]


def pin_gemm_exact(m=of):
    rng = np.random.default_rng(11)
    M, N, K = 5, 7, 33
    qa = rng.integers(0, 255, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 255, (N, K), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x38                    # no NaN codes
    qb[(qb & 0x7F) == 0x7F] = 0xB8
    sa = np.float32(2.0) ** rng.integers(-3, 3, M).astype(np.float32)
    sb = np.float32(2.0) ** rng.integers(-3, 3, N).astype(np.float32)
    tab = m.e4m3_table()
    got = m.gemm(qa, sa, qb, sb)
    for i in range(M):
        for j in range(N):
            ref = sum(Fraction(float(tab[qa[i, k]])) * Fraction(float(tab[qb[j, k]])) for k in range(K))
            assert Fraction(float(got[i, j])) == ref * Fraction(float(sa[i])) * Fraction(float(sb[j]))


# ----------------------------------------------------------------------------
# the FP8 layer
# ----------------------------------------------------------------------------
def small_case(seed=3):
    dims = wl.Dims(d_model=64, n_q=4, n_kv=2, d_head=16, d_ff=96, theta=1e4)
    rng = np.random.default_rng(seed)
    w = wl.layer_weights(rng, dims, gamma_jitter=0.1)
    st = wl.make_state(rng, dims, [5, 19, 40], [(50, 16)], slack_pages=32)
    p = op.plan_batch([r.done for r in st.decodes], [r.pages for r in st.decodes],
                      [r.prompt_len for r in st.prefills], [r.done for r in st.prefills],
                      [r.pages for r in st.prefills], st.free_pool, 64, 64, dims.page)
    x = wl.activations(rng, p.n_rows, dims.d_model)
    return dims, w, st, p, x


def pin_layer_near_bf16_layer(m=of):
    dims, w, st, p, x = small_case()
    cos, sin = ol.rope_tables(256, dims.d_head, dims.theta)
    ref = ol.layer_forward(w, dims, p, x, st.k_pool.copy(), st.v_pool.copy(), cos, sin)
    got = m.layer_forward(m.prepare_weights(w), dims, p, x, st.k_pool.copy(), st.v_pool.copy(), cos, sin)
    delta = ref - x  # the layer's own contribution; the residual is carried exactly
    rl2 = np.linalg.norm(got - ref) / np.linalg.norm(delta)
    # E4M3 keeps 3 mantissa bits: per-element errors up to 2^-4, random in
    # sign, so a few percent of the layer's contribution, and never zero
    assert 0.003 < rl2 < 0.08, rl2


def pin_layer_qkv_exact_when_representable(m=of):
    """Inputs whose rows are already E4M3 values scaled so that amax = 448 * 2^k
    quantize without error: the FP8 QKV projection then equals the fp32 one."""
    dims, w, st, p, _ = small_case()
    rng = np.random.default_rng(4)
    tab = m.e4m3_table()[:127]

    def representable(rows, cols, k):
        v = rng.choice(tab, (rows, cols)) * rng.choice([-1.0, 1.0], (rows, cols))
        v[:, 0] = 448.0
        return (v * 2.0 ** k).astype(np.float32)

    w = dict(w, g1=np.ones(dims.d_model, np.float32), w_qkv=representable(dims.qkv_cols, dims.d_model, -12))
    x = representable(p.n_rows, dims.d_model, -8)
    cos, sin = ol.rope_tables(256, dims.d_head, dims.theta)
    f64 = np.float64
    _, ref = ol.layer_forward(w, dims, p, x, st.k_pool.copy(), st.v_pool.copy(), cos, sin, dtype=f64,
                              return_parts=True)
    _, got = m.layer_forward(m.prepare_weights(w), dims, p, x, st.k_pool.copy(), st.v_pool.copy(), cos, sin,
                             dtype=f64, return_parts=True)
    np.testing.assert_allclose(got["qkv"], ref["qkv"], rtol=1e-12, atol=1e-14)


def pin_layer_chunk_invariant(m=of):
    """Per-row scales: the same rows give the same outputs whether their
    prompt runs as one chunk or several."""
    dims = wl.Dims(d_model=64, n_q=4, n_kv=2, d_head=16, d_ff=96, theta=1e4)
    rng = np.random.default_rng(8)
    wq = m.prepare_weights(wl.layer_weights(rng, dims, gamma_jitter=0.1))
    L = 48
    x = wl.activations(rng, L, dims.d_model)
    cos, sin = ol.rope_tables(64, dims.d_head, dims.theta)
    n_pages = 8

    def run(chunk):
        kp = np.zeros((n_pages, dims.n_kv, dims.page, dims.d_head), np.float32)
        vp = np.zeros_like(kp)
        pages, done, outs = [], 0, []
        pool = list(range(n_pages))
        while done < L:
            p = op.plan_batch([], [], [L], [done], [pages], pool, chunk, chunk, dims.page)
            outs.append(m.layer_forward(wq, dims, p, x[done:done + p.n_rows], kp, vp, cos, sin))
            pages, pool, done = list(p.pf_pages[0]), list(p.free_pool), done + p.n_rows
        return np.concatenate(outs)

    one = run(L)
    for c in (7, 16):
        np.testing.assert_allclose(run(c), one, rtol=1e-5, atol=1e-6)


def pin_layer_assembly(m=of):
    """The FP8 layer's wiring against the closed forms of the hand-wired
    layer in test_oracle_pins (single routes through each projection).  Its
    weights and the +-1 inputs are exact in E4M3; the per-token codes of o
    and h carry up to half an E4M3 step (2^-4 relative) each, so the layer's
    contribution may move by a few percent, while a swapped gate/up or a
    residual taken from x moves it by 20% or more."""
    import test_oracle_pins as tp
    dims, st, p, x, w, c = tp.assembly_case()
    w = dict(w, g1=ol.round_bf16(w["g1"]), g2=ol.round_bf16(w["g2"]))
    exp, k_new, v_new = tp.assembly_expected(dims, st, p, x, w, c)
    cos, sin = ol.rope_tables(64, dims.d_head, dims.theta)
    k_pool, v_pool = st.k_pool.astype(np.float64), st.v_pool.astype(np.float64)
    got = m.layer_forward(m.prepare_weights(w), dims, p, x, k_pool, v_pool, cos, sin, dtype=np.float64)
    contrib = exp - x
    assert np.linalg.norm(got - exp) <= 0.06 * np.linalg.norm(contrib)
    assert np.max(np.abs(got - exp)[:, c["m"]]) <= 0.1 * np.max(np.abs(contrib[:, c["m"]]))
    # K and V come from exact codes of x: rotated K and V land exactly
    page = dims.page
    for r, sl in enumerate(p.slot_mapping):
        np.testing.assert_allclose(k_pool[sl // page, :, sl % page, :], k_new[r], rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(v_pool[sl // page, :, sl % page, :], v_new[r], rtol=1e-6, atol=1e-7)


PINS = [pin_table, pin_round_against_library, pin_saturation, pin_quantize_rows, pin_gemm_exact,
        pin_layer_near_bf16_layer, pin_layer_qkv_exact_when_representable, pin_layer_chunk_invariant,
        pin_layer_assembly]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_fp8_oracle_pin(pin):
    pin()


# ----------------------------------------------------------------------------
# planted mistakes: each mutation of the oracle must fail at least one pin
# ----------------------------------------------------------------------------
def mutated(**over):
    m = types.ModuleType("fp8_mut")
    m.__dict__.update({k: v for k, v in of.__dict__.items() if not k.startswith("__")})
    m.__dict__.update(over)
    return m


def _round_truncating(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(np.isfinite(a), a, 1.0))
    step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / step) * step, 448.0), v)


def _round_half_up(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(np.isfinite(a), a, 1.0))
    step = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 448.0), v)


def _quant_per_tensor(x):
    x = np.asarray(x, np.float32)
    amax = np.float32(np.max(np.abs(x)))
    inv = np.float32(448) / amax
    return of.e4m3_encode((x * inv).astype(np.float32)), np.full(x.shape[0], amax / np.float32(448), np.float32)


def _gemm_dropped_scale(qa, sa, qb, sb):
    return (of.e4m3_decode(qa) @ of.e4m3_decode(qb).T) * np.asarray(sa, np.float64)[:, None]


def _table_no_subnormals():
    t = of.e4m3_table().copy()
    c = np.arange(256)
    E, M = (c >> 3) & 15, c & 7
    sub = (E == 0) & (M > 0)
    t[sub] = np.where(c[sub] >> 7, -1.0, 1.0) * (8.0 + M[sub]) * 2.0 ** -10   # as if E were 1
    return t


def _fp8_layer_variant(mutation):
    """The FP8 oracle's layer with one wiring mistake (names resolve in the
    mutated module, like the oracle's own functions)."""
    def layer_forward(wq, dims, plan, x, k_pool, v_pool, cos, sin, storage=None, dtype=np.float32,
                      return_parts=False):
        T = len(plan.row_seq)
        nq, nkv, dh = dims.n_q, dims.n_kv, dims.d_head

        def inv_rms(v):
            v = np.asarray(v, dtype)
            return 1.0 / np.sqrt(np.mean(v * v, axis=-1) + dtype(dims.eps))

        def proj(v, name):
            qa, sa = of.quantize_rows(v)
            qb, sb = wq[name]
            return of.gemm(qa, sa, qb, sb).astype(dtype)

        x = np.asarray(x, dtype)
        qkv = inv_rms(x)[:, None] * proj(x, "qkv")
        q = qkv[:, :nq * dh].reshape(T, nq, dh)
        k = qkv[:, nq * dh:(nq + nkv) * dh].reshape(T, nkv, dh)
        v = qkv[:, (nq + nkv) * dh:].reshape(T, nkv, dh)
        pos = np.asarray(plan.row_pos)
        q, k = ol.rope(q, pos, cos, sin, dtype), ol.rope(k, pos, cos, sin, dtype)
        ol.kv_append(k, v, plan.slot_mapping, k_pool, v_pool, dims.page)
        o = ol.attention(q, k_pool, v_pool, plan, nq, nkv, dims.page, dtype)
        h = x + proj(o.reshape(T, nq * dh), "o")
        r = inv_rms(h)[:, None]
        gate, up = r * proj(h, "g"), r * proj(h, "u")
        if mutation == "gate and up swapped":
            gate, up = up, gate
        a = ol.silu(gate) * up
        out = (x if mutation == "final residual from x" else h) + proj(a, "d")
        return (out, dict(qkv=qkv, o=o, h=h, a=a)) if return_parts else out
    return layer_forward


MUTATIONS = {
    "truncating round": dict(e4m3_round=_round_truncating),
    "round half up": dict(e4m3_round=_round_half_up),
    "per-tensor scale": dict(quantize_rows=_quant_per_tensor),
    "dropped weight scale": dict(gemm=_gemm_dropped_scale),
    "subnormals decoded as normals": dict(e4m3_table=_table_no_subnormals),
    "layer: gate and up swapped": dict(layer_forward=_fp8_layer_variant("gate and up swapped")),
    "layer: final residual from x": dict(layer_forward=_fp8_layer_variant("final residual from x")),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_fp8_mistake_is_caught(name):
    m = mutated(**MUTATIONS[name])
    # functions that call module globals must see the mutated ones
    for fn in ("e4m3_encode", "e4m3_decode", "quantize_rows", "dequantize_rows", "gemm", "prepare_weights",
               "layer_forward"):
        f = of.__dict__[fn]
        m.__dict__[fn] = types.FunctionType(f.__code__, m.__dict__, fn, f.__defaults__, f.__closure__) \
            if fn not in MUTATIONS[name] else m.__dict__[fn]
    m._POS = m.e4m3_table()[:127]
    failed = 0
    for pin in PINS:
        try:
            pin(m)
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake: {name}"
