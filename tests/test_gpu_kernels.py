"""Kernel-level parity: each CUDA entry point against the oracle's step on the
same seeded inputs (GPU required)."""
import numpy as np
import pytest

import oracle.layer as ol
import workloads as wl
from workloads import device as wd
from tests.gpu_harness import assert_close, plan_both

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402
from chunked_prefill_hybrid_tau_gb300 import _lib as L  # noqa: E402


def test_device_is_sm103():
    n, ok = hb.hb_device_info()
    assert ok and n > 100


def test_rope_table_matches_oracle():
    for max_pos, d, theta in [(4096, 128, 1e6), (512, 64, 1e4), (16384, 128, 5e6)]:
        dims = wl.Dims(d_model=256, n_q=2, n_kv=1, d_head=d, d_ff=64, theta=theta)
        t = wd.to_numpy(wd.rope_table_device(max_pos, dims))
        cos, sin = ol.rope_tables(max_pos, d, theta)
        ulp_c = np.abs(t[..., 0] - cos) / np.spacing(np.abs(cos).astype(np.float32) + np.float32(1e-30))
        ulp_s = np.abs(t[..., 1] - sin) / np.spacing(np.abs(sin).astype(np.float32) + np.float32(1e-30))
        assert ulp_c.max() <= 1 and ulp_s.max() <= 1
        assert np.mean(t[..., 0] == cos) > 0.999 and np.mean(t[..., 1] == sin) > 0.999


def test_gemm_swiglu_padded_ffn():
    """F = 688 (not a multiple of 64): the interleave pads gate/up to 704 rows
    of zeros and the padded output columns are silu(0) * 0 = 0."""
    rng = np.random.default_rng(688)
    M, K, F = 68, 256, 688
    Fp = 704
    A = wl.bf16_round(rng.standard_normal((M, K), dtype=np.float32))
    Wg = wl.bf16_round(rng.standard_normal((F, K), dtype=np.float32) * np.float32(0.02))
    Wu = wl.bf16_round(rng.standard_normal((F, K), dtype=np.float32) * np.float32(0.02))
    Wgu = torch.full((2 * Fp, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    hb.hb_interleave_gate_up(wd.bf16_tensor(Wg), wd.bf16_tensor(Wu), Wgu)
    out = torch.empty((M, Fp), dtype=torch.bfloat16, device="cuda")
    hb.hb_gemm(wd.bf16_tensor(A), Wgu, out, None, L.HB_EPI_SWIGLU)
    hb.hb_check_status()
    got = wd.to_numpy(out)
    assert_close(got[:, :F], ol.silu(A @ Wg.T) * (A @ Wu.T), "swiglu padded")
    assert np.all(got[:, F:] == 0)


@pytest.mark.parametrize("rows,d", [(1, 256), (77, 4096), (300, 7168)])
def test_rmsnorm(rows, d):
    rng = np.random.default_rng(rows)
    x = wl.bf16_round(rng.standard_normal((rows, d), dtype=np.float32) * 3)
    g = wl.bf16_round(1 + 0.1 * rng.standard_normal(d, dtype=np.float32))
    xt, gt = wd.bf16_tensor(x), wd.bf16_tensor(g)
    y = torch.empty_like(xt)
    hb.hb_rmsnorm(xt, gt, y, 1e-6)
    hb.hb_check_status()
    assert_close(wd.to_numpy(y), ol.rmsnorm(x, g, 1e-6), "rmsnorm")


GEMM_CASES = [
    (1, 128, 64, L.HB_EPI_STORE),
    (68, 512, 256, L.HB_EPI_STORE),
    (200, 6144, 512, L.HB_EPI_STORE),        # 192-wide tiles
    (128, 25600, 128, L.HB_EPI_STORE),       # 256-wide tiles
    (333, 1024, 640, L.HB_EPI_STORE),        # ragged M
    (512, 4096, 4096, L.HB_EPI_RESIDUAL),
    (512, 4096, 14336, L.HB_EPI_RESIDUAL),
    (70, 768, 192, L.HB_EPI_RESIDUAL),
    (300, 1024, 384, L.HB_EPI_SWIGLU),
    (128, 25600, 256, L.HB_EPI_SWIGLU),      # 256-wide tiles
    (512, 28672, 4096, L.HB_EPI_SWIGLU),
    (333, 4096, 8192, L.HB_EPI_RESIDUAL),   # split K on CTA pairs, odd number of 128-row tiles
    (65, 32000, 4096, L.HB_EPI_F32),
    (3, 640, 128, L.HB_EPI_F32),
    (68, 200, 688, L.HB_EPI_STORE),          # K and N not multiples of 64 / 32
    (68, 256, 688, L.HB_EPI_RESIDUAL),
    (5, 1000, 72, L.HB_EPI_F32),
]


@pytest.mark.parametrize("M,N,K,epi", GEMM_CASES)
def test_gemm(M, N, K, epi):
    rng = np.random.default_rng(M * 7 + N + K)
    A = wl.bf16_round(rng.standard_normal((M, K), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    At = wd.bf16_tensor(A)
    if epi == L.HB_EPI_SWIGLU:
        F = N // 2
        Wg, Wu = W[:F], W[F:]
        Wgu = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        hb.hb_interleave_gate_up(wd.bf16_tensor(Wg), wd.bf16_tensor(Wu), Wgu)
        out = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
        hb.hb_gemm(At, Wgu, out, None, epi)
        ref = ol.silu(A @ Wg.T) * (A @ Wu.T)
    elif epi == L.HB_EPI_F32:
        out = torch.empty((M, N), dtype=torch.float32, device="cuda")
        hb.hb_gemm(At, wd.bf16_tensor(W), out, None, epi)
        ref = A @ W.T
    elif epi == L.HB_EPI_RESIDUAL:
        R = wl.bf16_round(rng.standard_normal((M, N), dtype=np.float32))
        out = wd.bf16_tensor(R)  # residual added in place (R aliases C)
        hb.hb_gemm(At, wd.bf16_tensor(W), out, out, epi)
        ref = R + A @ W.T
    else:
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        hb.hb_gemm(At, wd.bf16_tensor(W), out, None, epi)
        ref = A @ W.T
    hb.hb_check_status()
    got = wd.to_numpy(out)
    if epi == L.HB_EPI_F32:
        assert_close(got, ref, "gemm f32", atol=1e-3, rtol=1e-3, rel_l2=1e-4)
    else:
        assert_close(got, ref, f"gemm epi={epi}")


@pytest.mark.parametrize("N,K,epi", [(1024, 512, L.HB_EPI_SWIGLU), (28672, 4096, L.HB_EPI_SWIGLU),
                                     (4096, 8192, L.HB_EPI_RESIDUAL), (4096, 4096, L.HB_EPI_RESIDUAL),
                                     (6144, 4096, L.HB_EPI_STORE), (512, 256, L.HB_EPI_STORE)])
def test_gemm_pair_tiles_match_single_cta_tiles_bitwise(N, K, epi):
    """Projections with more than one 128-row tile run on 256 x 256 CTA-pair
    tiles, a single 128-row tile on one CTA: a row's result must not depend on
    which, so 128 rows computed alone equal the same rows computed inside a
    512-row batch bit for bit."""
    rng = np.random.default_rng(N + K)
    A = wl.bf16_round(rng.standard_normal((512, K), dtype=np.float32))
    W = wl.bf16_round(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    Wt = wd.bf16_tensor(W)
    if epi == L.HB_EPI_SWIGLU:
        Wgu = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        hb.hb_interleave_gate_up(wd.bf16_tensor(W[:N // 2]), wd.bf16_tensor(W[N // 2:]), Wgu)
        Wt = Wgu
    cols = N // 2 if epi == L.HB_EPI_SWIGLU else N
    R = wl.bf16_round(rng.standard_normal((512, cols), dtype=np.float32))
    outs = []
    for M in (512, 128):
        At = wd.bf16_tensor(A[:M])
        out = wd.bf16_tensor(R[:M]) if epi == L.HB_EPI_RESIDUAL else torch.empty((M, cols), dtype=torch.bfloat16,
                                                                                  device="cuda")
        hb.hb_gemm(At, Wt, out, out if epi == L.HB_EPI_RESIDUAL else None, epi)
        hb.hb_check_status()
        outs.append(out[:128])
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("n_q,n_kv,d_head", [(8, 2, 128), (4, 2, 64), (14, 2, 128)])
def test_kv_append(n_q, n_kv, d_head):
    rng = np.random.default_rng(n_q + d_head)
    dims = wl.Dims(d_model=256, n_q=n_q, n_kv=n_kv, d_head=d_head, d_ff=64, theta=1e6)
    T, num_pages, max_pos = 50, 40, 2048
    qkv = wl.bf16_round(rng.standard_normal((T, dims.qkv_cols), dtype=np.float32))
    pos = rng.integers(0, max_pos, T).astype(np.int32)
    slots = rng.permutation(num_pages * 16)[:T].astype(np.int32)
    slots[7] = -1  # padding row: q is rotated, nothing is written to the cache
    k0 = wl.bf16_round(rng.standard_normal((num_pages, n_kv, 16, d_head), dtype=np.float32))
    v0 = wl.bf16_round(rng.standard_normal((num_pages, n_kv, 16, d_head), dtype=np.float32))
    kt, vt = wd.bf16_tensor(k0), wd.bf16_tensor(v0)
    q_out = torch.empty((T, n_q, d_head), dtype=torch.bfloat16, device="cuda")
    rope = wd.rope_table_device(max_pos, dims)
    hb.hb_kv_append(wd.bf16_tensor(qkv), torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(), rope, max_pos,
                    dims, q_out, kt, vt)
    hb.hb_check_status()
    cos, sin = ol.rope_tables(max_pos, d_head, dims.theta)
    q = qkv[:, :n_q * d_head].reshape(T, n_q, d_head)
    k = qkv[:, n_q * d_head:(n_q + n_kv) * d_head].reshape(T, n_kv, d_head)
    v = qkv[:, (n_q + n_kv) * d_head:].reshape(T, n_kv, d_head)
    assert_close(wd.to_numpy(q_out), ol.rope(q, pos, cos, sin), "rotated q", atol=1e-2, rtol=1e-2)
    kr = ol.rope(k, pos, cos, sin)
    kexp, vexp = k0.copy(), v0.copy()
    keep = slots >= 0
    ol.kv_append(kr[keep], v[keep], slots[keep], kexp, vexp, 16)
    kg, vg = wd.to_numpy(kt), wd.to_numpy(vt)
    assert_close(kg, kexp, "k cache", atol=1e-2, rtol=1e-2)
    assert np.array_equal(vg, vexp)  # v is copied bit for bit, other slots untouched
    untouched = np.ones(num_pages * 16, bool)
    untouched[slots[keep]] = False
    assert np.array_equal(kg.transpose(0, 2, 1, 3).reshape(-1, n_kv, d_head)[untouched],
                          k0.transpose(0, 2, 1, 3).reshape(-1, n_kv, d_head)[untouched])


def attention_case(dims, dec_ctx, prefills, tau, chunk, seed, poison=True):
    """Random q and cache through hb_attention and the oracle.  Every unused
    slot of the GPU cache holds NaN, which the kernel must never let reach
    an output."""
    rng = np.random.default_rng(seed)
    st = wl.make_state(rng, dims, dec_ctx, prefills, slack_pages=64)
    hp, o = plan_both(st, tau, chunk)
    # values of this iteration's new tokens
    for sl in hp.slot_mapping:
        st.k_pool[sl // 16, :, sl % 16] = wl.bf16_round(rng.standard_normal((dims.n_kv, dims.d_head), dtype=np.float32))
        st.v_pool[sl // 16, :, sl % 16] = wl.bf16_round(rng.standard_normal((dims.n_kv, dims.d_head), dtype=np.float32))
    kg, vg = st.k_pool.copy(), st.v_pool.copy()
    if poison:
        used = np.zeros(st.num_pages * 16, bool)
        for r in st.decodes + st.prefills:
            for t in range(r.done):
                used[r.pages[t // 16] * 16 + t % 16] = True
        used[hp.slot_mapping] = True
        flat_k = kg.transpose(0, 2, 1, 3).reshape(-1, dims.n_kv, dims.d_head)
        flat_v = vg.transpose(0, 2, 1, 3).reshape(-1, dims.n_kv, dims.d_head)
        flat_k[~used] = np.nan
        flat_v[~used] = np.nan
        kg = flat_k.reshape(st.num_pages, 16, dims.n_kv, dims.d_head).transpose(0, 2, 1, 3).copy()
        vg = flat_v.reshape(st.num_pages, 16, dims.n_kv, dims.d_head).transpose(0, 2, 1, 3).copy()
    q = wl.bf16_round(rng.standard_normal((hp.n_rows, dims.n_q, dims.d_head), dtype=np.float32))
    max_kv = int(hp.seq_kv_len.max())
    dp = hb.DevicePlan(hp)
    out = torch.empty((hp.n_rows, dims.n_q * dims.d_head), dtype=torch.bfloat16, device="cuda")
    ws = wd.workspace(hb.hb_attention_workspace_bytes(dims, hp.n_rows, hp.n_seqs, max_kv))
    hb.hb_attention(wd.bf16_tensor(q), wd.bf16_tensor(kg), wd.bf16_tensor(vg), dp, dims, max_kv, out, ws)
    hb.hb_check_status()
    ref = ol.attention(q, st.k_pool, st.v_pool, o, dims.n_q, dims.n_kv, 16).reshape(hp.n_rows, -1)
    return wd.to_numpy(out), ref, hp


# decode contexts at page edges (16 keys) and at the 1024-key split edges: a
# decode row's kv_len is its context + 1, so 1023 fills one split exactly,
# 1024 leaves a one-key last split and 3072 a one-key fourth split
DEC_CTX = [0, 1, 15, 16, 17, 63, 64, 511, 512, 513, 1023, 1024, 1500, 2047, 3072]


# (8, 2, 128), (32, 8, 128), (6, 3, 128): chunk rows on CTA pairs (an even number
# of q heads per kv head; 6 q heads = 3 head pairs); (14, 2, 128) odd group and
# (4, 2, 64) d_head 64: one CTA per unit
@pytest.mark.parametrize("n_q,n_kv,d_head", [(8, 2, 128), (14, 2, 128), (4, 2, 64), (32, 8, 128), (6, 3, 128)])
def test_attention_hybrid(n_q, n_kv, d_head):
    dims = wl.Dims(d_model=256, n_q=n_q, n_kv=n_kv, d_head=d_head, d_ff=64)
    got, ref, hp = attention_case(dims, DEC_CTX, [(600, 100)], len(DEC_CTX) + 130, 130, seed=n_q + d_head)
    assert hp.n_rows == len(DEC_CTX) + 130
    assert_close(got, ref, f"attention {n_q}/{n_kv}/{d_head}")


def test_attention_chunk_only_from_zero():
    dims = wl.Dims(d_model=256, n_q=8, n_kv=2, d_head=128, d_ff=64)
    got, ref, _ = attention_case(dims, [], [(1000, 0)], 200, 200, seed=3)
    assert_close(got, ref, "attention chunk from position 0")


def test_attention_several_chunks_and_one_token_chunk():
    dims = wl.Dims(d_model=256, n_q=8, n_kv=2, d_head=128, d_ff=64)
    # three prompts; budget leaves a 1-token chunk for the last one
    got, ref, hp = attention_case(dims, [40, 700], [(300, 50), (90, 0), (500, 499)], 2 + 100 + 90 + 1, 100, seed=4)
    assert list(hp.pf_take) == [100, 90, 1]
    assert_close(got, ref, "attention multi-chunk")


def test_attention_decode_batch_invariance():
    """A decode row's output is bit-identical whatever shares its batch."""
    dims = wl.Dims(d_model=256, n_q=8, n_kv=2, d_head=128, d_ff=64)
    rng = np.random.default_rng(5)
    st = wl.make_state(rng, dims, [100, 1300, 2100], [(800, 300)], slack_pages=64)
    q_all = wl.bf16_round(rng.standard_normal((3 + 200, dims.n_q, dims.d_head), dtype=np.float32))
    kt, vt = wd.bf16_tensor(st.k_pool), wd.bf16_tensor(st.v_pool)

    def run(dec_idx, with_chunk):
        dec = [st.decodes[i] for i in dec_idx]
        pfs = st.prefills if with_chunk else []
        hp = hb.hb_plan_batch([r.done for r in dec], [r.pages for r in dec], [r.prompt_len for r in pfs],
                              [r.done for r in pfs], [r.pages for r in pfs], st.free_pool, 256, 200)
        q = np.concatenate([q_all[dec_idx], q_all[3:3 + hp.n_rows - len(dec_idx)]])
        dp = hb.DevicePlan(hp)
        out = torch.empty((hp.n_rows, dims.n_q * dims.d_head), dtype=torch.bfloat16, device="cuda")
        ws = wd.workspace(hb.hb_attention_workspace_bytes(dims, hp.n_rows, hp.n_seqs, 4096))
        hb.hb_attention(wd.bf16_tensor(q), kt, vt, dp, dims, 4096, out, ws)
        hb.hb_check_status()
        o = wd.to_numpy(out)
        return {i: o[j] for j, i in enumerate(dec_idx)}

    base = run([0, 1, 2], True)
    for idx, ch in [([2], False), ([2, 1, 0], True), ([1], True), ([0, 2], False)]:
        got = run(idx, ch)
        for i in idx:
            assert np.array_equal(got[i], base[i]), (idx, ch, i)


def test_attention_sm_split_never_changes_results():
    """The plan's scheduling hints only move chunk and decode work between
    SMs: real hints, none (the two paths one after the other), and hints
    that push the split to either extreme give bit-identical outputs, which
    match the oracle."""
    dims = wl.Dims(d_model=256, n_q=32, n_kv=8, d_head=128, d_ff=64)
    rng = np.random.default_rng(8)
    st = wl.make_state(rng, dims, [5, 300, 1500, 2900, 700, 64], [(1500, 900), (400, 0)], slack_pages=64)
    hp, o = plan_both(st, 6 + 300, 256)
    assert hp.chunk_pairs > 0 and hp.decode_pairs > 0 and hp.chunk_rows == 300
    q = wl.bf16_round(rng.standard_normal((hp.n_rows, dims.n_q, dims.d_head), dtype=np.float32))
    qt, kt, vt = wd.bf16_tensor(q), wd.bf16_tensor(st.k_pool), wd.bf16_tensor(st.v_pool)
    max_kv = int(hp.seq_kv_len.max())
    ws = wd.workspace(hb.hb_attention_workspace_bytes(dims, hp.n_rows, hp.n_seqs, max_kv))
    dp = hb.DevicePlan(hp)
    outs = []
    for hints in [dp.hints, (0, 0, 0), (1, 10**12, 300), (10**12, 1, 300)]:
        dp.hints = hints
        out = torch.empty((hp.n_rows, dims.n_q * dims.d_head), dtype=torch.bfloat16, device="cuda")
        hb.hb_attention(qt, kt, vt, dp, dims, max_kv, out, ws)
        hb.hb_check_status()
        outs.append(out)
    for k in range(1, len(outs)):
        assert torch.equal(outs[k], outs[0]), k
    ref = ol.attention(q, st.k_pool, st.v_pool, o, dims.n_q, dims.n_kv, 16).reshape(hp.n_rows, -1)
    assert_close(wd.to_numpy(outs[0]), ref, "attention with an SM split")


def test_status_word_reports_bad_slot():
    dims = wl.Dims(d_model=256, n_q=4, n_kv=2, d_head=64, d_ff=64)
    qkv = torch.zeros((2, dims.qkv_cols), dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 10**6], dtype=torch.int32, device="cuda")  # second slot beyond the pool
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    q_out = torch.empty((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    rope = wd.rope_table_device(16, dims)
    hb.hb_kv_append(qkv, pos, slots, rope, 16, dims, q_out, kc, vc)
    with pytest.raises(hb.HBError) as e:
        hb.hb_check_status()
    assert e.value.status == L.HB_ERR_DEVICE
    hb.hb_check_status()  # cleared
