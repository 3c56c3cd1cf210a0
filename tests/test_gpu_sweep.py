"""Chunk-equivalence and token-budget points on the Mistral-7B-shaped layer (GPU).

* A prompt prefilled in chunks of C with the KV cache carried between
  iterations gives the same outputs and KV as unchunked prefill
  (Sarathi-Serve reading notes, sections 3.1 and 7.5b): on the GPU every stage
  is computed per row in an order that does not depend on the batch, so the
  results are compared bit for bit at 32768 tokens, and against the oracle
  at 2048 tokens.
* Token-budget points of the sweep (b = 64 decodes with contexts uniform in
  [512, 8192], c = tau - 64 at offset 0) against the full oracle.
"""
import numpy as np
import pytest

import oracle.layer as ol
import oracle.plan as op
import workloads as wl
from workloads import device as wd
from tests.gpu_harness import GpuLayer, assert_close, assert_layer, oracle_layer_both, plan_both

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402


def prefill_in_chunks(lw, dims, x, C, rope, max_pos, num_pages, seed):
    """Run a prompt through the layer in chunks of C; returns (out, k, v)."""
    L = x.shape[0]
    shape = (num_pages, dims.n_kv, 16, dims.d_head)
    k = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.empty_like(x)
    pool = [int(p) for p in np.random.default_rng(seed).permutation(num_pages)]
    done, pages = 0, []
    ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, C, 1, L))
    while done < L:
        hp = hb.hb_plan_batch([], [], [L], [done], [pages], pool, C, C)
        pages, pool = hp.pf_pages[0], hp.free_pool
        dp = hb.DevicePlan(hp)
        t = int(hp.pf_take[0])
        hb.hb_layer_forward(lw, dims, dp, rope, max_pos, x[done:done + t], out[done:done + t], k, v, L, ws)
        done += t
    hb.hb_check_status()
    return out, k, v, pages


def test_chunked_equals_unchunked_32k_bitwise():
    dims = wl.MISTRAL
    L = 32768
    gen = wd.device_generator(41)
    lw = wd.layer_weights_random(dims, 4100)
    x = wd.randn_bf16((L, dims.d_model), gen)
    rope = wd.rope_table_device(L + 1, dims)
    num_pages = L // 16 + 8
    ref, kr, vr, pr = prefill_in_chunks(lw, dims, x, L, rope, L + 1, num_pages, seed=5)
    for C in [512, 1024, 2048]:
        out, k, v, pg = prefill_in_chunks(lw, dims, x, C, rope, L + 1, num_pages, seed=5)
        assert pg == pr  # same page sequence: pages popped in position order either way
        assert torch.equal(out, ref), f"C={C}: outputs differ (max {float((out.float() - ref.float()).abs().max())})"
        assert torch.equal(k, kr) and torch.equal(v, vr), f"C={C}: KV differs"
    assert torch.isfinite(ref.float()).all()


def test_chunked_prefill_2048_against_oracle():
    rng = np.random.default_rng(6)
    dims = wl.MISTRAL
    w = wl.layer_weights(rng, dims)
    L, C = 2048, 512
    xp = wl.activations(rng, L, dims.d_model)
    st = wl.make_state(rng, dims, [], [(L, 0)], slack_pages=L // 16 + 4)
    gl = GpuLayer(w, dims, st.k_pool, st.v_pool, L + 1)
    p32 = (st.k_pool.copy(), st.v_pool.copy())
    p16 = (st.k_pool.copy(), st.v_pool.copy())
    outs, refs, emus, hs = [], [], [], []
    while st.prefills[0].done < L:
        hp, o = plan_both(st, C, C)
        xr = xp[np.asarray(hp.row_pos)]
        outs.append(gl.forward(hp, xr, L))
        ref, emu, h = oracle_layer_both(w, dims, o, xr, p32, p16, L + 1)
        refs.append(ref)
        emus.append(emu)
        hs.append(h)
        st.prefills[0].pages = list(hp.pf_pages[0])
        st.prefills[0].done += int(hp.pf_take[0])
        st.free_pool = list(hp.free_pool)
    assert_layer(np.concatenate(outs), np.concatenate(refs), np.concatenate(emus), np.concatenate(hs),
                 "chunked prefill 2048 / 512")
    sl = np.concatenate([[pg * 16 + t for t in range(16)] for pg in st.prefills[0].pages])[:L]
    kg = wd.to_numpy(gl.k)
    assert_close(kg[sl // 16, :, sl % 16], p16[0][sl // 16, :, sl % 16], "chunked prefill K cache")


@pytest.mark.parametrize("tau", [64, 1024, 2048, 4096])
def test_tau_sweep_point_against_oracle(tau):
    w = wl.mistral_layer(seed=7, tau=tau, n_dec=64, ctx_lo=512, ctx_hi=8192, prompt_len=8192, offset=0)
    st, dims = w.state, w.dims
    hp, o = plan_both(st, tau, tau)
    assert hp.n_rows == tau and (tau > 64 or hp.n_seqs == 64)
    max_pos = 8192 + tau + 1
    gl = GpuLayer(w.weights[0], dims, st.k_pool, st.v_pool, max_pos)
    got = gl.forward(hp, w.x, int(hp.seq_kv_len.max()))
    ref, emu, h = oracle_layer_both(w.weights[0], dims, o, w.x, (st.k_pool.copy(), st.v_pool.copy()),
                                 (st.k_pool.copy(), st.v_pool.copy()), max_pos)
    assert_layer(got, ref, emu, h, f"tau={tau} layer output")
