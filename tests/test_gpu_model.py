"""Model-level parity: the 32-layer Mistral-7B-shaped model with its LM head
(tau = 2048, layer by layer through hb_layer_forward) and the 60-layer
Yi-34B-shaped model (tau = 1024, the whole stack in one hb_layers_forward
call), the logits through hb_final_logits (GPU).

The oracle follows sampled decode rows through every layer from the original
inputs: a decode row's output depends only on its own hidden state and its
own KV (prior context + its new token), so the chunk rows, which the CPU
could not afford through every layer, are not needed for it.  For the
32-layer model, layers 0, 1 and 31 are also compared on every row (all 64
decode rows and the 1984 chunk rows), each fed the GPU's actual input to that
layer and its KV pools as they were before it, at the single-layer bounds.
The last chunk row's logits are compared with the oracle's final norm and LM
head applied to that row's final GPU hidden state.

Tolerance of a deep stack: the random-weight stack amplifies any per-layer
rounding, so the bound is derived from the arithmetic itself: the oracle is
run twice, in fp32 and with bf16 storage at the GPU's storage points
(storage="bf16"), and the GPU must be no farther from fp32 than 1.5x the
relative L2 distance and 2x the largest element deviation that bf16 storage
alone produces.  (Measured: 32 layers 3.1% GPU vs 3.1% emulation, 60 layers
4.6% vs 4.6%; a wrong head, row or projection is orders of magnitude
larger.)"""
import numpy as np
import pytest

import oracle.layer as ol
import oracle.plan as op
import workloads as wl
from workloads import device as wd
from tests.gpu_harness import assert_close, assert_layer

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402


def run_model(dims, tau, dec_ctx, prompt_len, sample, vocab, seed, full_layers=()):
    """full_layers: layers whose every row (decode and chunk) is compared with
    the oracle run on the GPU's own input to that layer and the layer's KV
    pools as they were before it."""
    rng = np.random.default_rng(seed)
    st = wl.make_state(rng, dims, [int(c) for c in dec_ctx], [(prompt_len, 0)],
                       slack_pages=wl.pages_for(tau) + len(dec_ctx) + 8, fill_kv=False)
    plan_args = ([r.done for r in st.decodes], [r.pages for r in st.decodes], [prompt_len], [0], [[]],
                 st.free_pool, tau, tau)
    hp = hb.hb_plan_batch(*plan_args)
    T = hp.n_rows
    n_dec = len(dec_ctx)
    assert T == tau and list(hp.pf_take) == [tau - n_dec]
    gen = wd.device_generator(seed)
    max_kv = int(hp.seq_kv_len.max())
    rope = wd.rope_table_device(max_kv + 1, dims)
    x = wd.randn_bf16((T, dims.d_model), gen)
    x_rows0 = wd.to_numpy(x[sample])
    dp = hb.DevicePlan(hp)
    ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, T, hp.n_seqs, max_kv))
    shape = (st.num_pages, dims.n_kv, 16, dims.d_head)
    layers, pools = [], []
    for l in range(dims.n_layers):
        layers.append(wd.layer_weights_random(dims, seed * 1000 + l))
        pools.append((wd.randn_bf16(shape, gen), wd.randn_bf16(shape, gen)))
    # the oracle's copy of the sampled rows' prior KV (before the GPU appends)
    sample_pages = sorted({pg for i in sample for pg in hp.dec_pages[i]})
    remap = {pg: k for k, pg in enumerate(sample_pages)}
    idx = torch.tensor(sample_pages, device="cuda")
    host_kv = [(wd.to_numpy(k[idx]), wd.to_numpy(v[idx])) for k, v in pools]
    full = {}
    if full_layers:
        for l in range(dims.n_layers):
            k, v = pools[l]
            if l in full_layers:
                full[l] = [wd.to_numpy(x), wd.to_numpy(k), wd.to_numpy(v)]
            hb.hb_layer_forward(layers[l], dims, dp, rope, max_kv + 1, x, x, k, v, max_kv, ws)
            if l in full_layers:
                full[l].append(wd.to_numpy(x))
    else:  # the whole stack in one call
        hb.hb_layers_forward(layers, dims, dp, rope, max_kv + 1, x, x, [k for k, _ in pools], [v for _, v in pools],
                             max_kv, ws)
    hb.hb_check_status()
    rows = torch.tensor(list(range(n_dec)) + [T - 1], dtype=torch.int32, device="cuda")
    logits = None
    if vocab:
        g_f = torch.ones(dims.d_model, dtype=torch.bfloat16, device="cuda")
        w_lm = wd.randn_bf16((vocab, dims.d_model), gen, 0.02)
        logits = torch.empty((rows.numel(), vocab), dtype=torch.float32, device="cuda")
        lws = wd.workspace(rows.numel() * dims.d_model * 2)
        hb.hb_final_logits(x, rows, g_f, w_lm, logits, lws, dims.eps)
        hb.hb_check_status()
    gpu_rows = wd.to_numpy(x[sample])

    # oracle: the sampled decode rows through every layer
    sub_pages = [[remap[pg] for pg in hp.dec_pages[i]] for i in sample]
    o_plan = op.plan_batch([int(dec_ctx[i]) for i in sample], sub_pages, [], [], [], [], len(sample), 1)
    cos, sin = ol.rope_tables(max_kv + 1, dims.d_head, dims.theta)
    xr, xe = x_rows0, x_rows0
    for l in range(dims.n_layers):
        w = wd.host_layer_weights(dims, seed * 1000 + l)
        kk, vv = host_kv[l]
        xr = ol.layer_forward(w, dims, o_plan, xr, kk.copy(), vv.copy(), cos, sin)
        xe = ol.layer_forward(w, dims, o_plan, xe, kk.copy(), vv.copy(), cos, sin, storage="bf16")

    def rl2(a, b):
        return float(np.linalg.norm(a - b) / np.linalg.norm(b))

    def check_stack(gpu, fp32, emu, what):
        assert np.all(np.isfinite(gpu)), what
        g, e = rl2(gpu, fp32), rl2(emu, fp32)
        gmax, emax = float(np.abs(gpu - fp32).max()), float(np.abs(emu - fp32).max())
        print(f"\n{what}: relL2 gpu/fp32 {g:.4g} emulation/fp32 {e:.4g} gpu/emulation {rl2(gpu, emu):.4g}; "
              f"max abs gpu {gmax:.4g} emulation {emax:.4g}")
        assert g <= max(1e-2, 1.5 * e), f"{what}: relative L2 {g:.4g} beyond 1.5 x bf16-storage {e:.4g}"
        assert gmax <= max(2e-2, 2.0 * emax), f"{what}: max abs {gmax:.4g} beyond 2 x bf16-storage {emax:.4g}"

    check_stack(gpu_rows, xr, xe, f"{dims.n_layers}-layer hidden state of sampled decode rows")
    if full_layers:
        # every row of the chosen layers (the chunk rows included), each layer
        # fed its actual GPU input and KV pools
        o_full = op.plan_batch(*plan_args, max_pages=hp.max_pages)
        for l in full_layers:
            x_in, kp, vp, x_out = full[l]
            w = wd.host_layer_weights(dims, seed * 1000 + l)
            ref = ol.layer_forward(w, dims, o_full, x_in, kp.copy(), vp.copy(), cos, sin)
            emu, parts = ol.layer_forward(w, dims, o_full, x_in, kp, vp, cos, sin, storage="bf16", return_parts=True)
            assert_layer(x_out, ref, emu, parts["h"], f"layer {l}, all {T} rows")
    if vocab:
        g_f_h = np.ones(dims.d_model, np.float32)
        w_lm_h = wd.to_numpy(w_lm)
        ref = ol.lm_head(xr, g_f_h, w_lm_h, dims.eps)
        emu = ol.lm_head(xe, g_f_h, w_lm_h, dims.eps)
        got = wd.to_numpy(logits)
        check_stack(got[sample], ref, emu, "logits of sampled decode rows")
        # the last chunk row: the final norm and LM head on its final GPU
        # hidden state (its path through the layers is covered by the
        # full-layer comparisons); the GPU rounds the normed row to bf16
        x_last = wd.to_numpy(x[T - 1:T])
        ref_c = ol.lm_head(x_last, g_f_h, w_lm_h, dims.eps)
        emu_c = ol.round_bf16(ol.rmsnorm(x_last, g_f_h, dims.eps)) @ w_lm_h.T
        check_stack(got[-1:], ref_c, emu_c, "logits of the last chunk row (final norm + LM head)")
    del layers, pools
    torch.cuda.empty_cache()


def test_mistral_32_layers_lm_head_tau2048():
    rng = np.random.default_rng(2)
    ctx = rng.integers(1024, 8192, size=64, endpoint=True)
    run_model(wl.MISTRAL_32L, 2048, ctx, 8192, sample=[0, 21, 63], vocab=32000, seed=2,
              full_layers=(0, 1, wl.MISTRAL_32L.n_layers - 1))


def test_yi34b_60_layers_tau1024():
    rng = np.random.default_rng(3)
    ctx = wl.log_uniform_ints(rng, 256, 16384, 128)
    run_model(wl.YI34B, 1024, ctx, 16384, sample=[int(np.argmin(ctx)), 64, int(np.argmax(ctx))], vocab=0, seed=3)
