"""The layer stack of one iteration through hb_layers_forward against the
same layers through hb_layer_forward one call at a time (GPU).

In the stack a bf16 layer after the first takes the row statistics of its
input from the previous layer's down projection instead of the statistics
kernel; both form every 32-column part and the row sum in the same order, so
outputs and KV caches must agree bit for bit.  Cases: the Mistral-7B-shaped
hybrid batch at tau = 512 (CTA-pair GEMM tiles, split-K O and down
projections), the tiny layer (one-CTA tiles, no split K), and a stack mixing
bf16 and E4M3 layers (an E4M3 down projection hands its statistics to a
bf16 layer)."""
import numpy as np
import pytest

import workloads as wl
from workloads import device as wd

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402


def stack_vs_calls(dims, dec_ctx, prompt_len, done, tau, formats, seed):
    rng = np.random.default_rng(seed)
    st = wl.make_state(rng, dims, [int(c) for c in dec_ctx], [(prompt_len, done)],
                       slack_pages=wl.pages_for(tau) + len(dec_ctx) + 8, fill_kv=False)
    hp = hb.hb_plan_batch([r.done for r in st.decodes], [r.pages for r in st.decodes], [prompt_len], [done],
                          [st.prefills[0].pages], st.free_pool, tau, tau)
    T = hp.n_rows
    assert T == tau
    gen = wd.device_generator(seed)
    max_kv = int(hp.seq_kv_len.max())
    rope = wd.rope_table_device(max_kv + 1, dims)
    x = wd.randn_bf16((T, dims.d_model), gen)
    dp = hb.DevicePlan(hp)
    ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, T, hp.n_seqs, max_kv))
    shape = (st.num_pages, dims.n_kv, 16, dims.d_head)
    layers = [wd.layer_weights_random(dims, seed * 100 + l, fmt=f) for l, f in enumerate(formats)]
    pools = [(wd.randn_bf16(shape, gen), wd.randn_bf16(shape, gen)) for _ in formats]

    # one call per layer, in place; each launches the kernels the library's rule says
    x1 = x.clone()
    p1 = [(k.clone(), v.clone()) for k, v in pools]
    per_layer = [hb.hb_layer_kernel_count(dims, T, 1 if f == "e4m3" else 0) for f in formats]
    for l, lw in enumerate(layers):
        n0 = hb.hb_kernel_launches()
        hb.hb_layer_forward(lw, dims, dp, rope, max_kv + 1, x1, x1, p1[l][0], p1[l][1], max_kv, ws)
        assert hb.hb_kernel_launches() - n0 == per_layer[l], f"layer {l}"
    hb.hb_check_status()
    # the stack, out of place (layer 0 reads x, every layer writes x2): a bf16
    # layer after the first launches no statistics kernel
    x2 = torch.full_like(x, float("nan"))
    p2 = [(k.clone(), v.clone()) for k, v in pools]
    n0 = hb.hb_kernel_launches()
    hb.hb_layers_forward(layers, dims, dp, rope, max_kv + 1, x, x2, [k for k, _ in p2], [v for _, v in p2], max_kv,
                         ws)
    carried = sum(1 for l, f in enumerate(formats) if l > 0 and f == "bf16")
    assert hb.hb_kernel_launches() - n0 == sum(per_layer) - carried
    hb.hb_check_status()
    assert torch.isfinite(x1.float()).all()
    assert torch.equal(x1, x2), f"outputs differ (max {float((x1.float() - x2.float()).abs().max())})"
    for l in range(len(formats)):
        assert torch.equal(p1[l][0], p2[l][0]) and torch.equal(p1[l][1], p2[l][1]), f"layer {l}: KV differs"
    # and in place, x_out aliasing x_in
    x3 = x.clone()
    p3 = [(k.clone(), v.clone()) for k, v in pools]
    hb.hb_layers_forward(layers, dims, dp, rope, max_kv + 1, x3, x3, [k for k, _ in p3], [v for _, v in p3], max_kv,
                         ws)
    hb.hb_check_status()
    assert torch.equal(x1, x3)
    del layers, pools, p1, p2, p3
    torch.cuda.empty_cache()


def test_stack_equals_layer_calls_mistral_tau512():
    rng = np.random.default_rng(3)
    dec_ctx = rng.integers(512, 4097, size=32)
    stack_vs_calls(wl.MISTRAL, dec_ctx, 4096, 1024, 512, ["bf16"] * 4, seed=11)


def test_stack_equals_layer_calls_tiny():
    stack_vs_calls(wl.TINY, [32, 77, 150, 200], 256, 128, 68, ["bf16"] * 3, seed=12)


def test_stack_equals_layer_calls_mixed_formats():
    rng = np.random.default_rng(4)
    dec_ctx = rng.integers(512, 4097, size=32)
    stack_vs_calls(wl.MISTRAL, dec_ctx, 4096, 1024, 512, ["bf16", "e4m3", "bf16", "e4m3"], seed=13)


def test_stack_equals_layer_calls_unfused_e4m3():
    """3 q heads and 1 kv head of 64 dims: 320 QKV columns, not whole
    256-column tiles, so E4M3 layers run the separate RoPE/KV append
    (11 kernels) and bf16 layers between them take carried statistics."""
    import dataclasses
    dims = dataclasses.replace(wl.TINY, n_q=3, n_kv=1, d_ff=256)
    stack_vs_calls(dims, [40, 90, 300], 256, 64, 67, ["e4m3", "bf16", "e4m3", "bf16"], seed=14)
