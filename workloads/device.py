"""Staging of the seeded inputs on the device (torch tensors) and back.

Input preparation only: bf16 bit patterns are moved as they are, weights are
interleaved and the RoPE table filled by the library's own set-up calls.
"""
from __future__ import annotations

import numpy as np

from . import to_bf16_bits


def bf16_tensor(x: np.ndarray, device="cuda"):
    import torch
    bits = to_bf16_bits(np.asarray(x, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def to_numpy(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return t.detach().float().cpu().numpy()


def layer_weights_device(w: dict, dims, device="cuda", fmt="bf16"):
    """Upload one layer's weights and prepare them with the library (gains
    folded, gate/up interleaved; fmt="e4m3": then quantized per row)."""
    import chunked_prefill_hybrid_tau_gb300 as hb
    return hb.prepare_layer_weights(*[bf16_tensor(w[k], device) for k in ("w_qkv", "w_o", "w_g", "w_u", "w_d",
                                                                          "g1", "g2")], fmt=fmt)


def rope_table_device(max_pos: int, dims, device="cuda"):
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    t = torch.empty((max_pos, dims.d_head // 2, 2), dtype=torch.float32, device=device)
    hb.hb_rope_table(t, max_pos, dims.d_head, dims.theta)
    return t


def workspace(nbytes: int, device="cuda"):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- device-side generation
# Model-scale inputs (tens of GB) are drawn on the device with torch's seeded
# Philox generator, directly in bf16 (the draw is rounded to bf16 once); the
# oracle side reads back exactly the tensors it needs.
def device_generator(seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, gen, scale=1.0, device="cuda"):
    import torch
    t = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if scale != 1.0:
        t.mul_(scale)
    return t.to(torch.bfloat16)


def _layer_draws(dims, seed, device):
    """The layer's tensors in a fixed draw order from its own seed."""
    gen = device_generator(seed, device)
    d, f = dims.d_model, dims.d_ff
    w_qkv = randn_bf16((dims.qkv_cols, d), gen, 0.02, device)
    w_o = randn_bf16((d, dims.n_q * dims.d_head), gen, 0.02, device)
    w_g = randn_bf16((f, d), gen, 0.02, device)
    w_u = randn_bf16((f, d), gen, 0.02, device)
    w_d = randn_bf16((d, f), gen, 0.02, device)
    return w_qkv, w_o, w_g, w_u, w_d


def layer_weights_random(dims, seed, device="cuda", fmt="bf16"):
    """One layer's weights on the device from `seed`: N(0, 0.02) projections,
    gains 1, prepared by the library (fmt as in layer_weights_device)."""
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    w_qkv, w_o, w_g, w_u, w_d = _layer_draws(dims, seed, device)
    ones = torch.ones(dims.d_model, dtype=torch.bfloat16, device=device)
    return hb.prepare_layer_weights(w_qkv, w_o, w_g, w_u, w_d, ones, ones, fmt=fmt)


def host_layer_weights(dims, seed, device="cuda") -> dict:
    """The oracle's view of layer `seed` (float32 arrays of the same bf16
    draws, regenerated from the seed)."""
    w_qkv, w_o, w_g, w_u, w_d = _layer_draws(dims, seed, device)
    ones = np.ones(dims.d_model, np.float32)
    return dict(w_qkv=to_numpy(w_qkv), w_o=to_numpy(w_o), w_g=to_numpy(w_g), w_u=to_numpy(w_u), w_d=to_numpy(w_d),
                g1=ones, g2=ones.copy())
