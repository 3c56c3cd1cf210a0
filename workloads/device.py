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


def layer_weights_device(w: dict, dims, device="cuda"):
    """Upload one layer's weights; gate/up are interleaved by the library."""
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    wg = bf16_tensor(w["w_g"], device)
    wu = bf16_tensor(w["w_u"], device)
    f_pad = (dims.d_ff + 63) // 64 * 64
    w_gu = torch.empty((2 * f_pad, dims.d_model), dtype=torch.bfloat16, device=device)
    hb.hb_interleave_gate_up(wg, wu, w_gu)
    del wg, wu
    return hb.LayerWeights(w_qkv=bf16_tensor(w["w_qkv"], device), w_o=bf16_tensor(w["w_o"], device), w_gu=w_gu,
                           w_d=bf16_tensor(w["w_d"], device), g1=bf16_tensor(w["g1"], device),
                           g2=bf16_tensor(w["g2"], device))


def rope_table_device(max_pos: int, dims, device="cuda"):
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    t = torch.empty((max_pos, dims.d_head // 2, 2), dtype=torch.float32, device=device)
    hb.hb_rope_table(t, max_pos, dims.d_head, dims.theta)
    return t


def workspace(nbytes: int, device="cuda"):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
