"""Shared helpers of the GPU parity tests: tolerance checks and layer runs
through the C ABI with the oracle beside them."""
from __future__ import annotations

import numpy as np

import oracle.layer as ol
import oracle.plan as op
import workloads as wl
from workloads import device as wd

# Tolerance for bf16 activations and outputs (2e-2 max-abs, 1e-2 relative L2):
#   kernel bound, for a kernel against the oracle fed the same bf16 inputs:
#   |gpu - ref| <= 2e-2 + 2e-2 |ref| elementwise (a bf16 value v is itself
#   rounded by up to 2^-9 |v|, and one ulp is 2^-8 |v|, so a purely absolute
#   bound cannot hold for |v| >= 4) and relative L2 <= 1e-2;
#   a layer's output against the oracle in fp32 (ref) and in its bf16-storage
#   variant (emu, which rounds where the GPU stores: qkv, q, k, P, o, h, a and
#   the output).  Two valid bf16 implementations do not round alike: the
#   softmax weights P are rounded against a running maximum on the GPU and
#   against the final one in the oracle, so about half of o's bf16 values
#   differ by an ulp, and that noise reaches the output (measured on the
#   Mistral-shaped layer: relative L2 3.2e-3 between GPU and emu, 3.3e-3
#   between emu and fp32).  The bounds are therefore taken from the oracle's
#   own rounding noise at the same inputs:
#     relative L2 (gpu, ref) <= 1.5 x relative L2 (emu, ref), and <= 1e-2;
#     relative L2 (gpu, emu) <= 1e-2;
#     elementwise, against either: the kernel bound plus one bf16 ulp of the
#     stored residual h (2^-7 |h|: out = h + mlp is formed from the stored h,
#     and a one-ulp flip of h passes into out unchanged even where mlp nearly
#     cancels it), or 1.5 x the largest |emu - ref|, whichever is larger.
ATOL = 2e-2
RTOL = 2e-2
REL_L2 = 1e-2


def assert_close(gpu, ref, what, atol=ATOL, rtol=RTOL, rel_l2=REL_L2, floor=None, extra=None):
    """Kernel bound by default; `extra` adds an elementwise term (the h ulp
    of a layer output); `floor` raises the elementwise bound to at least that
    absolute value (the bf16-storage deviation of a layer)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = atol + rtol * np.abs(ref)
    if extra is not None:
        bound = bound + np.asarray(extra, np.float64)
    if floor is not None:
        bound = np.maximum(bound, floor)
    denom = np.linalg.norm(ref)
    rl2 = float(np.linalg.norm(gpu - ref) / denom) if denom > 0 else 0.0
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (f"{what}: max excess at {np.unravel_index(worst, err.shape)}: "
                                  f"gpu {gpu.flat[worst]} ref {ref.flat[worst]} (max abs err {err.max():.4g}, "
                                  f"rms {rms:.4g}, max/rms {err.max() / max(rms, 1e-30):.4g}, relL2 {rl2:.4g}, "
                                  f"{int(np.sum(err > bound))} of {err.size} outside)")
    assert rl2 <= rel_l2, f"{what}: relative L2 {rl2:.4g} > {rel_l2}"
    return float(err.max())


H_ULP = 2.0 ** -7  # one bf16 ulp relative to |h|, at most


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def assert_layer(gpu, ref, emu, h, what):
    """A layer's output against the oracle in fp32 (ref) and in its
    bf16-storage variant (emu, with its stored residual h); bounds above."""
    extra = H_ULP * np.abs(np.asarray(h, np.float64))
    emax = float(np.max(np.abs(np.asarray(emu, np.float64) - np.asarray(ref, np.float64))))
    e_rl2 = rel_l2(emu, ref)
    g_rl2 = rel_l2(gpu, ref)
    print(f"\n{what}: relL2 gpu/fp32 {g_rl2:.4g} emu/fp32 {e_rl2:.4g} gpu/emu {rel_l2(gpu, emu):.4g}; "
          f"max abs gpu/fp32 {np.abs(np.asarray(gpu, np.float64) - ref).max():.4g} emu/fp32 {emax:.4g}")
    assert g_rl2 <= 1.5 * e_rl2, f"{what}: relative L2 {g_rl2:.4g} beyond 1.5 x bf16 storage's {e_rl2:.4g}"
    assert_close(gpu, emu, what + " (vs bf16-storage oracle)", extra=extra, floor=1.5 * emax)
    return assert_close(gpu, ref, what + " (vs fp32 oracle)", extra=extra, floor=1.5 * emax)


def plan_both(st: wl.State, tau: int, chunk: int, max_pages=None):
    """The C++ plan (through the ABI) and the oracle plan of the same state."""
    import chunked_prefill_hybrid_tau_gb300 as hb
    args = ([r.done for r in st.decodes], [r.pages for r in st.decodes], [r.prompt_len for r in st.prefills],
            [r.done for r in st.prefills], [r.pages for r in st.prefills], st.free_pool, tau, chunk, st.dims.page)
    hp = hb.hb_plan_batch(*args, max_pages=max_pages)
    o = op.plan_batch(*args, max_pages=hp.max_pages)
    assert list(hp.slot_mapping) == o.slot_mapping and hp.block_table.tolist() == o.block_table
    return hp, o


class GpuLayer:
    """One layer's weights, caches and RoPE table on the device."""

    def __init__(self, w: dict, dims, k_pool: np.ndarray, v_pool: np.ndarray, max_pos: int, device="cuda",
                 fmt="bf16"):
        self.dims = dims
        self.w = wd.layer_weights_device(w, dims, device, fmt=fmt)
        self.k = wd.bf16_tensor(k_pool, device)
        self.v = wd.bf16_tensor(v_pool, device)
        self.max_pos = max_pos
        self.rope = wd.rope_table_device(max_pos, dims, device)
        self.device = device

    def forward(self, hp, x: np.ndarray, max_kv_len: int):
        import torch
        import chunked_prefill_hybrid_tau_gb300 as hb
        dp = hb.DevicePlan(hp, self.device)
        xin = wd.bf16_tensor(x, self.device)
        xout = torch.empty_like(xin)
        ws = wd.workspace(hb.hb_layer_workspace_bytes(self.dims, hp.n_rows, hp.n_seqs, max_kv_len), self.device)
        hb.hb_layer_forward(self.w, self.dims, dp, self.rope, self.max_pos, xin, xout, self.k, self.v, max_kv_len, ws)
        hb.hb_check_status()
        return wd.to_numpy(xout)


def oracle_layer_both(w, dims, plan, x, pools32, pools16, max_pos):
    """The fp32 oracle and its bf16-storage variant on the same rows, each
    appending to its own (K, V) pools in place -> (ref, emu, h of emu)."""
    cos, sin = ol.rope_tables(max_pos, dims.d_head, dims.theta)
    ref = ol.layer_forward(w, dims, plan, x, pools32[0], pools32[1], cos, sin)
    emu, parts = ol.layer_forward(w, dims, plan, x, pools16[0], pools16[1], cos, sin, storage="bf16",
                                  return_parts=True)
    return ref, emu, parts["h"]
