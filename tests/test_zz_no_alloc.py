"""hb_attention_noalloc: the attention entry point for callers that cannot
allocate device memory (it uses the library's fixed device scratch array).

Checked through the C ABI against the oracle's attention and against
hb_attention with a caller workspace on the same inputs, for two calls in a
row (the shared scratch keeps the previous call's contents, so the second call
checks that they are cleared).  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest

import oracle.layer as ol
import oracle.plan as op
import workloads as wl
from workloads import device as wd
from tests.gpu_harness import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402
from chunked_prefill_hybrid_tau_gb300 import _lib as L  # noqa: E402


def make_case(seed):
    dims = wl.Dims(d_model=256, n_q=8, n_kv=2, d_head=128, d_ff=64)
    rng = np.random.default_rng(seed)
    st = wl.make_state(rng, dims, [0, 17, 511, 512, 1300, 2047], [(700, 120)], slack_pages=64)
    args = ([r.done for r in st.decodes], [r.pages for r in st.decodes], [r.prompt_len for r in st.prefills],
            [r.done for r in st.prefills], [r.pages for r in st.prefills], st.free_pool, 6 + 150, 150)
    hp = hb.hb_plan_batch(*args)
    q = wl.bf16_round(rng.standard_normal((hp.n_rows, dims.n_q, dims.d_head), dtype=np.float32))
    # the oracle's attention over the same pools and plan (fp32)
    o_plan = op.plan_batch(*args, max_pages=hp.max_pages)
    ref = ol.attention(q, st.k_pool, st.v_pool, o_plan, dims.n_q, dims.n_kv, dims.page)
    ref = ref.reshape(hp.n_rows, dims.n_q * dims.d_head)
    return dims, hp, wd.bf16_tensor(q), wd.bf16_tensor(st.k_pool), wd.bf16_tensor(st.v_pool), ref


def test_noalloc_matches_workspace_entry_point_twice():
    lib = hb.lib()
    for call, seed in enumerate([21, 22]):
        dims, hp, q, kc, vc, oracle_out = make_case(seed)
        max_kv = int(hp.seq_kv_len.max())
        dp = hb.DevicePlan(hp)
        ref = torch.empty((hp.n_rows, dims.n_q * dims.d_head), dtype=torch.bfloat16, device="cuda")
        ws = wd.workspace(hb.hb_attention_workspace_bytes(dims, hp.n_rows, hp.n_seqs, max_kv))
        hb.hb_attention(q, kc, vc, dp, dims, max_kv, ref, ws)
        out = torch.full_like(ref, float("nan"))
        ds = hb.dims_struct(dims)
        ps = dp.struct()
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.hb_attention_noalloc(C.c_void_p(q.data_ptr()), C.c_void_p(kc.data_ptr()), C.c_void_p(vc.data_ptr()),
                                      int(kc.shape[0]), C.byref(ps), C.byref(ds), max_kv, C.c_void_p(out.data_ptr()),
                                      stream)
        assert st == L.HB_OK, lib.hb_last_error().decode()
        hb.hb_check_status()
        assert_close(wd.to_numpy(out), oracle_out, f"noalloc call {call + 1} against the oracle")
        assert_close(wd.to_numpy(out), wd.to_numpy(ref), f"noalloc call {call + 1} against hb_attention")


def test_noalloc_rejects_plans_beyond_its_scratch():
    lib = hb.lib()
    dims, hp, q, kc, vc, _ = make_case(23)
    dp = hb.DevicePlan(hp)
    ds = hb.dims_struct(dims)
    ps = dp.struct()
    out = torch.empty((hp.n_rows, dims.n_q * dims.d_head), dtype=torch.bfloat16, device="cuda")
    # max_kv_len far above what 32 MiB of split records can hold
    st = lib.hb_attention_noalloc(C.c_void_p(q.data_ptr()), C.c_void_p(kc.data_ptr()), C.c_void_p(vc.data_ptr()),
                                  int(kc.shape[0]), C.byref(ps), C.byref(ds), 10**7, C.c_void_p(out.data_ptr()), None)
    assert st == L.HB_ERR_CAPACITY
    assert b"scratch" in lib.hb_last_error()
