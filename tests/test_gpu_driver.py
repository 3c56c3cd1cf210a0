"""The iteration driver end to end on the GPU (tiny layer).

A stream of requests (prompts of 1..150 tokens, 1..12 new tokens, arrivals
spread over the first iterations) runs through the C driver, with several
chunks per iteration, prompts turning into decodes and finished requests'
pages going back to the pool and being reused.  Every iteration's layer
output on the GPU is checked against the oracle running the same loop with
its own KV pool, so the KV each chunk and decode writes is carried across
iterations on both sides (Sarathi-Serve reading notes, sections 3.1 and 3.4).
"""
import numpy as np
import pytest

import oracle.layer as ol
import oracle.sched as osch
import workloads as wl
from workloads import device as wd
from tests.gpu_harness import GpuLayer, assert_layer

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402


def test_driver_stream_matches_oracle_every_iteration():
    rng = np.random.default_rng(31)
    dims = wl.TINY
    w = wl.layer_weights(rng, dims, gamma_jitter=0.1)
    n_pages, tau, C = 120, 96, 40
    pool = [int(v) for v in rng.permutation(n_pages)]
    reqs = [(int(rng.integers(1, 150)), int(rng.integers(1, 13))) for _ in range(14)]
    arrivals = {}
    for k, r in enumerate(reqs):
        arrivals.setdefault(int(rng.integers(0, 8)) if k > 2 else 0, []).append(r)
    # every request's input rows, one per position (its prompt, then the
    # rows that stand in for its generated tokens), by request id
    x_of = {}
    max_pos = max(pl + mn for pl, mn in reqs) + 1
    k0 = np.zeros((n_pages, dims.n_kv, 16, dims.d_head), np.float32)
    gl = GpuLayer(w, dims, k0, k0.copy(), max_pos)
    k_ref, v_ref = k0.copy(), k0.copy()
    k_emu, v_emu = k0.copy(), k0.copy()
    cos, sin = ol.rope_tables(max_pos, dims.d_head, dims.theta)

    drv = hb.Scheduler(tau, C, pool)
    loop = osch.SchedLoop(tau, C, pool)
    order = []  # request ids in arrival order, same on both sides
    it, multi_chunk, transitions = 0, 0, 0
    while True:
        for pl, mn in arrivals.get(it, []):
            rid = drv.add(pl, mn)
            assert loop.add(pl, mn) == rid
            order.append(rid)
            x_of[rid] = wl.activations(rng, pl + mn, dims.d_model)
        if loop.active() == 0 and it > max(arrivals):
            assert drv.active() == 0
            break
        hp, row_req = drv.plan()
        po, ro = loop.plan()
        assert list(row_req) == ro and list(hp.row_pos) == po.row_pos and list(hp.slot_mapping) == po.slot_mapping
        multi_chunk += int(np.count_nonzero(hp.seq_kind == 1) > 1)
        if hp.n_rows:  # an idle iteration (nothing arrived yet) has no forward
            x = np.stack([x_of[r][p] for r, p in zip(row_req, hp.row_pos)])
            got = gl.forward(hp, x, int(hp.seq_kv_len.max()))
            ref = ol.layer_forward(w, dims, po, x, k_ref, v_ref, cos, sin)
            emu, parts = ol.layer_forward(w, dims, po, x, k_emu, v_emu, cos, sin, storage="bf16", return_parts=True)
            assert_layer(got, ref, emu, parts["h"], f"iteration {it} ({hp.n_rows} rows)")
        before = [loop.reqs[i]["state"] for i in range(len(loop.reqs))]
        drv.commit()
        loop.commit()
        transitions += sum(1 for i, s in enumerate(before) if s == osch.PREFILLING and
                           loop.reqs[i]["state"] != osch.PREFILLING)
        it += 1
    hb.hb_check_status()
    assert drv.free_pages() == n_pages
    assert multi_chunk > 0 and transitions == len(reqs)  # the stream exercised both
