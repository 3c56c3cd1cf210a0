"""The bench's cost model (chunked_prefill_hybrid_tau_gb300/costs.py) against
closed forms: the projections' FLOPs are 2 T Psi (Sarathi-Serve reading
notes, section 1.6), attention's are 4 n_q d_head sum(p + 1) over the rows
(section 7.5b), E4M3 weights are read at one byte per parameter, and the FP8
roofline halves the projections' tensor time (section 7.7)."""
import numpy as np
import pytest

import oracle.plan as op
import workloads as wl
from chunked_prefill_hybrid_tau_gb300 import costs


@pytest.fixture(scope="module")
def plan():
    rng = np.random.default_rng(12)
    dims = wl.MISTRAL
    st = wl.make_state(rng, dims, [int(c) for c in rng.integers(100, 3000, 24)], [(4096, 1024)], slack_pages=64,
                       fill_kv=False)
    p = op.plan_batch([r.done for r in st.decodes], [r.pages for r in st.decodes],
                      [r.prompt_len for r in st.prefills], [r.done for r in st.prefills],
                      [r.pages for r in st.prefills], st.free_pool, 512, 512, dims.page)
    return dims, p


def test_flops_closed_forms(plan):
    dims, p = plan
    sc = costs.stage_costs(dims, p.row_pos, p.seq_q_start, p.seq_kv_len)
    T = len(p.row_pos)
    linear = sum(sc[k][0] for k in ("qkv", "o_proj", "gate_up", "down"))
    assert linear == 2.0 * T * dims.params_per_layer
    assert sc["attention"][0] == 4.0 * dims.n_q * dims.d_head * float(np.sum(np.asarray(p.row_pos) + 1))


def test_e4m3_weight_bytes_and_roofline(plan):
    dims, p = plan
    s2 = costs.stage_costs(dims, p.row_pos, p.seq_q_start, p.seq_kv_len)
    s1 = costs.stage_costs(dims, p.row_pos, p.seq_q_start, p.seq_kv_len, weight_bytes=1)
    b2 = sum(v[1] for v in s2.values())
    b1 = sum(v[1] for v in s1.values())
    assert b2 - b1 == dims.params_per_layer  # one byte less per weight
    # math-bound (infinite bandwidth): the projections take half as long with FP8
    tf = 1000.0
    t16 = costs.roofline_time(s2, tf, 1e30, f8=False)
    t8 = costs.roofline_time(s1, tf, 1e30, f8=True)
    proj = sum(s2[k][0] for k in ("qkv", "o_proj", "gate_up", "down")) / (tf * 1e12)
    assert t16 - t8 == pytest.approx(proj / 2, rel=1e-12)
    # memory-bound (infinite FLOP rate): bytes over bandwidth
    assert costs.roofline_time(s1, 1e30, 1000.0, f8=True) == pytest.approx(b1 / 1e12, rel=1e-12)


# ----------------------------------------------------------------------------
# tau calibration (the scheduling method's profiling step: largest budget n
# with T(n) <= T*, Sarathi-Serve reading notes section 3.3)
# ----------------------------------------------------------------------------
def test_select_tau_takes_the_largest_budget_within_the_slo():
    import bench
    # flat up to 512, then linear: T(n) = 10 ms below the knee, 10 + (n - 512) / 100 above
    prof = [(n, 10.0 if n <= 512 else 10.0 + (n - 512) / 100.0) for n in (64, 128, 256, 512, 1024, 2048, 4096)]
    assert bench.select_tau(prof, 10.0) == (512, 1024)      # every budget up to the knee fits
    assert bench.select_tau(prof, 15.2) == (1024, 1024)     # 1024 -> 15.12 ms fits, 2048 -> 25.36 does not
    assert bench.select_tau(prof, 1e9) == (4096, 1024)
    assert bench.select_tau(prof, 5.0) == (None, 1024)      # nothing fits a tighter SLO
    # the knee is the first budget 10% above the smallest budget's time
    assert bench.select_tau([(64, 1.0), (128, 1.05), (256, 1.1), (512, 2.0)], 10.0) == (512, 256)
    assert bench.select_tau([(64, 1.0), (128, 1.0)], 10.0) == (128, None)
    # a non-monotone profile still returns the largest fitting budget
    assert bench.select_tau([(64, 1.0), (128, 3.0), (256, 2.0)], 2.5)[0] == 256


def test_launch_count_follows_the_fused_qkv_rule():
    """The bench's gpu_launches claim, from the library's own rule: 8
    kernels per bf16 layer; 10 per E4M3 layer whose QKV tiles hold whole
    heads (RoPE/KV append fused), else 11; nothing for an empty batch."""
    import bench
    import workloads as wl
    assert bench.launches_per_layer(wl.MISTRAL, False, 512) == 8
    assert bench.launches_per_layer(wl.TINY, False, 68) == 8
    assert bench.launches_per_layer(wl.MISTRAL, False, 0) == 0
    assert bench.launches_per_layer(wl.MISTRAL, True, 512) == 10     # 6144 QKV columns, d_head 128
    assert bench.launches_per_layer(wl.YI34B, True, 1024) == 10      # 9216 columns
    odd = wl.Dims(d_model=256, n_q=3, n_kv=1, d_head=64, d_ff=64)  # 320 columns: not whole 256-column tiles
    assert bench.launches_per_layer(odd, True, 68) == 11
    import chunked_prefill_hybrid_tau_gb300 as hb
    with pytest.raises(hb.HBError):
        hb.hb_layer_kernel_count(wl.MISTRAL, -1, 0)
    with pytest.raises(hb.HBError):
        hb.hb_layer_kernel_count(wl.MISTRAL, 512, 7)
