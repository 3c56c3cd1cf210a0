"""Layer-level parity: hb_layer_forward against the oracle's layer on the
tiny configuration and the Mistral-7B-shaped layer at tau = 512 (GPU)."""
import numpy as np
import pytest

import workloads as wl
from workloads import device as wd
from tests.gpu_harness import GpuLayer, assert_close, oracle_layer, plan_both

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def advance(st: wl.State, hp):
    """Apply a plan to the host state: pages appended, pool consumed, progress
    advanced (the caller's side of an iteration)."""
    for i, r in enumerate(st.decodes):
        r.pages = list(hp.dec_pages[i])
        r.done += 1
    for j, r in enumerate(st.prefills):
        r.pages = list(hp.pf_pages[j])
        r.done += int(hp.pf_take[j])
    st.free_pool = list(hp.free_pool)


def test_tiny_layer_two_iterations():
    w = wl.tiny_layer(seed=0)
    st, dims = w.state, w.dims
    max_pos = 512
    gl = GpuLayer(w.weights[0], dims, st.k_pool, st.v_pool, max_pos)
    k_ref, v_ref = st.k_pool.copy(), st.v_pool.copy()
    # iteration A: the prompt's first 128 tokens alone (computes the prefix KV)
    saved_dec = st.decodes
    st.decodes = []
    hp, o = plan_both(st, 128, 128)
    got = gl.forward(hp, w.x_prompt[:128], 512)
    ref = oracle_layer(w.weights[0], dims, o, w.x_prompt[:128], k_ref, v_ref, max_pos)
    assert_close(got, ref, "tiny iteration A", scale="rms")
    advance(st, hp)
    st.decodes = saved_dec
    # iteration B: 4 decodes + the 64-token chunk at positions 128..191
    hp, o = plan_both(st, 68, 64)
    assert hp.n_rows == 68 and list(hp.row_pos[4:]) == list(range(128, 192))
    got = gl.forward(hp, w.x, 512)
    ref = oracle_layer(w.weights[0], dims, o, w.x, k_ref, v_ref, max_pos)
    assert_close(got, ref, "tiny iteration B", scale="rms")
    assert_close(wd.to_numpy(gl.k), k_ref, "tiny K cache")
    assert_close(wd.to_numpy(gl.v), v_ref, "tiny V cache")


@pytest.fixture(scope="module")
def mistral():
    return wl.mistral_layer(seed=0)


def test_mistral_layer_tau512(mistral):
    w = mistral
    st, dims = w.state, w.dims
    max_pos = 4096
    hp, o = plan_both(st, 512, 512)
    assert hp.n_rows == 512 and list(hp.pf_take) == [480]
    gl = GpuLayer(w.weights[0], dims, st.k_pool, st.v_pool, max_pos)
    got = gl.forward(hp, w.x, int(hp.seq_kv_len.max()))
    k_ref, v_ref = st.k_pool.copy(), st.v_pool.copy()
    ref = oracle_layer(w.weights[0], dims, o, w.x, k_ref, v_ref, max_pos)
    assert_close(got, ref, "mistral layer output", scale="rms")
    # the appended KV (all other slots unchanged)
    sl = np.asarray(hp.slot_mapping)
    kg = wd.to_numpy(gl.k)[sl // 16, :, sl % 16]
    vg = wd.to_numpy(gl.v)[sl // 16, :, sl % 16]
    assert_close(kg, k_ref[sl // 16, :, sl % 16], "mistral appended K")
    assert_close(vg, v_ref[sl // 16, :, sl % 16], "mistral appended V")
