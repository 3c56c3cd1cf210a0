"""Layer-level parity: hb_layer_forward against the oracle's layer on the
tiny configuration and the Mistral-7B-shaped layer at tau = 512 (GPU)."""
import numpy as np
import pytest

import workloads as wl
from workloads import device as wd
from tests.gpu_harness import GpuLayer, assert_close, assert_layer, oracle_layer_both, plan_both

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
    p32 = (st.k_pool.copy(), st.v_pool.copy())
    p16 = (st.k_pool.copy(), st.v_pool.copy())
    # iteration A: the prompt's first 128 tokens alone (computes the prefix KV)
    saved_dec = st.decodes
    st.decodes = []
    hp, o = plan_both(st, 128, 128)
    got = gl.forward(hp, w.x_prompt[:128], 512)
    ref, emu, h = oracle_layer_both(w.weights[0], dims, o, w.x_prompt[:128], p32, p16, max_pos)
    assert_layer(got, ref, emu, h, "tiny iteration A")
    advance(st, hp)
    st.decodes = saved_dec
    # iteration B: 4 decodes + the 64-token chunk at positions 128..191
    hp, o = plan_both(st, 68, 64)
    assert hp.n_rows == 68 and list(hp.row_pos[4:]) == list(range(128, 192))
    got = gl.forward(hp, w.x, 512)
    ref, emu, h = oracle_layer_both(w.weights[0], dims, o, w.x, p32, p16, max_pos)
    assert_layer(got, ref, emu, h, "tiny iteration B")
    assert_close(wd.to_numpy(gl.k), p16[0], "tiny K cache")
    assert_close(wd.to_numpy(gl.v), p16[1], "tiny V cache")


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
    p32 = (st.k_pool.copy(), st.v_pool.copy())
    p16 = (st.k_pool.copy(), st.v_pool.copy())
    ref, emu, h = oracle_layer_both(w.weights[0], dims, o, w.x, p32, p16, max_pos)
    assert_layer(got, ref, emu, h, "mistral layer output")
    # the appended KV (all other slots unchanged)
    sl = np.asarray(hp.slot_mapping)
    kg = wd.to_numpy(gl.k)[sl // 16, :, sl % 16]
    vg = wd.to_numpy(gl.v)[sl // 16, :, sl % 16]
    assert_close(kg, p16[0][sl // 16, :, sl % 16], "mistral appended K")
    assert_close(vg, p16[1][sl // 16, :, sl % 16], "mistral appended V")
