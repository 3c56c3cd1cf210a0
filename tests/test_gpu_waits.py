"""Failure detection without a GPU fault: a bounded device wait that runs out.

A kernel waits on a barrier that nothing completes (hb_selftest_wait_timeout);
its wait gives up after a short limit, records a timeout in the device status
word and returns.  hb_check_status must then report HB_ERR_TIMEOUT, clear the
word, and the context must stay usable: a following kernel runs and the next
status check is clean.
"""
import time

import numpy as np
import pytest

import workloads as wl
from workloads import device as wd

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import chunked_prefill_hybrid_tau_gb300 as hb  # noqa: E402
from chunked_prefill_hybrid_tau_gb300 import _lib as L  # noqa: E402
import oracle.layer as ol  # noqa: E402


def test_expired_wait_is_reported_and_the_context_stays_usable():
    try:
        hb.hb_check_status()  # start from a clean status word, whatever an earlier test left
    except hb.HBError:
        pass
    for timeout_us in (2000, 20000):
        t0 = time.perf_counter()
        hb.hb_selftest_wait_timeout(timeout_us)
        with pytest.raises(hb.HBError) as err:
            hb.hb_check_status()
        waited = time.perf_counter() - t0
        assert err.value.status == L.HB_ERR_TIMEOUT
        # the wait held for about its limit before giving up (half of it, so a
        # coarse global timer cannot fail the check)
        assert waited >= 0.5 * timeout_us * 1e-6
        hb.hb_check_status()  # the word was cleared
    # the context still runs kernels: the RoPE table matches the oracle's
    dims = wl.Dims(d_model=256, n_q=4, n_kv=2, d_head=64, d_ff=64)
    max_pos = 64
    table = wd.rope_table_device(max_pos, dims)
    hb.hb_check_status()
    cos, sin = ol.rope_tables(max_pos, dims.d_head, dims.theta)
    got = wd.to_numpy(table)
    assert np.allclose(got[..., 0], cos, rtol=0, atol=1e-6)
    assert np.allclose(got[..., 1], sin, rtol=0, atol=1e-6)


def test_selftest_rejects_bad_limits():
    for bad in (0, -5, 1000001):
        with pytest.raises(hb.HBError) as err:
            hb.hb_selftest_wait_timeout(bad)
        assert err.value.status == L.HB_ERR_INVALID_ARG
    hb.hb_check_status()
