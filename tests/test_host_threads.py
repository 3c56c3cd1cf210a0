"""The host half of the C ABI is safe to call from several threads at once.

hb_plan_batch keeps no state between calls, each hb_sched handle owns its
state, and hb_last_error is per thread.  ctypes releases the GIL around each
call, so the threads below run inside the library concurrently.  CPU only.
"""
import concurrent.futures
import threading

import numpy as np

from chunked_prefill_hybrid_tau_gb300 import _lib as L
from chunked_prefill_hybrid_tau_gb300 import binding as B
import workloads as wl

N_THREADS = 8


def plan_problem(seed):
    rng = np.random.default_rng(seed)
    dims = wl.Dims(d_model=64, n_q=2, n_kv=1, d_head=32, d_ff=64)
    dec = [int(c) for c in rng.integers(0, 3000, size=int(rng.integers(0, 24)))]
    pfs = [(int(rng.integers(1, 5000)), 0) for _ in range(int(rng.integers(0, 4)))]
    pfs = [(L_, int(rng.integers(0, L_))) for L_, _ in pfs]
    st = wl.make_state(rng, dims, dec, pfs, slack_pages=400, fill_kv=False)
    tau = int(rng.integers(1, 2048))
    chunk = int(rng.integers(1, 2048))
    return ([r.done for r in st.decodes], [r.pages for r in st.decodes], [r.prompt_len for r in st.prefills],
            [r.done for r in st.prefills], [r.pages for r in st.prefills], st.free_pool, tau, chunk)


def plan_key(p):
    return (p.row_seq.tobytes(), p.row_pos.tobytes(), p.slot_mapping.tobytes(), p.seq_q_start.tobytes(),
            p.seq_kv_len.tobytes(), p.block_table.tobytes(), p.pf_take.tobytes(), tuple(p.free_pool),
            tuple(tuple(x) for x in p.dec_pages), tuple(tuple(x) for x in p.pf_pages))


def test_plan_batch_concurrent_equals_serial():
    problems = [plan_problem(s) for s in range(32)]
    serial = [plan_key(B.hb_plan_batch(*p)) for p in problems]

    def run(i):  # thread i plans problems i, i + 8, ... four times over
        return [(j % 32, plan_key(B.hb_plan_batch(*problems[j % 32]))) for j in range(i, 32 * 4, N_THREADS)]

    with concurrent.futures.ThreadPoolExecutor(N_THREADS) as ex:
        for out in ex.map(run, range(N_THREADS)):
            for j, key in out:
                assert key == serial[j]


def drive(seed):
    """One scheduler handle through a random stream; returns every
    iteration's row request ids and positions."""
    rng = np.random.default_rng(seed)
    s = B.Scheduler(int(rng.integers(8, 256)), int(rng.integers(4, 300)), [int(v) for v in rng.permutation(800)])
    for _ in range(int(rng.integers(2, 12))):
        s.add(int(rng.integers(1, 300)), int(rng.integers(1, 10)))
    trace = []
    while s.active():
        hp, req = s.plan()
        trace.append((req.tobytes(), hp.row_pos.tobytes(), hp.slot_mapping.tobytes()))
        s.commit()
    s.close()
    return trace


def test_scheduler_handles_run_concurrently():
    seeds = list(range(16))
    serial = [drive(sd) for sd in seeds]
    with concurrent.futures.ThreadPoolExecutor(N_THREADS) as ex:
        for sd, got in zip(seeds, ex.map(drive, seeds)):
            assert got == serial[sd]


def test_last_error_is_per_thread():
    lib = L.load()
    barrier = threading.Barrier(2)
    seen = {}

    def fail(name, fn):
        st = fn()
        barrier.wait()  # both threads have failed before either reads its message
        seen[name] = (st, lib.hb_last_error().decode())

    t1 = threading.Thread(target=fail, args=("gemm", lambda: lib.hb_gemm(None, None, None, None, 1, 8, 8, 0, None)))
    t2 = threading.Thread(target=fail, args=("wait", lambda: lib.hb_selftest_wait_timeout(0, None)))
    t1.start(); t2.start(); t1.join(); t2.join()
    assert seen["gemm"][0] == L.HB_ERR_INVALID_ARG and "hb_gemm" in seen["gemm"][1]
    assert seen["wait"][0] == L.HB_ERR_INVALID_ARG and "hb_selftest_wait_timeout" in seen["wait"][1]
