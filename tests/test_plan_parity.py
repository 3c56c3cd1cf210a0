"""C++ planner (hb_plan_batch through the C ABI) against the oracle planner:
bit-exact rows, positions, slots, sequences, block tables and page lists."""
import ctypes as C
import json
import os

import numpy as np
import pytest

import oracle.plan as op
import workloads as wl
from chunked_prefill_hybrid_tau_gb300 import _lib as L
from chunked_prefill_hybrid_tau_gb300 import binding as B

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def compare(args, **kw):
    o = op.plan_batch(*args, **kw)
    c = B.hb_plan_batch(*args, **kw)
    assert list(c.row_seq) == o.row_seq
    assert list(c.row_pos) == o.row_pos
    assert list(c.slot_mapping) == o.slot_mapping
    assert list(c.seq_q_start) == o.seq_q_start
    assert list(c.seq_pos0) == o.seq_pos0
    assert list(c.seq_kv_len) == o.seq_kv_len
    assert list(c.seq_kind) == o.seq_kind
    assert list(c.seq_req) == o.seq_req
    assert c.block_table.tolist() == o.block_table
    assert list(c.pf_take) == o.pf_take
    assert list(c.pf_finished) == o.pf_finished
    assert c.dec_pages == o.dec_pages and c.pf_pages == o.pf_pages
    assert c.free_pool == o.free_pool and c.pages_used == o.pages_used
    assert c.over_budget == o.over_budget
    # scheduling hints: query-key pairs (a row at position p sees p + 1 keys)
    # of one-row and of several-row sequences, and the latter's rows
    rows = [o.seq_q_start[k + 1] - o.seq_q_start[k] for k in range(len(o.seq_pos0))]
    pairs = [sum(p + 1 for p in o.row_pos[o.seq_q_start[k]:o.seq_q_start[k + 1]]) for k in range(len(rows))]
    assert c.decode_pairs == sum(pk for pk, n in zip(pairs, rows) if n == 1)
    assert c.chunk_pairs == sum(pk for pk, n in zip(pairs, rows) if n > 1)
    assert c.chunk_rows == sum(n for n in rows if n > 1)
    return o, c


def random_case(rng):
    b = int(rng.integers(0, 7))
    n_pf = int(rng.integers(0, 5))
    tau = int(rng.integers(1, 200))
    chunk = int(rng.integers(1, 120))
    ctx = [int(v) for v in rng.integers(0, 300, b)]
    pf_len = [int(v) for v in rng.integers(1, 400, n_pf)]
    pf_done = [int(rng.integers(0, L_)) for L_ in pf_len]
    dec_pages = [list(range(1000 * i, 1000 * i + wl.pages_for(c))) for i, c in enumerate(ctx)]
    pf_pages = [list(range(50000 + 1000 * j, 50000 + 1000 * j + wl.pages_for(d))) for j, d in enumerate(pf_done)]
    pool = [int(v) for v in rng.permutation(np.arange(90000, 90400))]
    return (ctx, dec_pages, pf_len, pf_done, pf_pages, pool, tau, chunk)


def test_random_queues_bit_exact():
    rng = np.random.default_rng(11)
    for _ in range(400):
        args = random_case(rng)
        compare(args, max_pages=64)


def test_worked_example_through_cpp():
    g = json.load(open(os.path.join(GOLDEN, "yi34b_worked_iteration.json")))
    ctx = g["decode_ctx"]
    pf = g["prefills"]
    dp = [list(range(1000 * (i + 1), 1000 * (i + 1) + wl.pages_for(c))) for i, c in enumerate(ctx)]
    pp = [list(range(50000, 50000 + wl.pages_for(pf[0]["done"]))), []]
    o, c = compare((ctx, dp, [r["prompt_len"] for r in pf], [r["done"] for r in pf], pp,
                    list(range(100000, 100400)), g["tau"], g["chunk"]))
    assert c.n_rows == g["expect"]["batch_tokens"]
    assert list(c.pf_take) == g["expect"]["take"]


def test_page_boundaries():
    # contexts 15 (last slot of a page), 16 (new page), 0 (fresh), 31, 32
    compare(([15, 16, 0, 31, 32], [[7], [8], [], [1, 2], [3, 4]], [40], [17], [[9, 10]],
             [100, 101, 102, 103, 104, 105, 106], 30, 30))


def test_over_budget_and_exact_budget():
    o, c = compare(([5, 6, 7], [[1], [2], [3]], [10], [0], [[]], [50, 51], 2, 4))
    assert c.over_budget == 1 and c.n_rows == 3 and list(c.pf_take) == [0]
    o, c = compare(([5, 6, 7], [[1], [2], [3]], [10], [0], [[]], [50, 51], 3, 4))
    assert c.over_budget == 0 and list(c.pf_take) == [0]


def test_out_of_pages_leaves_inputs_untouched(lib):
    pages = np.array([1, 0, 0, 0], np.int32)
    req = (L.hb_request * 1)(L.hb_request(0, 16, 1, 4, pages.ctypes.data_as(L.p_i32)))
    pool_arr = np.zeros(0, np.int32)
    pool = L.hb_page_pool(pool_arr.ctypes.data_as(L.p_i32), 0, 0)
    out = {k: np.zeros(8, np.int32) for k in ["a", "b", "c", "d", "e", "f", "g", "h", "i", "j", "k"]}
    P = L.hb_plan()
    P.row_cap = P.seq_cap = P.max_pages = 8
    P.pf_cap = 0
    names = ["row_seq", "row_pos", "slot_mapping", "seq_q_start", "seq_pos0", "seq_kv_len", "seq_kind", "seq_req",
             "block_table", "pf_take", "pf_finished"]
    for n, k in zip(names, out):
        setattr(P, n, out[k].ctypes.data_as(L.p_i32))
    st = lib.hb_plan_batch(req, 1, None, 0, C.byref(pool), 8, 8, 16, C.byref(P))
    assert st == L.HB_ERR_OUT_OF_PAGES
    assert P.need_pages == 1 and pool.head == 0 and req[0].n_pages == 1


def test_capacity_error_reports_sizes(lib):
    pages = np.zeros(8, np.int32)
    req = (L.hb_request * 1)(L.hb_request(100, 0, 0, 8, pages.ctypes.data_as(L.p_i32)))
    pool_arr = np.arange(20, dtype=np.int32)
    pool = L.hb_page_pool(pool_arr.ctypes.data_as(L.p_i32), 20, 0)
    P = L.hb_plan()
    P.row_cap, P.seq_cap, P.max_pages, P.pf_cap = 10, 4, 8, 1
    st = lib.hb_plan_batch(None, 0, req, 1, C.byref(pool), 64, 64, 16, C.byref(P))
    assert st == L.HB_ERR_CAPACITY
    assert P.need_rows == 64 and P.need_seqs == 1 and P.need_max_pages == 4 and P.need_pages == 4
    assert pool.head == 0 and req[0].n_pages == 0


def test_invalid_requests(lib):
    pages = np.zeros(4, np.int32)
    # holds 1 page for 40 cached tokens: inconsistent
    req = (L.hb_request * 1)(L.hb_request(0, 40, 1, 4, pages.ctypes.data_as(L.p_i32)))
    pool = L.hb_page_pool(None, 0, 0)
    P = L.hb_plan()
    assert lib.hb_plan_batch(req, 1, None, 0, C.byref(pool), 8, 8, 16, C.byref(P)) == L.HB_ERR_INVALID_ARG
    assert lib.hb_plan_batch(req, 1, None, 0, C.byref(pool), 0, 8, 16, C.byref(P)) == L.HB_ERR_INVALID_ARG


def test_config_packings_bit_exact():
    for wlf in [wl.tiny_layer]:
        w = wlf()
        st = w.state
        compare(([r.done for r in st.decodes], [r.pages for r in st.decodes], [256], [128],
                 [[int(v) for v in np.arange(8)]], st.free_pool, 68, 64))
    rng = np.random.default_rng(0)
    st = wl.make_state(rng, wl.MISTRAL, [int(v) for v in rng.integers(512, 4097, 32)], [(4096, 1024)],
                       slack_pages=80, fill_kv=False)
    o, c = compare(([r.done for r in st.decodes], [r.pages for r in st.decodes], [4096], [1024],
                    [st.prefills[0].pages], st.free_pool, 512, 512))
    assert c.n_rows == 512 and list(c.pf_take) == [480]


# ---------------------------------------------------------------- iteration driver
def test_scheduler_matches_oracle_loop_bit_exact():
    """The C iteration driver against the oracle loop on random streams with
    arrivals between iterations: every iteration's plan arrays and row
    request ids, and every request's state after each commit."""
    import oracle.sched as osch
    rng = np.random.default_rng(21)
    for trial in range(30):
        tau = int(rng.integers(4, 300))
        C = int(rng.integers(1, 2 * tau))
        pool = [int(v) for v in rng.permutation(600)]
        c = B.Scheduler(tau, C, pool)
        o = osch.SchedLoop(tau, C, pool)
        arrivals = {}
        for _ in range(int(rng.integers(1, 10))):
            arrivals.setdefault(int(rng.integers(0, 15)), []).append((int(rng.integers(1, 200)),
                                                                      int(rng.integers(1, 12))))
        it = 0
        while True:
            for pl, mn in arrivals.get(it, []):
                assert c.add(pl, mn) == o.add(pl, mn)
            if o.active() == 0 and it > max(arrivals):
                assert c.active() == 0
                break
            hc, rc = c.plan()
            po, ro = o.plan()
            assert list(rc) == ro
            assert list(hc.row_pos) == po.row_pos and list(hc.slot_mapping) == po.slot_mapping
            assert list(hc.seq_q_start) == po.seq_q_start and list(hc.seq_kv_len) == po.seq_kv_len
            assert list(hc.seq_kind) == po.seq_kind and list(hc.seq_req) == po.seq_req
            S = len(po.seq_pos0)
            assert [list(r) for r in hc.block_table] == [row[:hc.max_pages] + [-1] * (hc.max_pages - len(row))
                                                         if len(row) < hc.max_pages else row[:hc.max_pages]
                                                         for row in po.block_table][:S]
            c.commit()
            o.commit()
            for i, r in enumerate(o.reqs):
                assert c.info(i) == (r["state"], r["cached"], r["generated"], len(r["pages"]))
            assert c.free_pages() == len(o.pool)
            it += 1
        c.close()


def test_scheduler_errors_leave_state_unchanged(lib):
    s = B.Scheduler(32, 32, list(range(3)))  # three pages: room for one 48-token prompt
    a = s.add(40, 2)
    s.add(40, 2)
    hp, rr = s.plan()
    assert set(rr.tolist()) == {a} and hp.n_rows == 32  # the second prompt gets no tokens this iteration
    with pytest.raises(B.HBError):
        s.add(5, 1)  # refused between plan and commit
    s.commit()
    with pytest.raises(B.HBError) as e:
        s.plan()  # both prompts need pages now: out of pages, no preemption
    assert e.value.status == L.HB_ERR_OUT_OF_PAGES
    assert s.info(a) == (0, 32, 0, 2) and s.free_pages() == 1
    with pytest.raises(B.HBError):
        s.commit()  # nothing planned
    with pytest.raises(B.HBError):
        s.info(7)
    s.close()
