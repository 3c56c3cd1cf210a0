#!/usr/bin/env python3
"""Hybrid-iteration benchmark: tokens/s, ms/iter and roofline fraction.

One step = one pass of the whole hot path over the Mistral-7B-shaped layer
at tau = 512 (one 480-token chunk at offset 1024 of a 4096-token prompt + 32
decodes with contexts uniform in [512, 4096]): the C planner packs the batch
and maps slots, the plan is copied to the device (one pinned copy), and
hb_layer_forward runs RMSNorm, the QKV projection, RoPE + paged KV append,
the hybrid attention, the O projection + residual, RMSNorm, gate/up + SwiGLU
and the down projection + residual.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) each rank runs an independent replica on its own GPU
(the iteration has no exchange step); value = all ranks' tokens / max time.
--impl reference times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "hybrid-iteration tokens/s and ms/iter vs token budget; % of per-iteration roofline"
WORKLOAD = "mistral7b_layer_tau512"
MIN_CLOCK_S = 0.3  # seconds of layer steps the clock sampler sees at least (20 ms period)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="hb", choices=["hb", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tau", type=int, default=512)
    ap.add_argument("--decodes", type=int, default=32)
    ap.add_argument("--weights", default="bf16", choices=["bf16", "e4m3"],
                    help="projection weights: bf16, or E4M3 codes with per-row scales (FP8 projections)")
    ap.add_argument("--sweep", action="store_true",
                    help="token-budget sweep (tau 64..4096, 64 decodes, c = tau - 64): one JSON line per tau")
    ap.add_argument("--calibrate", type=float, default=None, metavar="SLO_MS",
                    help="pick tau from a time-per-iteration SLO: the largest swept tau whose --layers-layer "
                         "iteration fits the SLO, next to the c* closed form")
    ap.add_argument("--layers", type=int, default=32, help="layers per iteration for --calibrate")
    ap.add_argument("--chunk-study", action="store_true",
                    help="prefill time of 8K and 32K prompts chunked at C = 128..2048 against unchunked")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workload
def launches_per_layer(dims, f8: bool, n_rows: int) -> int:
    """Kernels one hb_layer_forward launches, by the library's own rule
    (hb_layer_kernel_count: the chunk and decode attention kernels are both
    launched whatever the batch holds)."""
    import chunked_prefill_hybrid_tau_gb300 as hb
    return hb.hb_layer_kernel_count(dims, n_rows, 1 if f8 else 0)


def make_workload(tau: int, n_dec: int):
    import workloads as wl
    if tau == 512 and n_dec == 32:
        return wl.mistral_layer(seed=0)
    return wl.mistral_layer(seed=0, tau=tau, n_dec=n_dec, ctx_lo=512, ctx_hi=8192, prompt_len=8192, offset=0)


class PlanRunner:
    """Per-step planning through the C ABI into pinned staging buffers, and
    one host-to-device copy per step of the kernel-facing plan arrays on a
    copy stream of its own, so the upload overlaps the previous step."""

    def __init__(self, lib, st, tau, chunk, device):
        import torch
        from chunked_prefill_hybrid_tau_gb300 import _lib as L
        self.lib, self.L, self.tau, self.chunk = lib, L, tau, chunk
        self.n_dec, self.n_pf = len(st.decodes), len(st.prefills)
        self.page_bufs = []
        self.dec = (L.hb_request * max(self.n_dec, 1))()
        self.pf = (L.hb_request * max(self.n_pf, 1))()
        grow = tau // 16 + 2
        self.n_pages0 = []
        for arr, reqs in ((self.dec, st.decodes), (self.pf, st.prefills)):
            for i, r in enumerate(reqs):
                b = np.zeros(len(r.pages) + grow, np.int32)
                b[:len(r.pages)] = r.pages
                self.page_bufs.append(b)
                arr[i] = L.hb_request(r.prompt_len, r.done, len(r.pages), b.size, b.ctypes.data_as(L.p_i32))
                self.n_pages0.append(len(r.pages))
        self.pool_arr = np.asarray(st.free_pool, np.int32)
        self.row_cap = max(tau, self.n_dec)
        self.seq_cap = self.n_dec + self.n_pf
        spans = [r.done + 1 for r in st.decodes] + [r.done + min(chunk, tau) for r in st.prefills]
        self.max_pages = max((s + 15) // 16 for s in spans)
        rc, sc, mp = self.row_cap, self.seq_cap, self.max_pages
        self.off = np.cumsum([0, rc, rc, sc + 1, sc, sc * mp])  # row_pos, slots, q_start, kv_len, table
        self.dev_ints = int(self.off[-1])
        self.host_only = {k: np.zeros(n, np.int32) for k, n in
                          (("row_seq", rc), ("seq_pos0", sc), ("seq_kind", sc), ("seq_req", sc),
                           ("pf_take", max(self.n_pf, 1)), ("pf_finished", max(self.n_pf, 1)))}
        # two pinned staging buffers and two device copies: step k's plan is
        # uploaded on a copy stream into dev[k % 2] while step k - 1 computes
        self.pinned = [torch.zeros(self.dev_ints, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.dev = [torch.zeros(self.dev_ints, dtype=torch.int32, device=device) for _ in range(2)]
        self.copied = [torch.cuda.Event(), torch.cuda.Event()]
        self.released = [torch.cuda.Event(), torch.cuda.Event()]
        self.copy_stream = torch.cuda.Stream(device=device)
        self.k = 0
        self.h2d_bytes = 0

    def step(self, stream):
        """Plan the iteration on the host, upload it on the copy stream and
        make `stream` wait for the upload.  Returns the hb_device_plan struct.
        The caller enqueues one layer forward on `stream` between two calls:
        that layer is the last reader of its device plan."""
        import torch
        L = self.L
        b = self.k & 1
        if self.k >= 1:
            self.released[b ^ 1].record(stream)  # end of the previous step's layer
        self.copied[b].synchronize()  # the copy that last read this staging buffer is done
        stage = self.pinned[b].numpy()
        for i in range(self.n_dec):
            self.dec[i].n_pages = self.n_pages0[i]
        for j in range(self.n_pf):
            self.pf[j].n_pages = self.n_pages0[self.n_dec + j]
        P = L.hb_plan()
        P.row_cap, P.seq_cap, P.max_pages, P.pf_cap = self.row_cap, self.seq_cap, self.max_pages, self.n_pf
        base = stage.ctypes.data

        def at(i):
            return C.cast(base + 4 * int(self.off[i]), L.p_i32)

        P.row_pos, P.slot_mapping, P.seq_q_start, P.seq_kv_len, P.block_table = at(0), at(1), at(2), at(3), at(4)
        for k, a in self.host_only.items():
            setattr(P, k, a.ctypes.data_as(L.p_i32))
        pool = L.hb_page_pool(self.pool_arr.ctypes.data_as(L.p_i32), int(self.pool_arr.size), 0)
        st = self.lib.hb_plan_batch(self.dec, self.n_dec, self.pf, self.n_pf, C.byref(pool), self.tau, self.chunk, 16,
                                    C.byref(P))
        if st != 0:
            raise RuntimeError(f"hb_plan_batch failed: {self.lib.hb_last_error().decode()}")
        cs = self.copy_stream
        if self.k >= 2:
            cs.wait_event(self.released[b])  # the layer of step k - 2 has read dev[b]
        with torch.cuda.stream(cs):
            self.dev[b].copy_(self.pinned[b], non_blocking=True)
        self.copied[b].record(cs)
        stream.wait_event(self.copied[b])
        self.h2d_bytes = self.dev_ints * 4
        self.k += 1
        self.n_rows, self.n_seqs = P.n_rows, P.n_seqs
        d = self.dev[b].data_ptr()
        return L.hb_device_plan(P.n_rows, P.n_seqs, self.max_pages, *[d + 4 * int(self.off[i]) for i in range(5)],
                                P.decode_pairs, P.chunk_pairs, P.chunk_rows)

    def host_plan_arrays(self):
        s = self.pinned[(self.k - 1) & 1].numpy()
        T, S = self.n_rows, self.n_seqs
        return (s[self.off[0]:self.off[0] + T].copy(), s[self.off[2]:self.off[2] + S + 1].copy(),
                s[self.off[3]:self.off[3] + S].copy())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.QUERY}",
                                       "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            self.f.close()
            os.unlink(self.f.name)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        self.f.close()
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- CPU oracle
def oracle_iteration_rate(w, budget_s: float, min_iters: int = 1):
    """Time the oracle's full layer iteration on the same workload until
    `budget_s` seconds (at least `min_iters` iterations)."""
    import oracle.layer as ol
    import oracle.plan as op
    st = w.state
    args = ([r.done for r in st.decodes], [r.pages for r in st.decodes], [r.prompt_len for r in st.prefills],
            [r.done for r in st.prefills], [r.pages for r in st.prefills], st.free_pool, w.tau, w.chunk)
    max_pos = max(r.done for r in st.decodes + st.prefills) + w.tau + 1
    cos, sin = ol.rope_tables(max_pos, w.dims.d_head, w.dims.theta)
    k, v = st.k_pool, st.v_pool  # the append writes the same slots each iteration
    n, rows = 0, 0
    t0 = time.perf_counter()
    while True:
        p = op.plan_batch(*args)
        ol.layer_forward(w.weights[0], w.dims, p, w.x, k, v, cos, sin)
        n += 1
        rows += p.n_rows
        if n >= min_iters and time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return rows / dt, n, dt


def oracle_decode_sample_rate(w, n_rows: int):
    """Oracle on a sub-batch of the workload's first n_rows decodes."""
    import oracle.layer as ol
    import oracle.plan as op
    st = w.state
    dec = st.decodes[:n_rows]
    p = op.plan_batch([r.done for r in dec], [r.pages for r in dec], [], [], [], st.free_pool, w.tau, w.chunk)
    max_pos = max(r.done for r in dec) + 2
    cos, sin = ol.rope_tables(max_pos, w.dims.d_head, w.dims.theta)
    t0 = time.perf_counter()
    ol.layer_forward(w.weights[0], w.dims, p, w.x[:p.n_rows], st.k_pool, st.v_pool, cos, sin)
    return p.n_rows, time.perf_counter() - t0


def cores():
    return len(os.sched_getaffinity(0))


def workload_config(w, weights, world, T, n_dec):
    """The `config` of the bench line, the same for the GPU arm and the
    reference arm (T rows per iteration, n_dec of them decodes)."""
    dims = w.dims
    return {"workload": WORKLOAD + ("_e4m3" if weights == "e4m3" else ""), "tau": w.tau, "weights": weights,
            "chunk_tokens": T - n_dec, "decodes": n_dec, "rows": T, "d_model": dims.d_model,
            "heads": f"{dims.n_q}q/{dims.n_kv}kv", "d_head": dims.d_head, "d_ff": dims.d_ff, "page": 16,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "inputs larger than L2 (436 MB weights + 308 MB KV per step), no flush"}


# ---------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = make_workload(args.tau, args.decodes)
    n_steps = args.steps + args.warmup
    budget = max(0.05, 150.0 / n_steps)  # whole run within a few minutes
    rows_cal, t_cal = oracle_decode_sample_rate(w, 4)
    per_row = t_cal / rows_cal
    T = args.tau
    full = per_row * T <= budget
    n_rows = T if full else max(1, min(len(w.state.decodes), int(budget / per_row)))
    import oracle.layer as ol
    import oracle.plan as op
    st = w.state
    if full:
        args_p = ([r.done for r in st.decodes], [r.pages for r in st.decodes], [r.prompt_len for r in st.prefills],
                  [r.done for r in st.prefills], [r.pages for r in st.prefills], st.free_pool, w.tau, w.chunk)
        sample = f"full iteration of {T} rows per step"
    else:
        dec = st.decodes[:n_rows]
        args_p = ([r.done for r in dec], [r.pages for r in dec], [], [], [], st.free_pool, w.tau, w.chunk)
        sample = f"{n_rows} decode rows of the iteration per step (full context each)"
    max_pos = max(r.done for r in st.decodes + st.prefills) + w.tau + 1
    cos, sin = ol.rope_tables(max_pos, w.dims.d_head, w.dims.theta)

    def step():
        p = op.plan_batch(*args_p)
        ol.layer_forward(w.weights[0], w.dims, p, w.x[:p.n_rows], st.k_pool, st.v_pool, cos, sin)
        return p.n_rows

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    rows = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, args.weights, world, w.tau, len(st.decodes)),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def run_hb(args, world, rank, local):
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    from chunked_prefill_hybrid_tau_gb300 import costs
    from workloads import device as wd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = hb.lib()
    w = make_workload(args.tau, args.decodes)
    st, dims = w.state, w.dims
    max_pos = max(r.done for r in st.decodes + st.prefills) + w.tau + 1
    f8 = args.weights == "e4m3"
    gw = wd.layer_weights_device(w.weights[0], dims, dev, fmt=args.weights)
    kc, vc = wd.bf16_tensor(st.k_pool, dev), wd.bf16_tensor(st.v_pool, dev)
    rope = wd.rope_table_device(max_pos, dims, dev)
    x_dev = wd.bf16_tensor(w.x, dev)
    out_dev = torch.empty_like(x_dev)
    stream = torch.cuda.Stream(device=dev)
    runner = PlanRunner(lib, st, w.tau, w.chunk, dev)
    max_kv = max_pos
    ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, runner.row_cap, runner.seq_cap, max_kv), dev)
    ds = hb.dims_struct(dims)
    wstruct = gw.struct()
    n_events = 9
    prof_steps = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(prof_steps)]
    for row in ev:  # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    stream.synchronize()
    ev_arrays = [(C.c_void_p * n_events)(*[e.cuda_event for e in row]) for row in ev]
    from chunked_prefill_hybrid_tau_gb300 import _lib as L
    profs = [L.hb_profile(a, n_events) for a in ev_arrays]
    sptr = C.c_void_p(stream.cuda_stream)

    def layer(dplan, xin, xout, prof=None):
        rc = lib.hb_layer_forward(C.byref(wstruct), C.byref(ds), C.byref(dplan), C.c_void_p(rope.data_ptr()),
                                  max_pos, C.c_void_p(xin.data_ptr()), C.c_void_p(xout.data_ptr()),
                                  C.c_void_p(kc.data_ptr()), C.c_void_p(vc.data_ptr()), int(kc.shape[0]), max_kv,
                                  C.c_void_p(ws.data_ptr()), ws.numel(), sptr, C.byref(prof) if prof else None)
        if rc != 0:
            raise RuntimeError(f"hb_layer_forward: {lib.hb_last_error().decode()}")

    # ---- device-resident timing ------------------------------------------
    for _ in range(args.warmup):
        layer(runner.step(stream), x_dev, out_dev)
    stream.synchronize()
    hb.hb_check_status(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the clock sampler runs from here through the end-to-end pass
    clocks = ClockSampler(local)
    t_clock0 = time.perf_counter()
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = hb.hb_kernel_launches()
    start.record(stream)
    for _ in range(args.steps):
        layer(runner.step(stream), x_dev, out_dev)
    end.record(stream)
    launches = hb.hb_kernel_launches() - launches0  # this library's kernels in the timed region
    if launches != launches_per_layer(dims, f8, runner.n_rows) * args.steps:
        print(f"warning: {launches} kernels launched in the timed region, the library's rule says "
              f"{launches_per_layer(dims, f8, runner.n_rows) * args.steps}", file=sys.stderr)
    torch.cuda.synchronize(dev)
    barrier(world)
    hb.hb_check_status(stream)
    t_dev = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    T = runner.n_rows
    value = world * T * args.steps / t_dev

    # ---- per-stage breakdown (separate pass: events between the kernels
    # serialise them, so it is not part of the timed region) --------------
    for j in range(prof_steps):
        layer(runner.step(stream), x_dev, out_dev, profs[j])
    stream.synchronize()
    hb.hb_check_status(stream)

    stage_ms = np.zeros(8)
    for row in ev:
        for s in range(8):
            stage_ms[s] += row[s].elapsed_time(row[s + 1])
    stage_ms /= len(ev)

    # ---- end to end through the C ABI with host buffers ------------------
    # Every step uploads its input from pinned host memory and reads its
    # output back.  The copies run on their own streams with two device
    # buffers each way, so step i + 1's upload and step i's download overlap
    # step i's compute; a buffer is reused only after the step that last used
    # it (layer or copy) has finished with it.
    x_host = torch.from_numpy(wd.to_numpy(x_dev).astype(np.float32)).to(torch.bfloat16).pin_memory()
    out_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    x_in = [torch.empty_like(x_dev) for _ in range(2)]
    y_out = [torch.empty_like(x_dev) for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e_steps = max(1, args.steps)

    def e2e_run(n, e0=None):
        if n == 0:
            return
        uploaded, computed, fetched = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(3))
        if e0 is not None:
            up.wait_event(e0)
            down.wait_event(e0)

        def upload(i):
            b = i % 2
            if i >= 2:
                up.wait_event(computed[b])  # the layer of step i - 2 has read x_in[b]
            with torch.cuda.stream(up):
                x_in[b].copy_(x_host, non_blocking=True)
            uploaded[b].record(up)

        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(uploaded[b])
            if i >= 2:
                stream.wait_event(fetched[b])  # step i - 2's output has been read back
            layer(runner.step(stream), x_in[b], y_out[b])
            computed[b].record(stream)
            down.wait_event(computed[b])
            with torch.cuda.stream(down):
                out_host[b].copy_(y_out[b], non_blocking=True)
            fetched[b].record(down)
        stream.wait_event(fetched[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(fetched[(n - 2) % 2])

    # warm-up of the copy streams and pinned buffers, so the timed steps are
    # steady state (fill and drain of the copy pipeline are one step each)
    e2e_run(max(args.warmup, 10))
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    hb.hb_check_status(stream)
    # short runs: keep the layer running (untimed) until the sampler has seen
    # at least MIN_CLOCK_S of it, so the clock record is never empty
    while time.perf_counter() - t_clock0 < MIN_CLOCK_S:
        for _ in range(50):
            layer(runner.step(stream), x_dev, out_dev)
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    out_host = out_host[0]
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e = {"value": world * T * e_steps / t_e2e, "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_host.numel() * 2 + runner.h2d_bytes),
           "d2h_bytes_per_step": int(out_host.numel() * 2)}

    # ---- roofline --------------------------------------------------------
    peaks = load_peaks()
    row_pos, q_start, kv_len = runner.host_plan_arrays()
    sc = costs.stage_costs(dims, row_pos, q_start, kv_len, weight_bytes=1 if f8 else 2)
    flops, byts = costs.iteration_totals(sc)
    t_step = t_dev / args.steps
    t_roof = costs.roofline_time(sc, peaks["bf16_tflops"], peaks["hbm_gbs"], f8)
    dom = int(np.argmax(stage_ms))
    name = costs.STAGES[dom]
    f_dom, b_dom, bound = sc[name]
    dur = stage_ms[dom] / 1e3
    peak_source = peaks["source"] + " burst"
    if bound == "tensor":
        tensor_peak = peaks["bf16_tflops"] * (2.0 if f8 else 1.0)
        achieved, peak, unit = f_dom / dur / 1e12, tensor_peak, "TFLOP/s"
        if f8:
            peak_source += " x 2 (nominal FP8/bf16 dense ratio, 4.5/2.25 PFLOP/s)"
    else:
        achieved, peak, unit = b_dom / dur / 1e9, peaks["hbm_gbs"], "GB/s"
    traffic = None  # measured DRAM bytes per launch (ncu), when recorded for this kernel and workload
    prof_path = os.path.join(ROOT, "profiles", "traffic.txt")
    if os.path.exists(prof_path):
        entries = dict(ln.split(None, 1) for ln in open(prof_path).read().splitlines()
                       if ln.strip() and not ln.startswith("#"))
        if entries.get("workload", "").strip() == WORKLOAD and name in entries and not f8:
            traffic = float(entries[name])

    n_dec = sum(1 for r in st.decodes)
    c = T - n_dec
    s_bar = float(np.mean([r.done for r in st.decodes])) if n_dec else 0.0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 projections, bf16 attention" if f8 else "bf16", "data": "synthetic",
        "config": workload_config(w, args.weights, world, T, n_dec),
        "roofline": {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_source,
                     "launch_ms": stage_ms[dom]},
        "iteration_roofline": {"flops": flops, "bytes": byts, "t_roof_ms": 1e3 * t_roof,
                               "frac": t_roof / t_step, "intensity_flop_per_byte": flops / byts,
                               "intensity_page": costs.page_intensity(c, n_dec, dims.params_per_layer,
                                                                      1 if f8 else 2, 1, dims.n_kv, dims.d_head,
                                                                      s_bar)},
        "stages_ms": {k: round(float(v), 5) for k, v in zip(costs.STAGES, stage_ms)},
        "e2e": e2e,
        # counted by the library (per layer forward: row statistics, QKV, RoPE/KV
        # append, chunk and decode attention, O, gate/up, down; E4M3: three more
        # quantization kernels, RoPE/KV append inside the QKV projection when
        # its tiles hold whole heads), checked against its rule below
        "gpu_launches": launches,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt = oracle_iteration_rate(w, budget_s=10.0)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                                "sample": f"{n} full oracle iterations ({n * T} rows) in {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_sweep(args, taus=None, emit=True):
    """ms/iter, tokens/s and roofline fraction against the token budget on the
    Mistral-7B-shaped layer: 64 decodes with contexts uniform in [512, 8192]
    plus a chunk of c = tau - 64 tokens at offset 0 of an 8192-token prompt.
    Returns the per-tau records (and prints them as JSON lines if emit)."""
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    from chunked_prefill_hybrid_tau_gb300 import costs
    from workloads import device as wd
    lib = hb.lib()
    taus = taus or [64, 128, 256, 512, 1024, 2048, 4096]
    records = []
    w = make_workload(max(taus), 64)
    st, dims = w.state, w.dims
    max_pos = 8192 + max(taus) + 1
    f8 = args.weights == "e4m3"
    gw = wd.layer_weights_device(w.weights[0], dims, fmt=args.weights)
    kc, vc = wd.bf16_tensor(st.k_pool), wd.bf16_tensor(st.v_pool)
    rope = wd.rope_table_device(max_pos, dims)
    x_all = wd.bf16_tensor(w.x)
    peaks = load_peaks()
    s_bar = float(np.mean([r.done for r in st.decodes]))
    s_psi = 1 if f8 else 2  # bytes per weight
    balance = peaks["bf16_tflops"] * (2.0 if f8 else 1.0) * 1e12 / (peaks["hbm_gbs"] * 1e9)
    for tau in taus:
        stream = torch.cuda.Stream()
        runner = PlanRunner(lib, st, tau, tau, "cuda")
        ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, runner.row_cap, runner.seq_cap, max_pos))
        x = x_all[:tau].contiguous()
        out = torch.empty_like(x)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(9)]
        for e in ev:
            e.record(stream)
        arr = (C.c_void_p * 9)(*[e.cuda_event for e in ev])
        from chunked_prefill_hybrid_tau_gb300 import _lib as L
        prof = L.hb_profile(arr, 9)
        ds, wsr = hb.dims_struct(dims), gw.struct()

        def layer(dp, with_prof=False):
            rc = lib.hb_layer_forward(C.byref(wsr), C.byref(ds), C.byref(dp), C.c_void_p(rope.data_ptr()), max_pos,
                                      C.c_void_p(x.data_ptr()), C.c_void_p(out.data_ptr()), C.c_void_p(kc.data_ptr()),
                                      C.c_void_p(vc.data_ptr()), int(kc.shape[0]), max_pos, C.c_void_p(ws.data_ptr()),
                                      ws.numel(), C.c_void_p(stream.cuda_stream),
                                      C.byref(prof) if with_prof else None)
            if rc != 0:
                raise RuntimeError(lib.hb_last_error().decode())

        for _ in range(10):
            layer(runner.step(stream))
        steps = max(50, min(args.steps, 400))
        stage_ms = np.zeros(8)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        s0.record(stream)
        for _ in range(steps):
            layer(runner.step(stream))
        s1.record(stream)
        stream.synchronize()
        t_step = s0.elapsed_time(s1) / 1e3 / steps
        for _ in range(20):
            layer(runner.step(stream), with_prof=True)
            stream.synchronize()
            for s in range(8):
                stage_ms[s] += ev[s].elapsed_time(ev[s + 1]) / 20
        hb.hb_check_status(stream)
        row_pos, q_start, kv_len = runner.host_plan_arrays()
        sc = costs.stage_costs(dims, row_pos, q_start, kv_len, weight_bytes=s_psi)
        flops, byts = costs.iteration_totals(sc)
        t_roof = costs.roofline_time(sc, peaks["bf16_tflops"], peaks["hbm_gbs"], f8)
        T = runner.n_rows
        c = T - 64
        rec = {
            "sweep": "tau", "weights": args.weights, "tau": tau, "rows": T, "chunk_tokens": c, "decodes": 64, "ms_per_step": 1e3 * t_step,
            "tokens_per_s": T / t_step, "t_roof_ms": 1e3 * t_roof, "roofline_frac": t_roof / t_step,
            "flops": flops, "bytes": byts, "intensity_flop_per_byte": flops / byts,
            "intensity_page": costs.page_intensity(c, 64, dims.params_per_layer, s_psi, 1, dims.n_kv, dims.d_head,
                                                   s_bar),
            "stages_ms": {k: round(float(v), 5) for k, v in zip(costs.STAGES, stage_ms)}}
        records.append(rec)
        if emit:
            print(json.dumps(rec), flush=True)
    # the page's optimal chunk for this machine balance (I* = peak FLOP/s / peak B/s)
    psi = dims.params_per_layer
    c_star = balance / (2.0 * psi) * (s_psi * psi + 2.0 * dims.n_kv * dims.d_head * s_bar * 64) - 64
    cs = {"sweep": "c_star", "weights": args.weights, "machine_balance_flop_per_byte": balance, "c_star_tokens": c_star,
          "s_bar": s_bar}
    records.append(cs)
    if emit:
        print(json.dumps(cs), flush=True)
    return records


def select_tau(profile, slo_ms):
    """The pages' calibration rule (profile T(n), take the largest n with
    T(n) <= T*) on a measured profile [(tau, iteration_ms), ...] in
    increasing tau.  Returns (tau or None, knee) where the knee is the first
    tau whose time is 10% above the smallest budget's."""
    fits = [t for t, ms in profile if ms <= slo_ms]
    base = profile[0][1]
    knee = next((t for t, ms in profile if ms >= 1.1 * base), None)
    return (max(fits) if fits else None), knee


def run_calibrate(args):
    """The scheduling method's tau calibration (the Sarathi-Serve reading notes'
    profiling step): measure the iteration time T(tau) of a --layers-deep
    model (distinct random weights and KV pools per layer, the layers through
    one hb_layers_forward call; the same layers as hb_layer_forward calls
    are timed beside it) over a range of token budgets, then take the largest
    tau whose time fits the per-iteration SLO.  The batch at each tau is 64
    decodes with contexts uniform in [512, 8192] plus a chunk of tau - 64
    tokens.  Prints the profile and one summary line."""
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    from workloads import device as wd
    lib = hb.lib()
    taus = [64, 128, 192, 256, 384, 512, 640, 768, 1024, 1536, 2048, 3072, 4096]
    L = args.layers
    w = make_workload(max(taus), 64)
    st, dims = w.state, w.dims
    max_pos = 8192 + max(taus) + 1
    fmt = args.weights
    gen = wd.device_generator(77)
    layers = [wd.layer_weights_random(dims, 7700 + l, fmt=fmt) for l in range(L)]
    shape = (st.num_pages, dims.n_kv, 16, dims.d_head)
    pools = [(wd.randn_bf16(shape, gen), wd.randn_bf16(shape, gen)) for _ in range(L)]
    rope = wd.rope_table_device(max_pos, dims)
    x_all = wd.randn_bf16((max(taus), dims.d_model), gen)
    profile = []
    for tau in taus:
        stream = torch.cuda.Stream()
        runner = PlanRunner(lib, st, tau, tau, "cuda")
        ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, runner.row_cap, runner.seq_cap, max_pos))
        x = x_all[:tau].clone()
        ds = hb.dims_struct(dims)
        wstructs = [lw.struct() for lw in layers]
        warr = (type(wstructs[0]) * L)(*wstructs)
        karr = (C.c_void_p * L)(*[k.data_ptr() for k, _ in pools])
        varr = (C.c_void_p * L)(*[v.data_ptr() for _, v in pools])

        def iteration(stacked):
            dp = runner.step(stream)
            if stacked:  # the model's layers in one call (statistics carried between layers)
                rc = lib.hb_layers_forward(warr, L, C.byref(ds), C.byref(dp), C.c_void_p(rope.data_ptr()), max_pos,
                                           C.c_void_p(x.data_ptr()), C.c_void_p(x.data_ptr()), karr, varr,
                                           int(pools[0][0].shape[0]), max_pos, C.c_void_p(ws.data_ptr()), ws.numel(),
                                           C.c_void_p(stream.cuda_stream))
                if rc != 0:
                    raise RuntimeError(lib.hb_last_error().decode())
                return
            for l in range(L):
                k, v = pools[l]
                rc = lib.hb_layer_forward(C.byref(wstructs[l]), C.byref(ds), C.byref(dp), C.c_void_p(rope.data_ptr()),
                                          max_pos, C.c_void_p(x.data_ptr()), C.c_void_p(x.data_ptr()),
                                          C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()), int(k.shape[0]),
                                          max_pos, C.c_void_p(ws.data_ptr()), ws.numel(),
                                          C.c_void_p(stream.cuda_stream), None)
                if rc != 0:
                    raise RuntimeError(lib.hb_last_error().decode())

        def timed(stacked):
            for _ in range(3):
                iteration(stacked)
            stream.synchronize()
            n = max(5, min(args.steps, 20))
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(n):
                iteration(stacked)
            s1.record(stream)
            stream.synchronize()
            hb.hb_check_status(stream)
            return s0.elapsed_time(s1) / n

        ms = timed(True)
        ms_calls = timed(False)
        T = runner.n_rows
        profile.append((tau, ms))
        print(json.dumps({"calibrate": "profile", "weights": fmt, "layers": L, "tau": tau, "rows": T,
                          "iteration_ms": ms, "layer_ms": ms / L, "tokens_per_s": T / (ms / 1e3),
                          "layer_calls_ms": ms_calls}), flush=True)
        del ws
    c_star = [r for r in run_sweep(args, [64], emit=False) if r["sweep"] == "c_star"][0]
    tau, knee = select_tau(profile, args.calibrate)
    best = dict(profile).get(tau)
    print(json.dumps({"calibrate": "tau", "slo_ms": args.calibrate, "layers": L, "tau": tau, "iteration_ms": best,
                      "tau_knee_10pct": knee, "c_star_tokens": c_star["c_star_tokens"], "decodes": 64,
                      "weights": fmt}), flush=True)
    return 0


def run_chunk_study(args):
    """Prefill cost of chunking (the pages' chunk-size overhead claims): one
    prompt of P tokens through the Mistral-7B-shaped layer in chunks of C,
    every chunk attending to the KV the earlier chunks wrote, against one
    unchunked pass.  Time is the whole prefill, best of three."""
    import torch
    import chunked_prefill_hybrid_tau_gb300 as hb
    from workloads import device as wd
    import workloads as wl
    dims = wl.MISTRAL
    lw = wd.layer_weights_random(dims, 4100)
    gen = wd.device_generator(41)
    for P in (8192, 32768, 65536):
        x = wd.randn_bf16((P, dims.d_model), gen)
        out = torch.empty_like(x)
        rope = wd.rope_table_device(P + 1, dims)
        num_pages = P // 16 + 8
        kc = torch.zeros((num_pages, dims.n_kv, 16, dims.d_head), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        pool = list(range(num_pages))
        results = {}
        for C in [P, 2048, 1024, 512, 256, 128]:
            plans = []
            done, pages, fp = 0, [], pool
            while done < P:
                hp = hb.hb_plan_batch([], [], [P], [done], [pages], fp, C, C)
                pages, fp = hp.pf_pages[0], hp.free_pool
                plans.append((done, int(hp.pf_take[0]), hb.DevicePlan(hp)))
                done += int(hp.pf_take[0])
            ws = wd.workspace(hb.hb_layer_workspace_bytes(dims, C, 1, P))
            best = None
            for _ in range(3):
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                s0.record()
                for d0, t, dp in plans:
                    hb.hb_layer_forward(lw, dims, dp, rope, P + 1, x[d0:d0 + t], out[d0:d0 + t], kc, vc, P, ws)
                s1.record()
                torch.cuda.synchronize()
                ms = s0.elapsed_time(s1)
                best = ms if best is None else min(best, ms)
            hb.hb_check_status()
            results[C] = best
            print(json.dumps({"chunk_study": "prefill", "prompt": P, "chunk": C, "chunks": len(plans), "ms": best,
                              "tokens_per_s": P / (best / 1e3),
                              "overhead_vs_unchunked": best / results[P] - 1.0}), flush=True)
            del ws, plans
        del x, out, kc, vc
        torch.cuda.empty_cache()
    return 0


def main():
    args = parse()
    if args.sweep:
        run_sweep(args)
        return 0
    if args.calibrate is not None:
        return run_calibrate(args)
    if args.chunk_study:
        return run_chunk_study(args)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
    else:
        rc = run_hb(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
