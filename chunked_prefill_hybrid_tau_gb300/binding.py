"""Thin Python binding of the C ABI (include/hb.h): argument marshalling only.

Every function carries the name of the C entry point it calls.  Device
buffers are torch tensors (torch provides device memory and streams); host
arrays are numpy arrays or Python lists.  A non-OK status raises HBError with
the library's message.  There is no fallback: if libhb.so cannot be built or
loaded, the first call raises.
"""
from __future__ import annotations

import ctypes as C
import dataclasses

import numpy as np

from . import _lib as L


class HBError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib():
    return L.load()


def _check(status: int, name: str):
    if status != L.HB_OK:
        lb = lib()
        raise HBError(status, f"{name}: {lb.hb_status_string(status).decode()}: {lb.hb_last_error().decode()}")


def _stream(stream):
    import torch
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _p(t):
    """Device pointer of a tensor (None -> NULL)."""
    return None if t is None else C.c_void_p(t.data_ptr())


def dims_struct(dims) -> L.hb_layer_dims:
    return L.hb_layer_dims(int(dims.d_model), int(dims.n_q), int(dims.n_kv), int(dims.d_head), int(dims.d_ff),
                           int(getattr(dims, "page", 16)), float(dims.eps), float(dims.theta))


def hb_version() -> int:
    return int(lib().hb_version())


def hb_device_info():
    n = C.c_int32()
    s = C.c_int32()
    _check(lib().hb_device_info(C.byref(n), C.byref(s)), "hb_device_info")
    return int(n.value), bool(s.value)


def hb_kernel_launches() -> int:
    return int(lib().hb_kernel_launches())


def hb_check_status(stream=None):
    _check(lib().hb_check_status(_stream(stream)), "hb_check_status")


def hb_selftest_wait_timeout(timeout_us: int, stream=None):
    _check(lib().hb_selftest_wait_timeout(int(timeout_us), _stream(stream)), "hb_selftest_wait_timeout")


# ---------------------------------------------------------------- planner
@dataclasses.dataclass
class HostPlan:
    row_seq: np.ndarray
    row_pos: np.ndarray
    slot_mapping: np.ndarray
    seq_q_start: np.ndarray
    seq_pos0: np.ndarray
    seq_kv_len: np.ndarray
    seq_kind: np.ndarray
    seq_req: np.ndarray
    block_table: np.ndarray      # [n_seqs, max_pages]
    pf_take: np.ndarray
    pf_finished: np.ndarray
    dec_pages: list
    pf_pages: list
    free_pool: list
    pages_used: int
    over_budget: int
    decode_pairs: int = 0        # scheduling hints (include/hb.h, hb_plan)
    chunk_pairs: int = 0
    chunk_rows: int = 0

    @property
    def n_rows(self) -> int:
        return int(self.row_seq.shape[0])

    @property
    def n_seqs(self) -> int:
        return int(self.seq_pos0.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def hb_plan_batch(dec_ctx, dec_pages, pf_len, pf_done, pf_pages, free_pool, tau, chunk, page_size=16,
                  max_pages=None) -> HostPlan:
    """Pack one hybrid iteration (see hb_plan_batch in include/hb.h).  Inputs
    are not modified; the returned plan carries the updated page lists and
    the remaining free pool."""
    n_dec, n_pf = len(dec_ctx), len(pf_len)
    grow = tau // page_size + 2
    bufs = []
    reqs_d = (L.hb_request * max(n_dec, 1))()
    reqs_p = (L.hb_request * max(n_pf, 1))()
    for i in range(n_dec):
        b = np.zeros(len(dec_pages[i]) + grow, np.int32)
        b[:len(dec_pages[i])] = dec_pages[i]
        bufs.append(b)
        reqs_d[i] = L.hb_request(0, int(dec_ctx[i]), len(dec_pages[i]), b.size, b.ctypes.data_as(L.p_i32))
    for j in range(n_pf):
        b = np.zeros(len(pf_pages[j]) + grow, np.int32)
        b[:len(pf_pages[j])] = pf_pages[j]
        bufs.append(b)
        reqs_p[j] = L.hb_request(int(pf_len[j]), int(pf_done[j]), len(pf_pages[j]), b.size,
                                 b.ctypes.data_as(L.p_i32))
    pool_arr = np.ascontiguousarray(np.asarray(free_pool, np.int32))
    rows_cap = max(tau, n_dec, 1)
    seq_cap = max(n_dec + n_pf, 1)
    if max_pages is None:
        spans = [c + 1 for c in dec_ctx] + [d + min(chunk, tau) for d in pf_done]
        max_pages = max([(s + page_size - 1) // page_size for s in spans], default=1)
    for _attempt in range(2):
        out = {k: np.zeros(rows_cap, np.int32) for k in ("row_seq", "row_pos", "slot_mapping")}
        out.update({k: np.zeros(seq_cap, np.int32) for k in ("seq_pos0", "seq_kv_len", "seq_kind", "seq_req")})
        out["seq_q_start"] = np.zeros(seq_cap + 1, np.int32)
        out["block_table"] = np.zeros(seq_cap * max_pages, np.int32)
        out["pf_take"] = np.zeros(max(n_pf, 1), np.int32)
        out["pf_finished"] = np.zeros(max(n_pf, 1), np.int32)
        P = L.hb_plan()
        P.row_cap, P.seq_cap, P.max_pages, P.pf_cap = rows_cap, seq_cap, max_pages, n_pf
        for k in ("row_seq", "row_pos", "slot_mapping", "seq_q_start", "seq_pos0", "seq_kv_len", "seq_kind",
                  "seq_req", "block_table", "pf_take", "pf_finished"):
            setattr(P, k, out[k].ctypes.data_as(L.p_i32))
        pool = L.hb_page_pool(pool_arr.ctypes.data_as(L.p_i32), int(pool_arr.size), 0)
        st = lib().hb_plan_batch(reqs_d, n_dec, reqs_p, n_pf, C.byref(pool), int(tau), int(chunk), int(page_size),
                                 C.byref(P))
        if st == L.HB_ERR_CAPACITY:
            rows_cap, seq_cap, max_pages = P.need_rows, P.need_seqs, P.need_max_pages
            continue
        _check(st, "hb_plan_batch")
        T, S = P.n_rows, P.n_seqs
        return HostPlan(
            row_seq=out["row_seq"][:T].copy(), row_pos=out["row_pos"][:T].copy(),
            slot_mapping=out["slot_mapping"][:T].copy(), seq_q_start=out["seq_q_start"][:S + 1].copy(),
            seq_pos0=out["seq_pos0"][:S].copy(), seq_kv_len=out["seq_kv_len"][:S].copy(),
            seq_kind=out["seq_kind"][:S].copy(), seq_req=out["seq_req"][:S].copy(),
            block_table=out["block_table"][:S * max_pages].reshape(S, max_pages).copy(),
            pf_take=out["pf_take"][:n_pf].copy(), pf_finished=out["pf_finished"][:n_pf].copy(),
            dec_pages=[list(bufs[i][:reqs_d[i].n_pages]) for i in range(n_dec)],
            pf_pages=[list(bufs[n_dec + j][:reqs_p[j].n_pages]) for j in range(n_pf)],
            free_pool=[int(v) for v in pool_arr[pool.head:]], pages_used=int(P.pages_used),
            over_budget=int(P.over_budget), decode_pairs=int(P.decode_pairs), chunk_pairs=int(P.chunk_pairs),
            chunk_rows=int(P.chunk_rows))
    raise HBError(L.HB_ERR_CAPACITY, "hb_plan_batch: capacity retry failed")


# ---------------------------------------------------------------- iteration driver
class Scheduler:
    """The scheduling loop around the planner (include/hb.h, hb_sched):
    add requests, then per iteration plan() -> run the forward -> commit()."""

    def __init__(self, tau, chunk, pool, page_size=16):
        self._lib = lib()
        self.h = C.c_void_p()
        arr = np.ascontiguousarray(np.asarray(pool, np.int32))
        _check(self._lib.hb_sched_create(int(tau), int(chunk), int(page_size), arr.ctypes.data_as(L.p_i32),
                                         int(arr.size), C.byref(self.h)), "hb_sched_create")
        self.tau, self.chunk = int(tau), int(chunk)
        self.caps = [max(int(tau), 1), 16, 16, 16]  # rows, seqs, max_pages, prefills

    def close(self):
        if self.h:
            self._lib.hb_sched_destroy(self.h)
            self.h = C.c_void_p()

    def __del__(self):
        self.close()

    def add(self, prompt_len, max_new) -> int:
        rid = C.c_int32()
        _check(self._lib.hb_sched_add(self.h, int(prompt_len), int(max_new), C.byref(rid)), "hb_sched_add")
        return int(rid.value)

    def plan(self):
        """-> (HostPlan, row_req): the next iteration and each row's request id."""
        for _attempt in range(4):
            rc, sc, mp, pc = self.caps
            out = {k: np.zeros(rc, np.int32) for k in ("row_seq", "row_pos", "slot_mapping")}
            out.update({k: np.zeros(sc, np.int32) for k in ("seq_pos0", "seq_kv_len", "seq_kind", "seq_req")})
            out["seq_q_start"] = np.zeros(sc + 1, np.int32)
            out["block_table"] = np.zeros(sc * mp, np.int32)
            out["pf_take"] = np.zeros(pc, np.int32)
            out["pf_finished"] = np.zeros(pc, np.int32)
            row_req = np.zeros(rc, np.int32)
            P = L.hb_plan()
            P.row_cap, P.seq_cap, P.max_pages, P.pf_cap = rc, sc, mp, pc
            for k, a in out.items():
                setattr(P, k, a.ctypes.data_as(L.p_i32))
            st = self._lib.hb_sched_plan(self.h, C.byref(P), row_req.ctypes.data_as(L.p_i32))
            if st == L.HB_ERR_CAPACITY:
                self.caps = [max(rc, P.need_rows), max(sc, P.need_seqs), max(mp, P.need_max_pages),
                             max(pc, 2 * pc)]
                continue
            _check(st, "hb_sched_plan")
            T, S = P.n_rows, P.n_seqs
            n_pf = int(np.count_nonzero(out["seq_kind"][:S] == 1))
            hp = HostPlan(
                row_seq=out["row_seq"][:T].copy(), row_pos=out["row_pos"][:T].copy(),
                slot_mapping=out["slot_mapping"][:T].copy(), seq_q_start=out["seq_q_start"][:S + 1].copy(),
                seq_pos0=out["seq_pos0"][:S].copy(), seq_kv_len=out["seq_kv_len"][:S].copy(),
                seq_kind=out["seq_kind"][:S].copy(), seq_req=out["seq_req"][:S].copy(),
                block_table=out["block_table"][:S * mp].reshape(S, mp).copy(),
                pf_take=out["pf_take"][:pc].copy(), pf_finished=out["pf_finished"][:pc].copy(),
                dec_pages=[], pf_pages=[], free_pool=[], pages_used=int(P.pages_used),
                over_budget=int(P.over_budget), decode_pairs=int(P.decode_pairs), chunk_pairs=int(P.chunk_pairs),
                chunk_rows=int(P.chunk_rows))
            del n_pf
            return hp, row_req[:T].copy()
        raise HBError(L.HB_ERR_CAPACITY, "hb_sched_plan: capacity retry failed")

    def commit(self):
        _check(self._lib.hb_sched_commit(self.h), "hb_sched_commit")

    def info(self, rid):
        v = [C.c_int32() for _ in range(4)]
        _check(self._lib.hb_sched_info(self.h, int(rid), *[C.byref(x) for x in v]), "hb_sched_info")
        return tuple(int(x.value) for x in v)  # state, cached, generated, pages

    def active(self) -> int:
        return int(self._lib.hb_sched_active(self.h))

    def free_pages(self) -> int:
        return int(self._lib.hb_sched_free_pages(self.h))


# ---------------------------------------------------------------- device plan
class DevicePlan:
    """Device copy of a plan's kernel-facing arrays in one int32 buffer
    (uploaded with a single host-to-device copy)."""

    FIELDS = ("row_pos", "slot_mapping", "seq_q_start", "seq_kv_len", "block_table")

    def __init__(self, hp: HostPlan, device="cuda", stream=None, pinned=True):
        import torch
        parts = [np.ascontiguousarray(getattr(hp, f), np.int32).ravel() for f in self.FIELDS]
        self.offsets = np.cumsum([0] + [p.size for p in parts])
        host = np.concatenate(parts)
        self.host = torch.from_numpy(host)
        if pinned:
            self.host = self.host.pin_memory()
        self.dev = torch.empty(host.size, dtype=torch.int32, device=device)
        self.n_rows, self.n_seqs, self.max_pages = hp.n_rows, hp.n_seqs, hp.max_pages
        self.hints = (int(hp.decode_pairs), int(hp.chunk_pairs), int(hp.chunk_rows))
        self.h2d_bytes = int(host.size * 4)
        self.upload(stream)

    def upload(self, stream=None):
        import torch
        if stream is None:
            self.dev.copy_(self.host, non_blocking=True)
        else:
            with torch.cuda.stream(stream):
                self.dev.copy_(self.host, non_blocking=True)

    def field(self, name):
        i = self.FIELDS.index(name)
        return self.dev[self.offsets[i]:self.offsets[i + 1]]

    def struct(self) -> L.hb_device_plan:
        base = self.dev.data_ptr()
        ptr = [base + 4 * int(self.offsets[i]) for i in range(len(self.FIELDS))]
        return L.hb_device_plan(self.n_rows, self.n_seqs, self.max_pages, *ptr, *self.hints)


# ---------------------------------------------------------------- device ops
def hb_rope_table(table, max_pos, d_head, theta, stream=None):
    _check(lib().hb_rope_table(_p(table), int(max_pos), int(d_head), float(theta), _stream(stream)), "hb_rope_table")


def hb_rmsnorm(x, gamma, y, eps, stream=None):
    rows, d = x.shape
    _check(lib().hb_rmsnorm(_p(x), _p(gamma), _p(y), rows, d, float(eps), _stream(stream)), "hb_rmsnorm")


def hb_kv_append(qkv, row_pos, slot_mapping, rope, max_pos, dims, q_out, k_cache, v_cache, stream=None):
    ds = dims_struct(dims)
    _check(lib().hb_kv_append(_p(qkv), int(qkv.shape[0]), _p(row_pos), _p(slot_mapping), _p(rope), int(max_pos),
                              C.byref(ds), _p(q_out), _p(k_cache), _p(v_cache), int(k_cache.shape[0]),
                              _stream(stream)), "hb_kv_append")


def hb_attention_workspace_bytes(dims, max_rows, max_seqs, max_kv_len) -> int:
    ds = dims_struct(dims)
    return int(lib().hb_attention_workspace_bytes(C.byref(ds), int(max_rows), int(max_seqs), int(max_kv_len)))


def hb_attention(q, k_cache, v_cache, dplan: DevicePlan, dims, max_kv_len, out, workspace, stream=None):
    ds = dims_struct(dims)
    ps = dplan.struct()
    _check(lib().hb_attention(_p(q), _p(k_cache), _p(v_cache), int(k_cache.shape[0]), C.byref(ps), C.byref(ds),
                              int(max_kv_len), _p(out), _p(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream)), "hb_attention")


def hb_gemm(A, B, Cout, R=None, epilogue=L.HB_EPI_STORE, stream=None):
    M, K = A.shape
    N = B.shape[0]
    _check(lib().hb_gemm(_p(A), _p(B), _p(Cout), _p(R), M, N, K, int(epilogue), _stream(stream)), "hb_gemm")


def hb_gemm_e4m3(A, s_a, B, s_b, Cout, R=None, epilogue=L.HB_EPI_STORE, stream=None):
    """E4M3 codes A [M][K], B [N][K] (uint8 tensors) with fp32 per-row scales."""
    M, K = A.shape
    N = B.shape[0]
    _check(lib().hb_gemm_e4m3(_p(A), _p(s_a), _p(B), _p(s_b), _p(Cout), _p(R), M, N, K, int(epilogue),
                              _stream(stream)), "hb_gemm_e4m3")


def hb_quantize_e4m3(x, q=None, scale=None, stream=None):
    """Per-row E4M3 codes (uint8 [rows][cols]) and fp32 scales [rows] of a
    device bf16 matrix x; returns (q, scale)."""
    import torch
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device) if q is None else q
    scale = torch.empty(max(rows, 4), dtype=torch.float32, device=x.device) if scale is None else scale
    _check(lib().hb_quantize_e4m3(_p(x), _p(q), _p(scale), rows, cols, _stream(stream)), "hb_quantize_e4m3")
    return q, scale[:rows]


def hb_interleave_gate_up(w_gate, w_up, w_gu, stream=None):
    F, d = w_gate.shape
    _check(lib().hb_interleave_gate_up(_p(w_gate), _p(w_up), _p(w_gu), F, d, _stream(stream)),
           "hb_interleave_gate_up")


def hb_fold_gamma(w, gamma, out=None, stream=None):
    """out = bf16(w * gamma) column-wise (in place when out is None)."""
    rows, cols = w.shape
    out = w if out is None else out
    _check(lib().hb_fold_gamma(_p(w), _p(gamma), _p(out), rows, cols, _stream(stream)), "hb_fold_gamma")
    return out


def prepare_layer_weights(w_qkv, w_o, w_g, w_u, w_d, g1, g2, stream=None, fmt="bf16") -> "LayerWeights":
    """Raw device bf16 weights of one layer -> the prepared form that
    hb_layer_forward takes: g1 folded into W_qkv, gate/up interleaved and g2
    folded into them (include/hb.h, hb_layer_weights).  w_qkv is folded in
    place; w_g and w_u are left as they are.  fmt="e4m3": each prepared
    matrix is then quantized per row (hb_quantize_e4m3) and the bf16 forms
    are released."""
    import torch
    F, d = w_g.shape
    f_pad = (F + 63) // 64 * 64
    w_gu = torch.empty((2 * f_pad, d), dtype=torch.bfloat16, device=w_g.device)
    hb_interleave_gate_up(w_g, w_u, w_gu, stream)
    hb_fold_gamma(w_gu, g2, stream=stream)
    hb_fold_gamma(w_qkv, g1, stream=stream)
    if fmt == "bf16":
        return LayerWeights(w_qkv=w_qkv, w_o=w_o, w_gu=w_gu, w_d=w_d)
    if fmt != "e4m3":
        raise ValueError(f"unknown weight format {fmt!r}")
    q = {k: hb_quantize_e4m3(v, stream=stream) for k, v in
         (("qkv", w_qkv), ("o", w_o), ("gu", w_gu), ("d", w_d))}
    return LayerWeights(w_qkv=q["qkv"][0], w_o=q["o"][0], w_gu=q["gu"][0], w_d=q["d"][0], s_qkv=q["qkv"][1],
                        s_o=q["o"][1], s_gu=q["gu"][1], s_d=q["d"][1], fmt="e4m3")


def hb_layer_workspace_bytes(dims, max_rows, max_seqs, max_kv_len) -> int:
    ds = dims_struct(dims)
    return int(lib().hb_layer_workspace_bytes(C.byref(ds), int(max_rows), int(max_seqs), int(max_kv_len)))


def hb_layer_kernel_count(dims, n_rows, fmt) -> int:
    ds = dims_struct(dims)
    n = C.c_int32()
    _check(lib().hb_layer_kernel_count(C.byref(ds), int(n_rows), int(fmt), C.byref(n)), "hb_layer_kernel_count")
    return int(n.value)


@dataclasses.dataclass
class LayerWeights:
    """Prepared device weights of one layer (prepare_layer_weights): bf16
    tensors, or E4M3 codes (uint8) with fp32 per-row scales."""
    w_qkv: object
    w_o: object
    w_gu: object
    w_d: object
    s_qkv: object = None
    s_o: object = None
    s_gu: object = None
    s_d: object = None
    fmt: str = "bf16"

    def struct(self) -> L.hb_layer_weights:
        ptrs = [self.__dict__[k].data_ptr() for k in ("w_qkv", "w_o", "w_gu", "w_d")]
        if self.fmt == "e4m3":
            scales = [self.__dict__[k].data_ptr() for k in ("s_qkv", "s_o", "s_gu", "s_d")]
            return L.hb_layer_weights(*ptrs, *scales, L.HB_WEIGHTS_E4M3)
        return L.hb_layer_weights(*ptrs, None, None, None, None, L.HB_WEIGHTS_BF16)


def hb_layer_forward(w: LayerWeights, dims, dplan: DevicePlan, rope, max_pos, x_in, x_out, k_cache, v_cache,
                     max_kv_len, workspace, stream=None, events=None):
    ds = dims_struct(dims)
    ws = w.struct()
    ps = dplan.struct()
    prof = None
    if events is not None:
        for e in events:  # torch creates the CUDA event lazily, on first record
            if e.cuda_event == 0:
                e.record()
        arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
        prof = L.hb_profile(arr, len(events))
    _check(lib().hb_layer_forward(C.byref(ws), C.byref(ds), C.byref(ps), _p(rope), int(max_pos), _p(x_in), _p(x_out),
                                  _p(k_cache), _p(v_cache), int(k_cache.shape[0]), int(max_kv_len), _p(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream),
                                  C.byref(prof) if prof is not None else None), "hb_layer_forward")


def hb_layers_forward(ws_list, dims, dplan: DevicePlan, rope, max_pos, x_in, x_out, k_caches, v_caches, max_kv_len,
                      workspace, stream=None):
    """Layers back to back: ws_list[l] with k_caches[l], v_caches[l]."""
    n = len(ws_list)
    assert len(k_caches) == n and len(v_caches) == n
    ds = dims_struct(dims)
    ps = dplan.struct()
    warr = (L.hb_layer_weights * max(n, 1))(*[w.struct() for w in ws_list])
    karr = (C.c_void_p * max(n, 1))(*[k.data_ptr() for k in k_caches])
    varr = (C.c_void_p * max(n, 1))(*[v.data_ptr() for v in v_caches])
    num_pages = int(k_caches[0].shape[0]) if n else 1
    _check(lib().hb_layers_forward(warr, n, C.byref(ds), C.byref(ps), _p(rope), int(max_pos), _p(x_in), _p(x_out),
                                   karr, varr, num_pages, int(max_kv_len), _p(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "hb_layers_forward")


def hb_final_logits(x, rows, g_f, w_lm, logits, workspace, eps, stream=None):
    T, d = x.shape
    vocab = w_lm.shape[0]
    _check(lib().hb_final_logits(_p(x), T, _p(rows), int(rows.numel()), _p(g_f), _p(w_lm), vocab, d, float(eps),
                                 _p(logits), _p(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "hb_final_logits")
