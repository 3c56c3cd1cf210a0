"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module draws random numbers and lays out request state; it contains none
of the method's arithmetic (no normalisation, projection, rotation, attention
or packing).  Both the CPU oracle (through the tests and the bench) and the
GPU path receive exactly the arrays built here.

Value conventions (the configurations of the hybrid-iteration workloads):
  * weights ~ N(0, 0.02), activations ~ N(0, 1), cached K/V ~ N(0, 1),
    RMSNorm gains = 1, all rounded once to bf16 (round-to-nearest-even) so
    both sides see identical bf16-representable values;
  * decode context lengths uniform (or log-uniform) in a range, integers;
  * the KV page pool is a seeded random permutation of page ids, so block
    tables are non-contiguous.

The shapes stand in for the pages' workloads (production chat and
summarisation traces with median prompts of 1730 and 7059 tokens, reading
notes on Sarathi-Serve, section 4.1), which are not available here.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PAGE = 16


# ----------------------------------------------------------------------------
# bf16 rounding (input preparation only)
# ----------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16-representable float32."""
    out = np.array(x, dtype=np.float32, copy=True)
    bf16_round_(out)
    return out


_CHUNK = 1 << 22


def bf16_round_(x: np.ndarray) -> np.ndarray:
    """In-place round-to-nearest-even of a contiguous float32 array to bf16 values."""
    u = x.reshape(-1).view(np.uint32)
    tmp = np.empty(min(u.size, _CHUNK), np.uint32)
    for i in range(0, u.size, _CHUNK):
        c = u[i:i + _CHUNK]
        t = tmp[:c.size]
        np.right_shift(c, 16, out=t)
        np.bitwise_and(t, 1, out=t)
        t += np.uint32(0x7FFF)
        c += t
        c &= np.uint32(0xFFFF0000)
    return x


def normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) samples rounded to bf16, generated in place chunk by chunk."""
    out = np.empty(shape, np.float32)
    flat = out.reshape(-1)
    for i in range(0, flat.size, _CHUNK):
        c = flat[i:i + _CHUNK]
        rng.standard_normal(out=c, dtype=np.float32)
        if scale != 1.0:
            c *= np.float32(scale)
    return bf16_round_(out)


# ----------------------------------------------------------------------------
# shapes
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Dims:
    d_model: int
    n_q: int
    n_kv: int
    d_head: int
    d_ff: int
    page: int = PAGE
    eps: float = 1e-6
    theta: float = 1e4
    n_layers: int = 1
    vocab: int = 0

    @property
    def qkv_cols(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.d_head

    @property
    def params_per_layer(self) -> int:
        d, dh = self.d_model, self.d_head
        return d * self.qkv_cols + self.n_q * dh * d + 3 * d * self.d_ff


TINY = Dims(d_model=256, n_q=4, n_kv=2, d_head=64, d_ff=688, theta=1e4)
MISTRAL = Dims(d_model=4096, n_q=32, n_kv=8, d_head=128, d_ff=14336, theta=1e6)
MISTRAL_32L = dataclasses.replace(MISTRAL, n_layers=32, vocab=32000)
YI34B = Dims(d_model=7168, n_q=56, n_kv=8, d_head=128, d_ff=20480, theta=5e6, n_layers=60)


# ----------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------
def layer_weights(rng: np.random.Generator, dims: Dims, gamma_jitter: float = 0.0) -> dict:
    """One decoder layer's weights (float32 arrays holding bf16 values).

    w_qkv [ (n_q + 2 n_kv) d_head, d ]   rows: q heads, then k heads, then v heads
    w_o   [ d, n_q d_head ]
    w_g   [ d_ff, d ],  w_u [ d_ff, d ],  w_d [ d, d_ff ]
    g1, g2 [ d ]  RMSNorm gains (1, or 1 + N(0, gamma_jitter) for unit tests)
    """
    d, f = dims.d_model, dims.d_ff

    def normal(*shape):
        return normal_bf16(rng, shape, 0.02)

    def gain():
        g = np.ones(d, np.float32)
        if gamma_jitter:
            g = g + rng.standard_normal(d, dtype=np.float32) * np.float32(gamma_jitter)
        return bf16_round(g)

    return dict(
        w_qkv=normal(dims.qkv_cols, d),
        w_o=normal(d, dims.n_q * dims.d_head),
        w_g=normal(f, d),
        w_u=normal(f, d),
        w_d=normal(d, f),
        g1=gain(),
        g2=gain(),
    )


def activations(rng: np.random.Generator, rows: int, d: int) -> np.ndarray:
    return normal_bf16(rng, (rows, d))


# ----------------------------------------------------------------------------
# request state and the paged KV pool
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Request:
    """Host-side request state.  `done` = tokens whose KV is already cached
    (the context length of a decode; the prefilled count of a prompt)."""
    done: int
    prompt_len: int = 0
    pages: list = dataclasses.field(default_factory=list)


@dataclasses.dataclass
class State:
    dims: Dims
    decodes: list
    prefills: list
    free_pool: list           # FIFO of free page ids (front = next to pop)
    num_pages: int
    k_pool: np.ndarray        # [num_pages, n_kv, page, d_head] float32 (bf16 values)
    v_pool: np.ndarray


def pages_for(tokens: int, page: int = PAGE) -> int:
    return (tokens + page - 1) // page


def make_state(rng: np.random.Generator, dims: Dims, dec_ctx, prefills, slack_pages: int,
               random_prefix: bool = True, fill_kv: bool = True) -> State:
    """Allocate pages for every token already cached and fill them.

    dec_ctx   : context lengths of the decodes (tokens already cached)
    prefills  : list of (prompt_len, done)
    slack_pages: free pages left in the pool after the prior allocation
    random_prefix: fill a prefill's cached prefix with N(0,1) (True) or leave
                   it zero for the caller to compute (False)
    fill_kv   : False leaves the pools zero-filled and unallocated in memory
                (shapes only), for callers that fill on the device
    """
    need = sum(pages_for(c, dims.page) for c in dec_ctx)
    need += sum(pages_for(d, dims.page) for _, d in prefills)
    num_pages = need + slack_pages
    perm = [int(p) for p in rng.permutation(num_pages)]
    decodes = []
    head = 0
    for c in dec_ctx:
        n = pages_for(int(c), dims.page)
        decodes.append(Request(done=int(c), pages=perm[head:head + n]))
        head += n
    pfs = []
    for L, d in prefills:
        n = pages_for(int(d), dims.page)
        pfs.append(Request(done=int(d), prompt_len=int(L), pages=perm[head:head + n]))
        head += n
    shape = (num_pages, dims.n_kv, dims.page, dims.d_head)
    if not fill_kv:
        return State(dims, decodes, pfs, perm[head:], num_pages, None, None)
    k_pool = np.zeros(shape, np.float32)
    v_pool = np.zeros(shape, np.float32)

    def fill(req):
        n = req.done
        if n == 0:
            return
        k = normal_bf16(rng, (n, dims.n_kv, dims.d_head))
        v = normal_bf16(rng, (n, dims.n_kv, dims.d_head))
        t = np.arange(n)
        pg = np.asarray(req.pages)[t // dims.page]
        off = t % dims.page
        k_pool[pg, :, off, :] = k
        v_pool[pg, :, off, :] = v

    for r in decodes:
        fill(r)
    if random_prefix:
        for r in pfs:
            fill(r)
    return State(dims, decodes, pfs, perm[head:], num_pages, k_pool, v_pool)


# ----------------------------------------------------------------------------
# the configurations
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    dims: Dims
    tau: int
    chunk: int
    state: State
    x: np.ndarray              # [T, d] hidden states of this iteration's rows
    weights: list              # per layer dicts
    notes: str = ""


def tiny_layer(seed: int = 0) -> Workload:
    """Tiny decoder layer: d=256, 4 q / 2 kv heads, d_head 64, FFN 688, theta 1e4.

    One 64-token chunk at positions 128..191 of a 256-token prompt whose first
    128 tokens are cached, plus 4 decodes (contexts 32, 77, 150, 200) with
    random prior KV.  The cached prefix is *computed* from the prompt's first
    128 input rows (a first iteration), so `x_prompt` holds all 256 prompt rows
    and `x` holds this iteration's 68 rows (4 decode rows, then the chunk).
    """
    rng = np.random.default_rng(seed)
    dims = TINY
    w = layer_weights(rng, dims)
    st = make_state(rng, dims, [32, 77, 150, 200], [(256, 0)], slack_pages=64, random_prefix=False)
    x_prompt = activations(rng, 256, dims.d_model)
    x_dec = activations(rng, 4, dims.d_model)
    wl = Workload("tiny_layer_T68", dims, tau=68, chunk=64, state=st,
                  x=np.concatenate([x_dec, x_prompt[128:192]]), weights=[w])
    wl.x_prompt = x_prompt
    return wl


def mistral_layer(seed: int = 0, tau: int = 512, n_dec: int = 32, ctx_lo: int = 512,
                  ctx_hi: int = 4096, prompt_len: int = 4096, offset: int = 1024,
                  fill_kv: bool = True, make_weights: bool = True) -> Workload:
    """Mistral-7B-shaped layer (d 4096, 32 q / 8 kv heads, d_head 128, FFN 14336,
    theta 1e6).  Default: tau=512, one 480-token chunk at offset 1024 of a
    4096-token prompt + 32 decodes with contexts uniform in [512, 4096]."""
    rng = np.random.default_rng(seed)
    dims = MISTRAL
    w = layer_weights(rng, dims) if make_weights else None
    ctx = rng.integers(ctx_lo, ctx_hi, size=n_dec, endpoint=True)
    c = tau - n_dec
    slack = pages_for(c + 16, dims.page) + n_dec + 8
    st = make_state(rng, dims, [int(v) for v in ctx], [(prompt_len, offset)], slack_pages=slack,
                    fill_kv=fill_kv)
    x = activations(rng, tau, dims.d_model)
    return Workload(f"mistral7b_layer_tau{tau}", dims, tau=tau, chunk=tau, state=st, x=x,
                    weights=[w])


def rng_for(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def log_uniform_ints(rng: np.random.Generator, lo: int, hi: int, n: int) -> np.ndarray:
    v = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    return np.clip(np.rint(v).astype(np.int64), lo, hi)
