"""Oracle of the hybrid-batch planner (test infrastructure only).

Follows the scheduling loop of the Sarathi-Serve reading notes (section 3.4,
"the whole scheduling algorithm"; section 3.2 stall-free hybrid batching):
every active decode contributes one token first; then, while the token count
n is below the budget tau and the prefill queue has requests, the next
request contributes take = min(chunk_size_for(r), tau - n) prompt tokens,
chunk_size_for(r) being C or the smaller remainder at the prompt's end.

Readings where the pages are silent or ambiguous:
  * at most one chunk per request per iteration, walking the FIFO in order
    (the worked example of section 7.6 moves on to R_B after one chunk of R_A);
  * take = min(prompt_len - done, C, tau - n); partial chunks are allowed;
  * b > tau: all decodes are admitted, no prefill, over_budget = 1;
  * pages (16 tokens) are allocated on demand, decode rows first, then chunk
    rows in position order, popped from the front of a FIFO free pool; a row
    at position p needs page index p // P of its request;
  * slot of a row = page_id * P + p % P.
"""
from __future__ import annotations

import dataclasses


class OutOfPages(Exception):
    pass


@dataclasses.dataclass
class Plan:
    row_seq: list
    row_pos: list
    slot_mapping: list
    seq_q_start: list
    seq_pos0: list
    seq_kv_len: list
    seq_kind: list          # 0 = decode, 1 = prefill chunk
    seq_req: list           # index into decodes (kind 0) or prefills (kind 1)
    block_table: list       # per sequence, page ids padded with -1 to max_pages
    max_pages: int
    pf_take: list
    pf_finished: list
    dec_pages: list         # page lists after allocation
    pf_pages: list
    free_pool: list         # remaining FIFO
    pages_used: int
    over_budget: int

    @property
    def n_rows(self) -> int:
        return len(self.row_seq)

    @property
    def n_seqs(self) -> int:
        return len(self.seq_pos0)


def plan_batch(dec_ctx, dec_pages, pf_len, pf_done, pf_pages, free_pool, tau, chunk,
               page=16, max_pages=None) -> Plan:
    """Pack one hybrid iteration.

    dec_ctx[i]  : tokens cached for decode i (its new token sits at that position)
    dec_pages[i]: page ids it holds
    pf_len[j], pf_done[j], pf_pages[j]: prompt length, tokens prefilled, pages held
    free_pool   : FIFO of free page ids
    """
    dec_pages = [list(p) for p in dec_pages]
    pf_pages = [list(p) for p in pf_pages]
    pool = list(free_pool)
    used = 0

    def need_page(pages, pos):
        nonlocal used
        while len(pages) <= pos // page:
            if used >= len(pool):
                raise OutOfPages(f"needed more than {len(pool)} free pages")
            pages.append(pool[used])
            used += 1

    row_seq, row_pos, slot = [], [], []
    q_start, pos0, kv_len, kind, req = [0], [], [], [], []
    seq_pages = []

    # 1. every active decode contributes one token
    for i, ctx in enumerate(dec_ctx):
        s = len(pos0)
        need_page(dec_pages[i], ctx)
        row_seq.append(s)
        row_pos.append(ctx)
        slot.append(dec_pages[i][ctx // page] * page + ctx % page)
        pos0.append(ctx)
        kv_len.append(ctx + 1)
        kind.append(0)
        req.append(i)
        q_start.append(len(row_seq))
        seq_pages.append(dec_pages[i])
    n = len(dec_ctx)
    over = 1 if n > tau else 0

    # 2. fill the remaining budget with prompt chunks, FIFO order, one chunk each
    take_out = [0] * len(pf_len)
    fin_out = [0] * len(pf_len)
    for j in range(len(pf_len)):
        if n >= tau:
            break
        remaining = min(chunk, pf_len[j] - pf_done[j])
        take = min(remaining, tau - n)
        if take <= 0:
            continue
        s = len(pos0)
        for t in range(take):
            p = pf_done[j] + t
            need_page(pf_pages[j], p)
            row_seq.append(s)
            row_pos.append(p)
            slot.append(pf_pages[j][p // page] * page + p % page)
        pos0.append(pf_done[j])
        kv_len.append(pf_done[j] + take)
        kind.append(1)
        req.append(j)
        q_start.append(len(row_seq))
        seq_pages.append(pf_pages[j])
        n += take
        take_out[j] = take
        fin_out[j] = 1 if pf_done[j] + take == pf_len[j] else 0

    need = max([(kl + page - 1) // page for kl in kv_len], default=0)
    mp = need if max_pages is None else max_pages
    if mp < need:
        raise ValueError("max_pages too small")
    table = []
    for s, pg in enumerate(seq_pages):
        n_used = (kv_len[s] + page - 1) // page
        table.append(list(pg[:n_used]) + [-1] * (mp - n_used))
    return Plan(row_seq, row_pos, slot, q_start, pos0, kv_len, kind, req, table, mp,
                take_out, fin_out, dec_pages, pf_pages, pool[used:], used, over)
