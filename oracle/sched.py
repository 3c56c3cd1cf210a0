"""Oracle of the iteration driver (test infrastructure only).

The scheduling loop of the Sarathi-Serve reading notes (section 3.4, "the
whole scheduling algorithm") around the planner oracle: each iteration
packs every running decode and then prompt chunks from the FIFO of waiting
requests under the budget tau (plan.plan_batch).  After the iteration:

  * a decode has one more token in its cache and one more generated token;
  * a chunk has advanced its prompt; when the prompt is complete, its last
    row produced the first generated token and the request starts decoding,
    behind the decodes already running;
  * a request with all its new tokens generated is finished and its pages go
    back to the end of the free pool in page order.

Readings (the pages are silent): decodes run in the order their prompts
completed; within one iteration, decodes are advanced before chunks; the
last generated token is never written to the cache, so a request holds at
most ceil((prompt_len + max_new - 1) / P) pages.
"""
from __future__ import annotations

from collections import deque

from . import plan as op

PREFILLING, DECODING, FINISHED = 0, 1, 2


class SchedLoop:
    def __init__(self, tau, chunk, pool, page=16):
        self.tau, self.chunk, self.page = tau, chunk, page
        self.pool = list(pool)
        self.reqs = []          # dicts: prompt_len, max_new, cached, generated, state, pages
        self.waiting = deque()  # prefilling, FIFO
        self.running = []       # decoding, in order
        self.last = None

    def add(self, prompt_len, max_new):
        self.reqs.append(dict(prompt_len=prompt_len, max_new=max_new, cached=0, generated=0, state=PREFILLING,
                              pages=[]))
        self.waiting.append(len(self.reqs) - 1)
        return len(self.reqs) - 1

    def plan(self):
        """-> (Plan, row_req) for the next iteration (state advances on commit)."""
        dec = list(self.running)
        pf = list(self.waiting)
        p = op.plan_batch([self.reqs[i]["cached"] for i in dec], [self.reqs[i]["pages"] for i in dec],
                          [self.reqs[i]["prompt_len"] for i in pf], [self.reqs[i]["cached"] for i in pf],
                          [self.reqs[i]["pages"] for i in pf], self.pool, self.tau, self.chunk, self.page)
        row_req = [(dec if p.seq_kind[q] == 0 else pf)[p.seq_req[q]] for q in p.row_seq]
        self.last = (dec, pf, p)
        return p, row_req

    def commit(self):
        dec, pf, p = self.last
        for k, i in enumerate(dec):
            self.reqs[i]["pages"] = list(p.dec_pages[k])
        for k, i in enumerate(pf):
            self.reqs[i]["pages"] = list(p.pf_pages[k])
        self.pool = list(p.free_pool)

        def finish(r):
            r["state"] = FINISHED
            self.pool.extend(r["pages"])
            r["pages"] = []

        running = []
        for i in dec:
            r = self.reqs[i]
            r["cached"] += 1
            r["generated"] += 1
            if r["generated"] >= r["max_new"]:
                finish(r)
            else:
                running.append(i)
        waiting = deque()
        for k, i in enumerate(pf):
            r = self.reqs[i]
            r["cached"] += p.pf_take[k]
            if r["cached"] < r["prompt_len"]:
                waiting.append(i)
                continue
            r["generated"] = 1
            r["state"] = DECODING
            if r["generated"] >= r["max_new"]:
                finish(r)
            else:
                running.append(i)
        self.running, self.waiting, self.last = running, waiting, None

    def active(self):
        return len(self.waiting) + len(self.running)
