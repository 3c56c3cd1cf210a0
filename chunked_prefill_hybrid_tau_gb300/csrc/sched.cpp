// hb_sched: the iteration driver of the scheduling loop (host).
//
// The loop of the Sarathi-Serve reading notes (section 3.4, "the whole
// scheduling algorithm"): every iteration admits all running decodes, then
// fills the token budget tau with prompt chunks from the FIFO of waiting
// requests (hb_plan_batch packs it); after the iteration's forward, each
// decode has one more token in the cache, each chunk has advanced its
// prompt, a prompt whose last chunk ran starts decoding (that chunk's last
// row produced the first new token), and a request with all its new tokens
// generated is finished and returns its pages to the back of the free pool.
// Requests that are still prefilling keep their FIFO order; decodes run in
// the order their prompts completed.  There is no preemption: running out of
// pages is an error (KV-cache management is orthogonal to the method,
// section 3.5).
#include <cstdint>
#include <deque>
#include <memory>
#include <new>
#include <vector>

#include "common.h"

struct hb_sched {
  struct Req {
    int32_t prompt_len, max_new, generated, state;  // state: 0 prefilling, 1 decoding, 2 finished
    std::vector<int32_t> pages;                      // capacity for the whole request
    hb_request view;                                 // planner view (done = cached tokens)
  };
  int32_t tau, chunk, page;
  std::vector<Req> reqs;
  std::deque<int32_t> waiting;  // prefilling, FIFO
  std::vector<int32_t> running; // decoding, in order
  std::deque<int32_t> pool;     // free pages, FIFO
  // the planned iteration, applied by hb_sched_commit
  bool planned = false;
  std::vector<int32_t> plan_dec, plan_pf, plan_take;
  std::vector<int32_t> pool_buf;
};

namespace {
constexpr int32_t kPrefilling = 0, kDecoding = 1, kFinished = 2;
}

extern "C" hb_status hb_sched_create(int32_t tau, int32_t chunk, int32_t page_size, const int32_t* pages,
                                     int32_t n_pages, hb_sched** out) {
  hb::clear_error();
  HB_REQUIRE(out != nullptr, "hb_sched_create: null output");
  HB_REQUIRE(tau >= 1 && chunk >= 1 && page_size >= 1, "hb_sched_create: tau, chunk, page_size must be >= 1");
  HB_REQUIRE(n_pages >= 0 && (n_pages == 0 || pages != nullptr), "hb_sched_create: bad page pool");
  for (int32_t i = 0; i < n_pages; ++i) HB_REQUIRE(pages[i] >= 0, "hb_sched_create: negative page id");
  hb_sched* s = new (std::nothrow) hb_sched();
  HB_REQUIRE(s != nullptr, "hb_sched_create: out of host memory");
  s->tau = tau;
  s->chunk = chunk;
  s->page = page_size;
  s->pool.assign(pages, pages + n_pages);
  *out = s;
  return HB_OK;
}

extern "C" void hb_sched_destroy(hb_sched* s) { delete s; }

extern "C" hb_status hb_sched_add(hb_sched* s, int32_t prompt_len, int32_t max_new, int32_t* id) {
  hb::clear_error();
  HB_REQUIRE(s != nullptr && id != nullptr, "hb_sched_add: null argument");
  HB_REQUIRE(prompt_len >= 1 && max_new >= 1, "hb_sched_add: prompt_len and max_new must be >= 1");
  HB_REQUIRE(!s->planned, "hb_sched_add: an iteration is planned and not committed");
  hb_sched::Req r;
  r.prompt_len = prompt_len;
  r.max_new = max_new;
  r.generated = 0;
  r.state = kPrefilling;
  // the last token generated is never written to the cache
  const int64_t tokens = static_cast<int64_t>(prompt_len) + max_new - 1;
  r.pages.assign(static_cast<size_t>((tokens + s->page - 1) / s->page), 0);
  r.view = hb_request{prompt_len, 0, 0, static_cast<int32_t>(r.pages.size()), nullptr};
  s->reqs.push_back(std::move(r));
  *id = static_cast<int32_t>(s->reqs.size() - 1);
  s->waiting.push_back(*id);
  return HB_OK;
}

extern "C" hb_status hb_sched_plan(hb_sched* s, hb_plan* plan, int32_t* row_req) {
  hb::clear_error();
  HB_REQUIRE(s != nullptr && plan != nullptr, "hb_sched_plan: null argument");
  HB_REQUIRE(!s->planned, "hb_sched_plan: the previous iteration is not committed");
  std::vector<hb_request> dec, pf;
  dec.reserve(s->running.size());
  pf.reserve(s->waiting.size());
  for (int32_t id : s->running) {
    hb_sched::Req& r = s->reqs[id];
    r.view.pages = r.pages.data();
    dec.push_back(r.view);
  }
  for (int32_t id : s->waiting) {
    hb_sched::Req& r = s->reqs[id];
    r.view.pages = r.pages.data();
    pf.push_back(r.view);
  }
  s->pool_buf.assign(s->pool.begin(), s->pool.end());
  hb_page_pool pool{s->pool_buf.data(), static_cast<int32_t>(s->pool_buf.size()), 0};
  hb_status st = hb_plan_batch(dec.data(), static_cast<int32_t>(dec.size()), pf.data(),
                               static_cast<int32_t>(pf.size()), &pool, s->tau, s->chunk, s->page, plan);
  if (st != HB_OK) return st;  // nothing changed: the planner leaves its inputs untouched on error
  // pages taken from the pool; each request's page count as the planner left it
  s->pool.erase(s->pool.begin(), s->pool.begin() + pool.head);
  for (size_t i = 0; i < dec.size(); ++i) s->reqs[s->running[i]].view.n_pages = dec[i].n_pages;
  for (size_t j = 0; j < pf.size(); ++j) s->reqs[s->waiting[j]].view.n_pages = pf[j].n_pages;
  s->plan_dec.assign(s->running.begin(), s->running.end());
  s->plan_pf.assign(s->waiting.begin(), s->waiting.end());
  s->plan_take.assign(plan->pf_take, plan->pf_take + pf.size());
  if (row_req != nullptr) {
    for (int32_t row = 0; row < plan->n_rows; ++row) {
      const int32_t q = plan->row_seq[row];
      row_req[row] = plan->seq_kind[q] == 0 ? s->plan_dec[plan->seq_req[q]] : s->plan_pf[plan->seq_req[q]];
    }
  }
  s->planned = true;
  return HB_OK;
}

extern "C" hb_status hb_sched_commit(hb_sched* s) {
  hb::clear_error();
  HB_REQUIRE(s != nullptr, "hb_sched_commit: null scheduler");
  HB_REQUIRE(s->planned, "hb_sched_commit: no planned iteration");
  auto finish = [&](hb_sched::Req& r) {
    r.state = kFinished;
    for (int32_t k = 0; k < r.view.n_pages; ++k) s->pool.push_back(r.pages[k]);
    r.view.n_pages = 0;
  };
  // decodes: the newest token is now cached, and one more token is out
  std::vector<int32_t> running;
  for (int32_t id : s->plan_dec) {
    hb_sched::Req& r = s->reqs[id];
    r.view.done += 1;
    r.generated += 1;
    if (r.generated >= r.max_new)
      finish(r);
    else
      running.push_back(id);
  }
  // chunks: prompts advance; a completed prompt produced its first token
  std::deque<int32_t> waiting;
  for (size_t j = 0; j < s->plan_pf.size(); ++j) {
    const int32_t id = s->plan_pf[j];
    hb_sched::Req& r = s->reqs[id];
    r.view.done += s->plan_take[j];
    if (r.view.done < r.prompt_len) {
      waiting.push_back(id);
      continue;
    }
    r.generated = 1;
    r.state = kDecoding;
    if (r.generated >= r.max_new)
      finish(r);
    else
      running.push_back(id);
  }
  // requests added after the plan are not in plan_pf (adding is refused while planned)
  s->running.swap(running);
  s->waiting.swap(waiting);
  s->planned = false;
  return HB_OK;
}

extern "C" hb_status hb_sched_info(const hb_sched* s, int32_t id, int32_t* state, int32_t* cached,
                                   int32_t* generated, int32_t* n_pages) {
  hb::clear_error();
  HB_REQUIRE(s != nullptr, "hb_sched_info: null scheduler");
  HB_REQUIRE(id >= 0 && id < static_cast<int32_t>(s->reqs.size()), "hb_sched_info: unknown request %d", id);
  const hb_sched::Req& r = s->reqs[id];
  if (state) *state = r.state;
  if (cached) *cached = r.view.done;
  if (generated) *generated = r.generated;
  if (n_pages) *n_pages = r.view.n_pages;
  return HB_OK;
}

extern "C" int32_t hb_sched_active(const hb_sched* s) {
  return s ? static_cast<int32_t>(s->waiting.size() + s->running.size()) : 0;
}

extern "C" int32_t hb_sched_free_pages(const hb_sched* s) { return s ? static_cast<int32_t>(s->pool.size()) : 0; }
