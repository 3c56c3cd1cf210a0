// hb_plan_batch: token-budget packing of one hybrid iteration (host).
//
// The scheduling loop of the Sarathi-Serve reading notes (section 3.4) with
// stall-free hybrid batching (section 3.2): decodes first, then prompt chunks
// from the FIFO until the budget tau is reached, at most one chunk per request
// per iteration.  Pages of the paged KV cache are allocated on demand from the
// front of a FIFO free pool, decode rows first, then chunk rows in position
// order.  Two passes: the first only sizes (so that an error leaves every
// input untouched), the second writes.
#include <algorithm>

#include "common.h"

namespace {

inline int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }

// Tokens prefill j contributes this iteration, given n tokens already packed.
inline int32_t take_for(const hb_request& r, int32_t n, int32_t tau, int32_t chunk) {
  if (n >= tau) return 0;
  int32_t remaining = std::min(chunk, r.prompt_len - r.done);
  return std::max(0, std::min(remaining, tau - n));
}

// Pages a request must gain so that position `last` has a page.
inline int32_t pages_missing(const hb_request& r, int32_t last, int32_t page) {
  return std::max(0, last / page + 1 - r.n_pages);
}

}  // namespace

extern "C" hb_status hb_plan_batch(hb_request* decodes, int32_t n_dec, hb_request* prefills, int32_t n_pf,
                                   hb_page_pool* pool, int32_t tau, int32_t chunk, int32_t page_size,
                                   hb_plan* plan) {
  hb::clear_error();
  HB_REQUIRE(plan != nullptr && pool != nullptr, "hb_plan_batch: null plan or pool");
  HB_REQUIRE(n_dec >= 0 && n_pf >= 0, "hb_plan_batch: negative request count");
  HB_REQUIRE(n_dec == 0 || decodes != nullptr, "hb_plan_batch: null decodes");
  HB_REQUIRE(n_pf == 0 || prefills != nullptr, "hb_plan_batch: null prefills");
  HB_REQUIRE(tau >= 1 && chunk >= 1 && page_size >= 1, "hb_plan_batch: tau, chunk, page_size must be >= 1");
  HB_REQUIRE(pool->count >= 0 && pool->head >= 0 && pool->head <= pool->count &&
                 (pool->count == 0 || pool->pages != nullptr),
             "hb_plan_batch: inconsistent page pool");
  for (int32_t i = 0; i < n_dec + n_pf; ++i) {
    const hb_request& r = i < n_dec ? decodes[i] : prefills[i - n_dec];
    const bool is_pf = i >= n_dec;
    HB_REQUIRE(r.done >= 0 && r.n_pages >= 0 && r.page_cap >= r.n_pages, "hb_plan_batch: request %d: bad sizes", i);
    HB_REQUIRE(r.n_pages == 0 || r.pages != nullptr, "hb_plan_batch: request %d: null pages", i);
    HB_REQUIRE(r.n_pages >= ceil_div(r.done, page_size),
               "hb_plan_batch: request %d holds %d pages for %d cached tokens", i, r.n_pages, r.done);
    if (is_pf) HB_REQUIRE(r.done < r.prompt_len, "hb_plan_batch: prefill %d: done >= prompt_len", i - n_dec);
    for (int32_t k = 0; k < r.n_pages; ++k)
      HB_REQUIRE(r.pages[k] >= 0, "hb_plan_batch: request %d: negative page id", i);
  }

  // ---- pass 1: sizes -------------------------------------------------------
  int32_t rows = n_dec, seqs = n_dec, pages = 0, width = 0;
  bool page_cap_ok = true;
  for (int32_t i = 0; i < n_dec; ++i) {
    const hb_request& r = decodes[i];
    int32_t miss = pages_missing(r, r.done, page_size);
    pages += miss;
    page_cap_ok &= r.n_pages + miss <= r.page_cap;
    width = std::max(width, ceil_div(r.done + 1, page_size));
  }
  int32_t n = n_dec;
  for (int32_t j = 0; j < n_pf; ++j) {
    const hb_request& r = prefills[j];
    int32_t t = take_for(r, n, tau, chunk);
    if (t == 0) continue;
    n += t;
    rows += t;
    seqs += 1;
    int32_t miss = pages_missing(r, r.done + t - 1, page_size);
    pages += miss;
    page_cap_ok &= r.n_pages + miss <= r.page_cap;
    width = std::max(width, ceil_div(r.done + t, page_size));
  }
  plan->need_rows = rows;
  plan->need_seqs = seqs;
  plan->need_max_pages = width;
  plan->need_pages = pages;
  plan->n_rows = plan->n_seqs = plan->n_decode_seqs = plan->pages_used = 0;
  plan->decode_pairs = plan->chunk_pairs = plan->chunk_rows = 0;
  plan->over_budget = n_dec > tau ? 1 : 0;

  if (pool->count - pool->head < pages) {
    hb::set_error("hb_plan_batch: %d pages needed, %d free", pages, pool->count - pool->head);
    return HB_ERR_OUT_OF_PAGES;
  }
  if (rows > plan->row_cap || seqs > plan->seq_cap || width > plan->max_pages || n_pf > plan->pf_cap ||
      !page_cap_ok) {
    hb::set_error("hb_plan_batch: capacity too small (rows %d/%d, seqs %d/%d, max_pages %d/%d, prefills %d/%d%s)",
                  rows, plan->row_cap, seqs, plan->seq_cap, width, plan->max_pages, n_pf, plan->pf_cap,
                  page_cap_ok ? "" : ", a request's page_cap");
    return HB_ERR_CAPACITY;
  }
  HB_REQUIRE(plan->row_seq && plan->row_pos && plan->slot_mapping && plan->seq_q_start && plan->seq_pos0 &&
                 plan->seq_kv_len && plan->seq_kind && plan->seq_req && plan->block_table &&
                 (n_pf == 0 || (plan->pf_take && plan->pf_finished)),
             "hb_plan_batch: null output array");

  // ---- pass 2: write -------------------------------------------------------
  int32_t head = pool->head;
  auto need_page = [&](hb_request& r, int32_t pos) {
    while (r.n_pages <= pos / page_size) r.pages[r.n_pages++] = pool->pages[head++];
  };
  int32_t row = 0, s = 0;
  auto open_seq = [&](hb_request& r, int32_t pos0, int32_t q_len, int32_t kind, int32_t req) {
    plan->seq_q_start[s] = row;
    plan->seq_pos0[s] = pos0;
    plan->seq_kv_len[s] = pos0 + q_len;
    plan->seq_kind[s] = kind;
    plan->seq_req[s] = req;
    for (int32_t t = 0; t < q_len; ++t) {
      int32_t p = pos0 + t;
      need_page(r, p);
      plan->row_seq[row] = s;
      plan->row_pos[row] = p;
      plan->slot_mapping[row] = r.pages[p / page_size] * page_size + p % page_size;
      ++row;
    }
    // a row at position p sees p + 1 keys: sum over p in [pos0, pos0 + q_len)
    const int64_t pairs = static_cast<int64_t>(q_len) * pos0 + static_cast<int64_t>(q_len) * (q_len + 1) / 2;
    if (q_len == 1) {
      plan->decode_pairs += pairs;
    } else {
      plan->chunk_pairs += pairs;
      plan->chunk_rows += q_len;
    }
    int32_t used = ceil_div(pos0 + q_len, page_size);
    int32_t* bt = plan->block_table + static_cast<int64_t>(s) * plan->max_pages;
    for (int32_t k = 0; k < plan->max_pages; ++k) bt[k] = k < used ? r.pages[k] : -1;
    ++s;
  };
  for (int32_t i = 0; i < n_dec; ++i) open_seq(decodes[i], decodes[i].done, 1, 0, i);
  n = n_dec;
  for (int32_t j = 0; j < n_pf; ++j) {
    hb_request& r = prefills[j];
    int32_t t = take_for(r, n, tau, chunk);
    plan->pf_take[j] = t;
    plan->pf_finished[j] = (t > 0 && r.done + t == r.prompt_len) ? 1 : 0;
    if (t == 0) continue;
    n += t;
    open_seq(r, r.done, t, 1, j);
  }
  plan->seq_q_start[s] = row;
  plan->n_rows = row;
  plan->n_seqs = s;
  plan->n_decode_seqs = n_dec;
  plan->pages_used = head - pool->head;
  pool->head = head;
  return HB_OK;
}
