// builder.cpp -- the stall-free batch builder behind hb_builder_* (host only).
//
// Each step forms one hybrid batch in the order the first page gives
// ("Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §核心机制 2): every running decode first (one token each), then a
// chunk of every unfinished prefill, then first chunks of waiting requests,
// first come first served, until the token budget B is spent; the caller runs
// the batch and calls complete(), which advances each request along
// waiting -> prefill (chunked) -> decode -> done ("In-flight Batching",
// §调度状态机) and returns finished requests' pages to the pool
// (§KV Cache 管理的协同优化).  The last prefill chunk produces the first output
// token (first page, §GPU / 系统数据路径 ⑦), whose KV the first decode step
// appends.
//
// Readings where the pages are silent: a chunk takes min(prompt left, budget
// left) tokens; an ongoing chunk is cut to the pages that can be had;
// admission stops at the first request whose first chunk's pages cannot be
// allocated; pages come from the front of a FIFO free list and go back to its
// end in block-table order; a decode that finds no free page is an error (no
// preemption); decodes that alone exceed B are all kept, no prefill is added
// and the batch is flagged over budget.
#include <algorithm>
#include <cstring>
#include <deque>
#include <memory>
#include <string>
#include <unordered_map>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "hb.h"

namespace {

enum Phase { kWaiting = 0, kPrefill = 1, kDecode = 2, kDone = 3 };

struct Request {
  int64_t id;
  int32_t prompt_len, max_new;
  Phase phase = kWaiting;
  int32_t prefilled = 0, generated = 0;
  std::vector<int32_t> pages;
};

struct Row {
  Request* req;
  int32_t kind;       // 0 decode, 1 prefill
  int32_t q_len;
  int32_t context_len;
};

thread_local std::string t_berr;

hb_status berr(hb_status s, const std::string& m) {
  t_berr = m;
  return s;
}

}  // namespace

struct hb_builder {
  int32_t budget, page_size, num_pages, max_pages_per_seq;
  std::deque<int32_t> free_pages;
  std::deque<Request*> waiting;
  std::vector<Request*> running;  // admission order
  std::unordered_map<int64_t, std::unique_ptr<Request>> reqs;
  bool pending = false;
  std::vector<Row> last_rows;

  int32_t pages_for(int64_t tokens) const {
    return (int32_t)((tokens + page_size - 1) / page_size);
  }
};

// A named range on the profiler's host timeline (NVTX; a no-op unless a
// profiling tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

extern "C" {

// These entry points report messages through the same per-thread channel as
// the CUDA entry points would; hb_last_error() in api.cu owns that channel,
// so builder messages are kept in their own thread-local string and exposed
// through hb_builder_last_error() below.
const char* hb_builder_last_error(void) { return t_berr.c_str(); }

hb_status hb_builder_create(int32_t budget, int32_t page_size, int32_t num_pages,
                            int32_t max_pages_per_seq, const int32_t* page_order,
                            hb_builder** out) {
  if (!out) return berr(HB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (budget < 1 || page_size < 1 || num_pages < 0 || max_pages_per_seq < 1)
    return berr(HB_ERR_INVALID_ARG, "bad builder parameters");
  std::unique_ptr<hb_builder> b(new hb_builder());
  b->budget = budget;
  b->page_size = page_size;
  b->num_pages = num_pages;
  b->max_pages_per_seq = max_pages_per_seq;
  if (page_order) {
    std::vector<char> seen(num_pages, 0);
    for (int32_t i = 0; i < num_pages; ++i) {
      const int32_t p = page_order[i];
      if (p < 0 || p >= num_pages || seen[p]) return berr(HB_ERR_INVALID_ARG, "page_order is not a permutation");
      seen[p] = 1;
      b->free_pages.push_back(p);
    }
  } else {
    for (int32_t i = 0; i < num_pages; ++i) b->free_pages.push_back(i);
  }
  *out = b.release();
  return HB_OK;
}

void hb_builder_destroy(hb_builder* b) { delete b; }

hb_status hb_builder_add_request(hb_builder* b, int64_t id, int32_t prompt_len, int32_t max_new) {
  if (!b) return berr(HB_ERR_INVALID_ARG, "builder is NULL");
  if (prompt_len < 1 || max_new < 1) return berr(HB_ERR_SHAPE, "prompt_len and max_new must be >= 1");
  const int64_t longest = (int64_t)prompt_len + max_new - 1;
  if (b->pages_for(longest) > b->max_pages_per_seq)
    return berr(HB_ERR_SHAPE, "request does not fit max_pages_per_seq");
  if (b->reqs.count(id)) return berr(HB_ERR_INVALID_ARG, "duplicate request id");
  std::unique_ptr<Request> r(new Request());
  r->id = id;
  r->prompt_len = prompt_len;
  r->max_new = max_new;
  b->waiting.push_back(r.get());
  b->reqs.emplace(id, std::move(r));
  return HB_OK;
}

hb_status hb_builder_step(hb_builder* b, int32_t max_rows, int32_t* num_rows, int32_t* q_len,
                          int32_t* context_len, int32_t* block_table, int64_t* row_ids,
                          int32_t* row_kind, int32_t* over_budget) {
  NvtxRange range("hb_builder_step");
  if (!b || !num_rows || !over_budget) return berr(HB_ERR_INVALID_ARG, "NULL argument");
  if (b->pending) return berr(HB_ERR_INVALID_ARG, "complete the previous batch first");
  if (max_rows < 0) return berr(HB_ERR_INVALID_ARG, "max_rows < 0");

  // Pages are taken from the front of the free list as the batch is formed;
  // a failed step puts them back (front, original order) and shortens the
  // requests' page lists again, so it leaves the builder unchanged.  The
  // cost of a step is that of its rows, not of the pool.
  std::deque<int32_t>& free_pages = b->free_pages;
  std::vector<int32_t> taken;                    // pages taken, in order
  std::unordered_map<Request*, size_t> grown;   // request -> page count before
  std::vector<Row> rows;
  int64_t tokens = 0;
  auto grow = [&](Request* r, int64_t n_tokens) -> bool {
    const int32_t need = b->pages_for(n_tokens) - (int32_t)r->pages.size();
    if (need > (int32_t)free_pages.size()) return false;
    if (need > 0 && !grown.count(r)) grown[r] = r->pages.size();
    for (int32_t i = 0; i < need; ++i) {
      r->pages.push_back(free_pages.front());
      taken.push_back(free_pages.front());
      free_pages.pop_front();
    }
    return true;
  };
  auto rollback = [&]() {
    for (auto& kv : grown) kv.first->pages.resize(kv.second);
    for (auto it = taken.rbegin(); it != taken.rend(); ++it) free_pages.push_front(*it);
  };

  // 1. running decodes
  for (Request* r : b->running) {
    if (r->phase != kDecode) continue;
    const int32_t ctx = r->prompt_len + r->generated;
    if (!grow(r, ctx)) {
      rollback();
      return berr(HB_ERR_OUT_OF_PAGES, "no free page for a decode");
    }
    rows.push_back({r, 0, 1, ctx});
    tokens += 1;
  }
  const bool over = tokens > b->budget;
  // 2. unfinished prefills continue
  for (Request* r : b->running) {
    if (r->phase != kPrefill) continue;
    const int64_t left = b->budget - tokens;
    if (left <= 0) break;
    int64_t c = std::min<int64_t>(r->prompt_len - r->prefilled, left);
    const int64_t cap = ((int64_t)r->pages.size() + (int64_t)free_pages.size()) * b->page_size - r->prefilled;
    c = std::min(c, cap);
    if (c <= 0) continue;
    grow(r, r->prefilled + c);
    rows.push_back({r, 1, (int32_t)c, (int32_t)(r->prefilled + c)});
    tokens += c;
  }
  // 3. admissions, first come first served
  size_t admitted = 0;
  while (admitted < b->waiting.size() && b->budget - tokens > 0) {
    Request* r = b->waiting[admitted];
    const int64_t c = std::min<int64_t>(r->prompt_len, b->budget - tokens);
    if (b->pages_for(c) > (int32_t)free_pages.size()) break;
    grow(r, c);
    rows.push_back({r, 1, (int32_t)c, (int32_t)c});
    tokens += c;
    ++admitted;
  }
  if ((int64_t)rows.size() > max_rows) {
    rollback();
    *num_rows = (int32_t)rows.size();
    return berr(HB_ERR_WORKSPACE, "max_rows too small for this batch");
  }
  if (!rows.empty() && (!q_len || !context_len || !block_table || !row_ids || !row_kind)) {
    rollback();
    return berr(HB_ERR_INVALID_ARG, "NULL output array");
  }
  // commit
  for (size_t i = 0; i < admitted; ++i) {
    Request* r = b->waiting.front();
    b->waiting.pop_front();
    r->phase = kPrefill;
    b->running.push_back(r);
  }
  const int32_t mp = b->max_pages_per_seq;
  for (size_t i = 0; i < rows.size(); ++i) {
    const Row& w = rows[i];
    q_len[i] = w.q_len;
    context_len[i] = w.context_len;
    row_ids[i] = w.req->id;
    row_kind[i] = w.kind;
    int32_t* bt = block_table + i * (size_t)mp;
    for (int32_t k = 0; k < mp; ++k)
      bt[k] = k < (int32_t)w.req->pages.size() ? w.req->pages[k] : -1;
  }
  *num_rows = (int32_t)rows.size();
  *over_budget = over ? 1 : 0;
  b->last_rows = rows;
  b->pending = !rows.empty();
  return HB_OK;
}

hb_status hb_builder_complete(hb_builder* b, int32_t max_finished, int32_t* num_finished,
                              int64_t* finished_ids) {
  NvtxRange range("hb_builder_complete");
  if (!b || !num_finished) return berr(HB_ERR_INVALID_ARG, "NULL argument");
  if (!b->pending) return berr(HB_ERR_INVALID_ARG, "no batch to complete");
  std::vector<Request*> done;
  for (const Row& w : b->last_rows) {
    Request* r = w.req;
    if (w.kind == 1) {
      r->prefilled += w.q_len;
      if (r->prefilled == r->prompt_len) {
        r->phase = kDecode;
        r->generated = 1;
      }
    } else {
      r->generated += 1;
    }
    if (r->phase == kDecode && r->generated >= r->max_new) done.push_back(r);
  }
  int32_t n = 0;
  for (Request* r : done) {
    r->phase = kDone;
    b->running.erase(std::find(b->running.begin(), b->running.end(), r));
    for (int32_t p : r->pages) b->free_pages.push_back(p);
    r->pages.clear();
    if (finished_ids && n < max_finished) finished_ids[n] = r->id;
    ++n;
  }
  *num_finished = n;
  b->pending = false;
  b->last_rows.clear();
  return HB_OK;
}

hb_status hb_builder_counts(const hb_builder* b, int32_t* waiting, int32_t* running,
                            int32_t* free_pages) {
  if (!b) return berr(HB_ERR_INVALID_ARG, "builder is NULL");
  if (waiting) *waiting = (int32_t)b->waiting.size();
  if (running) *running = (int32_t)b->running.size();
  if (free_pages) *free_pages = (int32_t)b->free_pages.size();
  return HB_OK;
}

hb_status hb_builder_free_list(const hb_builder* b, int32_t max, int32_t* n, int32_t* pages) {
  if (!b || !n) return berr(HB_ERR_INVALID_ARG, "NULL argument");
  *n = (int32_t)b->free_pages.size();
  for (int32_t i = 0; i < max && i < *n; ++i) pages[i] = b->free_pages[i];
  return HB_OK;
}

}  // extern "C"
