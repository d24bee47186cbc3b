// Host-side admission control and lazy page assignment for the shared KV
// page pool; the contract is in include/pkv_sched.h. Plain C++17, no CUDA.
//
// Credits and pages are kept apart, as the pages' engine does: `credits_`
// is what active requests have not reserved, the free heap holds physical
// page ids nobody owns. Invariant: for every active request, assigned pages
// <= budget, so free pages >= the reserved-but-unassigned remainder and
// extend() can always be served.

#include <algorithm>
#include <deque>
#include <functional>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_sched.h"

namespace {

struct Request {
  int prompt_tokens = 0;
  int prefix = 0;             // largest length it may reach
  int64_t budget = 0;         // credits it reserves
  bool active = false;
  bool waited = false;
  int pages_per_layer = 0;    // pages assigned in each layer
  std::vector<int32_t> pages; // [num_layers][max_pages_per_seq], first pages_per_layer valid
};

bool config_ok(const pkv_sched_config* c) {
  return c && c->num_layers >= 1 && c->num_pages >= 1 && c->page_size >= 1 &&
         c->max_seq_len >= c->page_size && c->max_seq_len % c->page_size == 0 &&
         (c->static_batching == 0 || c->static_batching == 1);
}

pkv_status budget_of(const pkv_sched_config& c, int prompt, int max_new, int* allowed,
                     int* prefix, int64_t* budget) {
  if (prompt < 1 || prompt >= c.max_seq_len || max_new < 1) return PKV_ERR_INVALID_ARG;
  const int n = std::min(max_new, c.max_seq_len - prompt);
  const int pre = prompt + n - 1;
  const int64_t per_layer = (pre + c.page_size - 1) / c.page_size;
  if (allowed) *allowed = n;
  if (prefix) *prefix = pre;
  if (budget) *budget = per_layer * c.num_layers;
  return PKV_OK;
}

}  // namespace

struct pkv_sched {
  pkv_sched_config cfg;
  int max_pages_per_seq;
  std::mutex lock;
  std::vector<int32_t> free_heap;     // min-heap of free page ids
  int64_t credits;
  std::deque<int> queue;              // waiting, FIFO
  std::vector<int> active;            // admitted, in admission order
  std::unordered_map<int, Request> requests;
  int next_id = 0;
  pkv_sched_stats stats{};

  int64_t assigned() const { return cfg.num_pages - static_cast<int64_t>(free_heap.size()); }

  int32_t take_page() {
    std::pop_heap(free_heap.begin(), free_heap.end(), std::greater<int32_t>());
    const int32_t p = free_heap.back();
    free_heap.pop_back();
    return p;
  }

  void give_page(int32_t p) {
    free_heap.push_back(p);
    std::push_heap(free_heap.begin(), free_heap.end(), std::greater<int32_t>());
  }
};

extern "C" {

pkv_status pkv_sched_budget(const pkv_sched_config* config, int prompt_tokens,
                            int max_new_tokens, int* allowed_new_tokens, int* prefix_tokens,
                            int64_t* budget_pages) {
  if (!config_ok(config)) return PKV_ERR_INVALID_ARG;
  return budget_of(*config, prompt_tokens, max_new_tokens, allowed_new_tokens, prefix_tokens,
                   budget_pages);
}

pkv_status pkv_sched_create(const pkv_sched_config* config, pkv_sched_t* out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(config)) return PKV_ERR_INVALID_ARG;
  pkv_sched* s = new (std::nothrow) pkv_sched();
  if (!s) return PKV_ERR_INVALID_ARG;
  s->cfg = *config;
  s->max_pages_per_seq = config->max_seq_len / config->page_size;
  s->free_heap.resize(static_cast<size_t>(config->num_pages));
  for (int i = 0; i < config->num_pages; ++i) s->free_heap[i] = i;   // sorted: a valid min-heap
  s->credits = config->num_pages;
  s->stats.pool_pages = config->num_pages;
  *out = s;
  return PKV_OK;
}

pkv_status pkv_sched_destroy(pkv_sched_t sched) {
  delete sched;
  return PKV_OK;
}

pkv_status pkv_sched_submit(pkv_sched_t s, int prompt_tokens, int max_new_tokens,
                            int* request_id) {
  if (!s || !request_id) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  *request_id = -1;
  Request r;
  r.prompt_tokens = prompt_tokens;
  if (budget_of(s->cfg, prompt_tokens, max_new_tokens, nullptr, &r.prefix, &r.budget) != PKV_OK)
    return PKV_ERR_INVALID_ARG;
  ++s->stats.submitted;
  if (r.budget > s->cfg.num_pages) {
    ++s->stats.rejected;
    return PKV_ERR_REJECTED;
  }
  const int id = s->next_id++;
  s->requests.emplace(id, std::move(r));
  s->queue.push_back(id);
  *request_id = id;
  return PKV_OK;
}

pkv_status pkv_sched_admit(pkv_sched_t s, int* ids, int capacity, int* count) {
  if (!s || !count || capacity < 0 || (capacity > 0 && !ids)) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  *count = 0;
  if (static_cast<size_t>(capacity) < s->queue.size()) return PKV_ERR_INVALID_ARG;
  int n = 0;
  if (!(s->cfg.static_batching && !s->active.empty())) {
    while (!s->queue.empty()) {
      Request& r = s->requests[s->queue.front()];
      if (r.budget > s->credits) break;
      const int id = s->queue.front();
      s->queue.pop_front();
      s->credits -= r.budget;
      r.active = true;
      r.pages.assign(static_cast<size_t>(s->cfg.num_layers) * s->max_pages_per_seq, -1);
      s->active.push_back(id);
      ids[n++] = id;
    }
  }
  for (int id : s->queue) {
    Request& r = s->requests[id];
    if (!r.waited) {
      r.waited = true;
      ++s->stats.admission_waits;
    }
  }
  s->stats.admitted += n;
  s->stats.peak_active = std::max<int64_t>(s->stats.peak_active, s->active.size());
  *count = n;
  return PKV_OK;
}

namespace {

pkv_status extend_locked(pkv_sched* s, int request_id, int length) {
  auto it = s->requests.find(request_id);
  if (it == s->requests.end() || !it->second.active) return PKV_ERR_INVALID_ARG;
  Request& r = it->second;
  if (length < 0 || length > r.prefix) return PKV_ERR_INVALID_ARG;
  const int need = (length + s->cfg.page_size - 1) / s->cfg.page_size;
  if (need > r.pages_per_layer) {
    for (int layer = 0; layer < s->cfg.num_layers; ++layer)
      for (int i = r.pages_per_layer; i < need; ++i)
        r.pages[static_cast<size_t>(layer) * s->max_pages_per_seq + i] = s->take_page();
    r.pages_per_layer = need;
    s->stats.peak_assigned_pages = std::max(s->stats.peak_assigned_pages, s->assigned());
  }
  return PKV_OK;
}

}  // namespace

pkv_status pkv_sched_extend(pkv_sched_t s, int request_id, int length) {
  if (!s) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  return extend_locked(s, request_id, length);
}

pkv_status pkv_sched_extend_batch(pkv_sched_t s, const int* ids, const int* lengths, int n) {
  if (!s || n < 0 || (n > 0 && (!ids || !lengths))) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  for (int i = 0; i < n; ++i) {
    const pkv_status st = extend_locked(s, ids[i], lengths[i]);
    if (st != PKV_OK) return st;
  }
  return PKV_OK;
}

pkv_status pkv_sched_finish(pkv_sched_t s, int request_id) {
  if (!s) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  auto it = s->requests.find(request_id);
  if (it == s->requests.end() || !it->second.active) return PKV_ERR_INVALID_ARG;
  Request& r = it->second;
  for (int layer = 0; layer < s->cfg.num_layers; ++layer)
    for (int i = 0; i < r.pages_per_layer; ++i)
      s->give_page(r.pages[static_cast<size_t>(layer) * s->max_pages_per_seq + i]);
  s->credits += r.budget;
  s->active.erase(std::find(s->active.begin(), s->active.end(), request_id));
  s->requests.erase(it);
  ++s->stats.finished;
  return PKV_OK;
}

pkv_status pkv_sched_decode_batch(pkv_sched_t s, int* ids, int capacity, int* count) {
  if (!s || !count || capacity < 0 || (capacity > 0 && !ids)) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  const int n = static_cast<int>(s->active.size());
  *count = n;
  if (capacity < n) return PKV_ERR_INVALID_ARG;
  std::copy(s->active.begin(), s->active.end(), ids);
  s->stats.largest_decode_batch = std::max<int64_t>(s->stats.largest_decode_batch, n);
  return PKV_OK;
}

pkv_status pkv_sched_block_tables(pkv_sched_t s, const int* ids, int n, int32_t* tables,
                                  int max_batch, int max_pages, int clear_tail) {
  if (!s || !tables || n < 0 || n > max_batch || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  std::vector<const Request*> rows(static_cast<size_t>(n));
  for (int b = 0; b < n; ++b) {
    auto it = s->requests.find(ids[b]);
    if (it == s->requests.end() || !it->second.active) return PKV_ERR_INVALID_ARG;
    if (it->second.pages_per_layer > max_pages) return PKV_ERR_INVALID_ARG;
    rows[b] = &it->second;
  }
  for (int layer = 0; layer < s->cfg.num_layers; ++layer) {
    for (int b = 0; b < max_batch; ++b) {
      int32_t* row = tables + (static_cast<size_t>(layer) * max_batch + b) * max_pages;
      int k = 0;
      if (b < n) {
        const Request& r = *rows[b];
        const int32_t* src = r.pages.data() + static_cast<size_t>(layer) * s->max_pages_per_seq;
        std::copy(src, src + r.pages_per_layer, row);
        k = r.pages_per_layer;
      } else if (!clear_tail) {
        continue;
      }
      if (clear_tail) std::fill(row + k, row + max_pages, -1);
    }
  }
  return PKV_OK;
}

pkv_status pkv_sched_get_stats(pkv_sched_t s, pkv_sched_stats* out) {
  if (!s || !out) return PKV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(s->lock);
  *out = s->stats;
  out->free_pages = static_cast<int64_t>(s->free_heap.size());
  out->free_credits = s->credits;
  out->active = static_cast<int64_t>(s->active.size());
  out->waiting = static_cast<int64_t>(s->queue.size());
  return PKV_OK;
}

}  // extern "C"
