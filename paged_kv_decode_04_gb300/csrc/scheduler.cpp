// scheduler.cpp -- host page allocator and request scheduler behind
// include/pkv_sched.h: page-credit admission with a FIFO queue, lazy physical
// page allocation, static or continuous batching, and run statistics.
// Plain C++17, no CUDA.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <deque>
#include <map>
#include <new>
#include <set>
#include <vector>

#include "pkv.h"
#include "pkv_sched.h"

namespace {

enum class State { kWaiting, kAdmitted, kRunning, kFinished };

struct Request {
  int64_t id = 0;
  int prompt = 0;
  int budget_new = 0;      // allowed new tokens after clamping
  int64_t credits = 0;     // pages reserved (all layers)
  int32_t len = 0;         // tokens in the cache
  int generated = 0;       // output tokens produced so far
  State state = State::kWaiting;
  int64_t waited = 0;      // admit calls spent waiting
  std::vector<std::vector<int32_t>> pages;  // [layer][block]
};

}  // namespace

struct pkv_scheduler {
  int64_t num_pages = 0;
  int layers = 0;
  int max_context = 0;
  int page_size = 0;
  int max_blocks = 0;
  bool static_batching = false;

  std::set<int32_t> free_pages;   // lowest id first
  int64_t free_credits = 0;
  int64_t next_id = 0;
  std::deque<int64_t> waiting;    // FIFO of request ids
  std::vector<int64_t> admitted;  // admission order, unfinished or awaiting release
  std::vector<int64_t> to_release;
  std::map<int64_t, Request> reqs;

  pkv_sched_stats st{};

  int64_t budget(int prompt, int max_new) const {
    if (prompt < 1 || prompt > max_context || max_new < 1) return -1;
    const int allowed = std::min(max_new, max_context + 1 - prompt);
    const int64_t tokens = static_cast<int64_t>(prompt) + allowed - 1;
    return (tokens + page_size - 1) / page_size * layers;
  }

  int32_t take_page() {
    auto it = free_pages.begin();  // never empty: callers hold credits for it
    const int32_t p = *it;
    free_pages.erase(it);
    const int64_t held = num_pages - static_cast<int64_t>(free_pages.size());
    st.peak_allocated_pages = std::max(st.peak_allocated_pages, held);
    return p;
  }

  void release(Request& r) {
    for (auto& layer : r.pages)
      for (int32_t p : layer) free_pages.insert(p);
    r.pages.clear();
    free_credits += r.credits;
    r.credits = 0;
  }

  int64_t active_count() const {
    int64_t n = 0;
    for (int64_t id : admitted) {
      const Request& r = reqs.at(id);
      if (r.state == State::kAdmitted || r.state == State::kRunning) ++n;
    }
    return n;
  }
};

extern "C" {

PKV_API pkv_scheduler* pkv_sched_create(int64_t num_pages, int num_layers, int max_context,
                                        int page_size, int static_batching) {
  if (num_pages < 1 || num_pages > INT32_MAX || num_layers < 1 || page_size < 1 ||
      max_context < page_size || max_context % page_size != 0)
    return nullptr;
  pkv_scheduler* s = new (std::nothrow) pkv_scheduler();
  if (s == nullptr) return nullptr;
  s->num_pages = num_pages;
  s->layers = num_layers;
  s->max_context = max_context;
  s->page_size = page_size;
  s->max_blocks = max_context / page_size;
  s->static_batching = static_batching != 0;
  for (int64_t p = 0; p < num_pages; ++p) s->free_pages.insert(static_cast<int32_t>(p));
  s->free_credits = num_pages;
  s->st.pool_pages = num_pages;
  return s;
}

PKV_API void pkv_sched_destroy(pkv_scheduler* s) { delete s; }

PKV_API int64_t pkv_sched_budget_pages(const pkv_scheduler* s, int prompt_tokens,
                                       int max_new_tokens) {
  return s ? s->budget(prompt_tokens, max_new_tokens) : -1;
}

PKV_API int pkv_sched_submit(pkv_scheduler* s, int prompt_tokens, int max_new_tokens,
                             int64_t* id) {
  if (s == nullptr || id == nullptr) return PKV_EINVAL;
  const int64_t credits = s->budget(prompt_tokens, max_new_tokens);
  if (credits < 0) return PKV_EINVAL;
  s->st.submitted++;
  if (credits > s->num_pages) {
    s->st.rejected++;
    return PKV_EREJECTED;
  }
  Request r;
  r.id = s->next_id++;
  r.prompt = prompt_tokens;
  r.budget_new = std::min(max_new_tokens, s->max_context + 1 - prompt_tokens);
  r.credits = credits;
  s->reqs[r.id] = r;
  s->waiting.push_back(r.id);
  *id = r.id;
  return PKV_OK;
}

PKV_API int pkv_sched_admit(pkv_scheduler* s) {
  if (s == nullptr) return 0;
  for (int64_t id : s->to_release) s->release(s->reqs.at(id));
  s->to_release.clear();
  s->admitted.erase(std::remove_if(s->admitted.begin(), s->admitted.end(),
                                   [s](int64_t id) {
                                     return s->reqs.at(id).state == State::kFinished;
                                   }),
                    s->admitted.end());
  int n = 0;
  const bool may_admit = !s->static_batching || s->active_count() == 0;
  while (may_admit && !s->waiting.empty()) {
    Request& head = s->reqs.at(s->waiting.front());
    if (head.credits > s->free_credits) break;  // FIFO: nobody overtakes the head
    s->free_credits -= head.credits;
    head.state = State::kAdmitted;
    s->st.admission_wait_total += head.waited;
    s->st.admission_wait_max = std::max(s->st.admission_wait_max, head.waited);
    s->st.admitted++;
    s->admitted.push_back(head.id);
    s->waiting.pop_front();
    ++n;
  }
  for (int64_t id : s->waiting) s->reqs.at(id).waited++;
  s->st.peak_active = std::max(s->st.peak_active, s->active_count());
  return n;
}

PKV_API int pkv_sched_next_prefill(pkv_scheduler* s, int64_t* id, int32_t* prompt_tokens,
                                   int32_t* block_tables) {
  if (s == nullptr || id == nullptr || prompt_tokens == nullptr || block_tables == nullptr)
    return 0;
  for (int64_t rid : s->admitted) {
    Request& r = s->reqs.at(rid);
    if (r.state != State::kAdmitted) continue;
    const int blocks = (r.prompt + s->page_size - 1) / s->page_size;
    r.pages.assign(s->layers, std::vector<int32_t>());
    for (int l = 0; l < s->layers; ++l)
      for (int k = 0; k < blocks; ++k) r.pages[l].push_back(s->take_page());
    r.len = r.prompt;
    r.generated = 1;  // the prefill predicts the first output token
    r.state = State::kRunning;
    if (r.generated >= r.budget_new) {
      r.state = State::kFinished;
      s->st.finished++;
      s->to_release.push_back(r.id);
    }
    for (int l = 0; l < s->layers; ++l)
      for (int k = 0; k < s->max_blocks; ++k)
        block_tables[static_cast<int64_t>(l) * s->max_blocks + k] =
            k < blocks ? r.pages[l][k] : -1;
    *id = r.id;
    *prompt_tokens = r.prompt;
    return 1;
  }
  return 0;
}

PKV_API int pkv_sched_decode_batch(pkv_scheduler* s, int max_batch, int64_t* ids,
                                   int32_t* seq_lens, int32_t* block_tables) {
  if (s == nullptr || max_batch < 1 || ids == nullptr || seq_lens == nullptr ||
      block_tables == nullptr)
    return 0;
  int n = 0;
  for (int64_t rid : s->admitted) {
    if (n == max_batch) break;
    Request& r = s->reqs.at(rid);
    if (r.state != State::kRunning) continue;
    const int32_t pos = r.len;  // the token appended by this step
    if (pos % s->page_size == 0)
      for (int l = 0; l < s->layers; ++l) r.pages[l].push_back(s->take_page());
    r.len = pos + 1;
    r.generated++;
    ids[n] = r.id;
    seq_lens[n] = r.len;
    const int blocks = static_cast<int>(r.pages[0].size());
    for (int l = 0; l < s->layers; ++l) {
      int32_t* row = block_tables + (static_cast<int64_t>(l) * max_batch + n) * s->max_blocks;
      std::copy(r.pages[l].begin(), r.pages[l].begin() + blocks, row);
      std::fill(row + blocks, row + s->max_blocks, -1);
    }
    if (r.generated >= r.budget_new) {
      r.state = State::kFinished;
      s->st.finished++;
      s->to_release.push_back(r.id);
    }
    ++n;
  }
  s->st.largest_decode_batch = std::max<int64_t>(s->st.largest_decode_batch, n);
  return n;
}

PKV_API int pkv_sched_running(const pkv_scheduler* s) {
  if (s == nullptr) return 0;
  int n = 0;
  for (int64_t rid : s->admitted)
    if (s->reqs.at(rid).state == State::kRunning) ++n;
  return n;
}

PKV_API int pkv_sched_finish(pkv_scheduler* s, int64_t id) {
  if (s == nullptr) return PKV_EINVAL;
  auto it = s->reqs.find(id);
  if (it == s->reqs.end() || it->second.state == State::kFinished) return PKV_ENOTFOUND;
  Request& r = it->second;
  if (r.state == State::kWaiting) {
    s->waiting.erase(std::find(s->waiting.begin(), s->waiting.end(), id));
  } else {
    s->to_release.push_back(id);
  }
  r.state = State::kFinished;
  s->st.finished++;
  return PKV_OK;
}

PKV_API int32_t pkv_sched_seq_len(const pkv_scheduler* s, int64_t id) {
  if (s == nullptr) return -1;
  auto it = s->reqs.find(id);
  return it == s->reqs.end() ? -1 : it->second.len;
}

PKV_API void pkv_sched_get_stats(const pkv_scheduler* s, pkv_sched_stats* out) {
  if (s == nullptr || out == nullptr) return;
  *out = s->st;
  out->free_pages = static_cast<int64_t>(s->free_pages.size());
  out->free_credits = s->free_credits;
  out->waiting = static_cast<int64_t>(s->waiting.size());
  out->active = s->active_count();
}

}  // extern "C"
