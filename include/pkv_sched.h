/*
 * pkv_sched.h -- C ABI of the host-side page allocator and request scheduler
 * of libpkv (host code only; no GPU work, no CUDA calls).
 *
 * Source: the Tiny-vLLM README translation "Hours of YouTube and 85
 * handtyped pages of notes on LLM Inference - Start here", section
 * "現在のスコープ" (scope) and the static / continuous batching item of
 * "これまでの進捗":
 *  - admission guarantees room for each request's largest processed prefix,
 *    prompt_tokens + allowed_new_tokens - 1 tokens, rounded up to 16-token
 *    pages and charged for every layer; the allowed output budget is clamped
 *    to the context limit (the last predicted token is returned without being
 *    processed again);
 *  - these admission credits are separate from physical pages, which are
 *    handed out lazily as a sequence grows; finishing early returns both the
 *    pages and the unused credits;
 *  - waiting requests queue in FIFO order while their budget does not fit;
 *    because every admitted request holds credits for its whole run, growth
 *    can never exhaust the pool or deadlock; a request whose budget exceeds
 *    the whole pool is rejected with an error;
 *  - static batching admits the next group only after the current one has
 *    finished; continuous batching admits whenever credits free up;
 *  - statistics: pool size, peak active requests, largest decode batch, peak
 *    allocated pages, admission wait, final free pages.
 *
 * Lifecycle of a request: submitted (waiting) -> admitted (credits reserved)
 * -> prefilled (prompt pages allocated, first output token produced) ->
 * decoding (one token appended per decode batch) -> finished.  A sequence
 * whose prompt has P tokens and whose budget is N new tokens is prefilled
 * once and then takes part in N - 1 decode batches; in decode batch k it
 * appends the token at position P + k - 1.  Pages of a request finished by a
 * decode batch (budget reached) or by pkv_sched_finish are released at the
 * next pkv_sched_admit call, so the GPU work that reads them must be complete
 * or ordered before any later write into the pool (one stream suffices).
 *
 * All arrays are HOST memory owned by the caller.  Functions return PKV_OK
 * (0) or a PKV_E* code from pkv.h, or a count where stated.  A scheduler
 * object must not be used from two threads at once.
 */
#ifndef PKV_SCHED_H_
#define PKV_SCHED_H_

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_EREJECTED 7 /* request budget exceeds the whole pool */
#define PKV_ENOTFOUND 8 /* unknown or already finished request id */

typedef struct pkv_scheduler pkv_scheduler;

typedef struct {
  int64_t pool_pages;            /* physical pages managed */
  int64_t free_pages;            /* pages not held by any request now */
  int64_t free_credits;          /* admission credits not reserved now */
  int64_t peak_active;           /* most requests admitted at once */
  int64_t largest_decode_batch;  /* most sequences in one decode batch */
  int64_t peak_allocated_pages;  /* most physical pages held at once */
  int64_t admission_wait_total;  /* sum over admitted requests of admit calls waited */
  int64_t admission_wait_max;    /* longest wait of one request, in admit calls */
  int64_t submitted, admitted, rejected, finished;
  int64_t waiting, active;       /* current queue length / admitted, unfinished */
} pkv_sched_stats;

/*
 * num_pages: physical pages in the pool; num_layers: block tables per
 * sequence (credits are charged per layer); max_context: the context limit
 * in tokens (a multiple of page_size); page_size: tokens per page;
 * static_batching: 0 = continuous, 1 = static.  Returns NULL on bad sizes or
 * allocation failure.  Page ids are handed out lowest-free-first.
 */
PKV_API pkv_scheduler* pkv_sched_create(int64_t num_pages, int num_layers, int max_context,
                                        int page_size, int static_batching);
PKV_API void pkv_sched_destroy(pkv_scheduler* s);

/* Pages (credits) a request with these sizes reserves for all layers, after
 * clamping max_new_tokens to the context limit; -1 if the prompt is empty or
 * longer than the context, or max_new_tokens < 1. */
PKV_API int64_t pkv_sched_budget_pages(const pkv_scheduler* s, int prompt_tokens,
                                       int max_new_tokens);

/* Queue a request.  *id receives its id (ids count up from 0).  Returns
 * PKV_EREJECTED (and queues nothing) when its budget exceeds the pool,
 * PKV_EINVAL for sizes pkv_sched_budget_pages rejects. */
PKV_API int pkv_sched_submit(pkv_scheduler* s, int prompt_tokens, int max_new_tokens,
                             int64_t* id);

/* One scheduling point: releases what finished since the last call, then
 * admits waiting requests in FIFO order while the head's budget fits (static
 * batching: only when no admitted request is left).  Returns the number
 * admitted. */
PKV_API int pkv_sched_admit(pkv_scheduler* s);

/* Picks the oldest admitted request that has not been prefilled, allocates
 * the pages of its prompt in every layer and writes its block tables to
 * block_tables[layer * max_blocks + k] (max_blocks = max_context /
 * page_size; unused entries -1).  Returns 1 and fills *id / *prompt_tokens,
 * or 0 when there is nothing to prefill. */
PKV_API int pkv_sched_next_prefill(pkv_scheduler* s, int64_t* id, int32_t* prompt_tokens,
                                   int32_t* block_tables);

/* Builds the next decode batch from the prefilled, unfinished requests in
 * admission order, at most max_batch of them: allocates a page in every layer
 * for each sequence whose new token starts a page, advances its length and
 * writes ids[i], seq_lens[i] (length after this step's append) and
 * block_tables[(layer * max_batch + i) * max_blocks + k].  Sequences that
 * reach their budget with this batch are finished by it.  Returns the batch
 * size. */
PKV_API int pkv_sched_decode_batch(pkv_scheduler* s, int max_batch, int64_t* ids,
                                   int32_t* seq_lens, int32_t* block_tables);

/* The number of prefilled, unfinished requests: the size of the next decode
 * batch before its max_batch cap (so that a caller can size its buffers). */
PKV_API int pkv_sched_running(const pkv_scheduler* s);

/* Early finish (e.g. an end-of-sequence token): the request leaves the next
 * decode batches; its pages and unused credits return at the next admit. */
PKV_API int pkv_sched_finish(pkv_scheduler* s, int64_t id);

/* Current length (tokens in the cache) of a request, or -1. */
PKV_API int32_t pkv_sched_seq_len(const pkv_scheduler* s, int64_t id);

PKV_API void pkv_sched_get_stats(const pkv_scheduler* s, pkv_sched_stats* out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_SCHED_H_ */
