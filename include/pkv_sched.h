/*
 * pkv_sched.h - host-side admission control and page assignment for the
 * shared KV page pool (CPU only: no CUDA call, usable without a GPU).
 *
 * The rule follows the samir-vllm pages [6 Hours of YouTube and 85
 * handtyped pages of notes on LLM Inference - Start here, README paragraphs
 * on admission, FIFO waiting, rejection and --stats; samir-vllm: Build LLM
 * Inference From Scratch in C++ and CUDA, "Admission control: how the
 * scheduler avoids deadlock"]:
 *
 *   budget(P, max_new) = ceil((P + N - 1) / page_size) * num_layers pages,
 *   N = min(max_new, max_seq_len - P),
 *
 * the largest prefix the request ever processes (the last predicted token is
 * returned, not processed), rounded up to whole pages in every layer. These
 * budgets are admission credits, separate from physical pages: a request is
 * admitted in FIFO order (nothing overtakes a waiting request) once its
 * budget fits in the credits that active requests do not hold; its physical
 * pages are taken from the free list lazily, one per layer each time the
 * sequence grows into a new page. An admitted request therefore always has
 * pages to finish, so growth can neither exhaust the pool nor deadlock.
 * Completion (early or not) returns its pages and all its credits. A request
 * whose budget exceeds the pool is rejected at submission. Continuous
 * batching admits whenever credits allow; static batching admits a new group
 * only after the whole current group has finished.
 *
 * Readings where the pages are silent: a submission needs
 * 1 <= prompt_tokens < max_seq_len and max_new_tokens >= 1; free pages are
 * handed out lowest id first; a request counts once in admission_waits if
 * an admission pass after its submission left it queued.
 *
 * Every call takes the scheduler's lock, so calls from several host threads
 * are safe; the order in which they land is the caller's to fix.
 */
#ifndef PKV_SCHED_H
#define PKV_SCHED_H

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int num_layers;        /* 16 for the pages' model; >= 1 */
  int num_pages;         /* physical pages in the pool (all layers share them); >= 1 */
  int page_size;         /* tokens per page: 16 */
  int max_seq_len;       /* context: 2048; a multiple of page_size */
  int static_batching;   /* 0: continuous batching, 1: static batching */
} pkv_sched_config;

/* Counters as the pages' --stats flag reports them, plus running totals. */
typedef struct {
  int64_t pool_pages;
  int64_t submitted;             /* valid submissions, rejected ones included */
  int64_t rejected;
  int64_t admitted;
  int64_t finished;
  int64_t peak_active;           /* most requests admitted at once */
  int64_t largest_decode_batch;  /* largest batch pkv_sched_decode_batch returned */
  int64_t peak_assigned_pages;   /* most physical pages assigned at once */
  int64_t admission_waits;       /* requests that had to wait for admission */
  int64_t free_pages;
  int64_t free_credits;
  int64_t active;
  int64_t waiting;
} pkv_sched_stats;

typedef struct pkv_sched* pkv_sched_t;

/* Budget arithmetic alone: the output allowance after clamping, the largest
 * processed prefix and the pages reserved. INVALID_ARG for an invalid
 * submission (see above). Any output pointer may be NULL. */
pkv_status pkv_sched_budget(const pkv_sched_config* config, int prompt_tokens,
                            int max_new_tokens, int* allowed_new_tokens, int* prefix_tokens,
                            int64_t* budget_pages);

/* Creates a scheduler over an empty pool. INVALID_ARG for a bad config. */
pkv_status pkv_sched_create(const pkv_sched_config* config, pkv_sched_t* out);
pkv_status pkv_sched_destroy(pkv_sched_t sched);

/* Queues a request; *request_id receives its id (ids count up from 0).
 * PKV_ERR_REJECTED if its budget exceeds the pool (counted, not queued),
 * INVALID_ARG for an invalid submission (not counted). */
pkv_status pkv_sched_submit(pkv_sched_t sched, int prompt_tokens, int max_new_tokens,
                            int* request_id);

/* One admission pass: admits queued requests in FIFO order while the head's
 * budget fits (continuous), or a new group when none is active (static).
 * Writes up to `capacity` admitted ids to `ids` and their count to *count;
 * INVALID_ARG, admitting nothing, if capacity could be too small (capacity
 * must be at least the number of waiting requests). */
pkv_status pkv_sched_admit(pkv_sched_t sched, int* ids, int capacity, int* count);

/* Makes positions < length of an admitted request addressable: assigns one
 * page per layer for every page the sequence reaches that it does not own
 * yet. INVALID_ARG if the request is not active or length exceeds its
 * reserved prefix. Never fails for lack of pages (the credits guarantee them). */
pkv_status pkv_sched_extend(pkv_sched_t sched, int request_id, int length);

/* pkv_sched_extend for n requests at once (ids[i] to lengths[i]), in order;
 * stops at the first failure and returns its status. */
pkv_status pkv_sched_extend_batch(pkv_sched_t sched, const int* ids, const int* lengths, int n);

/* Ends an admitted request: its pages go back to the free list and its
 * credits to the pool. INVALID_ARG if it is not active. */
pkv_status pkv_sched_finish(pkv_sched_t sched, int request_id);

/* The active requests in admission order: one decode step's batch. Writes up
 * to `capacity` ids and the full count to *count (INVALID_ARG if capacity is
 * smaller than the count); records the largest batch for the counters. */
pkv_status pkv_sched_decode_batch(pkv_sched_t sched, int* ids, int capacity, int* count);

/* Host block tables for a batch: tables is int32
 * [num_layers][max_batch][max_pages], row b of layer l the physical pages of
 * ids[b] in layer l in logical order. With clear_tail != 0 every entry past
 * a row's assigned pages, and every row n .. max_batch - 1, is set to -1;
 * with clear_tail == 0 those entries are left as they are (the decode
 * kernels read only the pages a sequence's length covers, so a reused
 * buffer need not be cleared every step). The layout is the one the decode
 * entry points of pkv.h take (max_pages = max_seq_len / page_size there).
 * INVALID_ARG for an inactive id, n > max_batch or max_pages too small. */
pkv_status pkv_sched_block_tables(pkv_sched_t sched, const int* ids, int n, int32_t* tables,
                                  int max_batch, int max_pages, int clear_tail);

pkv_status pkv_sched_get_stats(pkv_sched_t sched, pkv_sched_stats* stats);

#ifdef __cplusplus
}
#endif

#endif /* PKV_SCHED_H */
