/*
 * pkv.h - paged KV cache decode path for one GB300 (sm_103a) GPU.
 *
 * A shared BF16 page pool holds the KV cache of every sequence and layer.
 * A physical page holds 16 tokens of K and of V for one layer, and a block
 * table per sequence and layer maps the sequence's logical pages to physical
 * page ids; decode appends one new token per sequence at its absolute
 * position and then attends over the sequence's pages in place, with an FP32
 * online softmax, without gathering a contiguous prefix or storing scores.
 *   [samir-vllm: Build LLM Inference From Scratch in C++ and CUDA,
 *    "Architecture walkthrough", KV cache paragraph, and "TL;DR" table, Decode
 *    row; 6 Hours of YouTube and 85 handtyped pages of notes on LLM Inference
 *    - Start here, README feature list: shared BF16 KV page pool bullet,
 *    batched decode bullet, direct paged decode attention bullet]
 *
 * Geometry (fixed by this library): 32 query heads over 8 KV heads (query
 * head h reads KV head h / 4), head_dim 64, 16-token pages, score scale
 * 1/sqrt(64), at most 2,048 tokens of context (128 pages per sequence).
 *
 * Layouts (all row-major, all device memory allocated by the caller):
 *   k_pool, v_pool   BF16 [num_pages][8][16][64]   (page, kv head, token, dim)
 *                    one (page, kv head) tile is 2 KiB, contiguous
 *   block_tables     int32 [num_layers][max_batch][max_seq_len / 16]
 *                    physical page id of logical page i of sequence b in
 *                    layer l; ids are global over the one pool
 *   q                BF16 [batch][32][64]   (one layer)
 *   k, v (new token) BF16 [batch][8][64]    (one layer)
 *   positions        int32 [batch]: absolute position of the appended token
 *   seq_lens         int32 [batch]: attended length AFTER the append; the
 *                    token at position seq_lens[b] - 1 is attended
 *   out              FP32 [batch][32][64]   (one layer)
 * Every pointer must be 16-byte aligned (the kernels move 16-byte vectors
 * and the page tiles are copied by the bulk-copy engine).
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream). Host-detectable problems (null or misaligned pointers,
 * layer or batch out of range, unsupported geometry) return an error status
 * synchronously and launch nothing. Index problems found in device data (a
 * page id outside [0, num_pages), a position outside [0, max_seq_len), a
 * seq_len outside [1, max_seq_len]) are recorded in the pool's sticky device
 * error flag; the kernel skips the offending unit and never faults or
 * traps. pkv_get_error reports and clears the flag.
 *
 * Block-table contract (the caller's, as in the pages' engine where each
 * request owns its pages): a page belongs to one (sequence, layer); no two
 * sequences of one call map to the same (page, slot).
 */
#ifndef PKV_H
#define PKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad layer/batch/splits */
  PKV_ERR_OUT_OF_RANGE = 2,   /* device data: page id, position or seq_len */
  PKV_ERR_CUDA = 3,           /* a CUDA runtime call failed */
  PKV_ERR_UNSUPPORTED = 4,    /* geometry this library is not built for */
  PKV_ERR_DEVICE_TIMEOUT = 5, /* a bounded in-kernel wait gave up */
  PKV_ERR_STATIC_LIMIT = 6,   /* request larger than pkv_decode_attention_noalloc's scratch */
  PKV_ERR_REJECTED = 7        /* admission: a request's budget exceeds the whole pool */
} pkv_status;

/* Pool geometry. page_size, num_q_heads, num_kv_heads and head_dim must be
 * 16, 32, 8 and 64. max_seq_len is a multiple of 16, at most 2048, and sets
 * the block-table row length (max_seq_len / 16). max_splits bounds the
 * split-KV count per sequence (0 selects 64; at most 128) and sizes the
 * handle's split workspace. flags: PKV_FLAG_* below (0 for none).
 * num_pages is the number of pages in the pool the caller allocates: 4096
 * pages is the pages' default 128 MiB pool
 * [samir-vllm: Build LLM Inference From Scratch in C++ and CUDA, "Hardware
 * expectations"]. */
typedef struct {
  int num_layers;
  int num_pages;
  int page_size;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int max_seq_len;
  int max_batch;
  int max_splits;
  int flags;        /* PKV_FLAG_* bits */
} pkv_pool_config;

/* Launch decode kernels with programmatic dependent launch: a launch may
 * start while the kernel before it in the stream is still running, and
 * before waiting for that kernel it reads block_tables, seq_lens, the rotary
 * tables (the _rope entry points) and the pool rows below position
 * seq_lens[b] - 1 (the unfused decode defers the page holding that
 * position). q, k, v, out and the appended slot are read or written only
 * after the wait. A decode launch lets the next one start only after its
 * own wait, so every kernel two or more places earlier in the stream has
 * completed before the next launch's pre-wait reads. Contract: the kernel
 * immediately before a decode launch in the stream must not write
 * block_tables, seq_lens, the rotary tables or those pool rows. (In a model
 * of two or more layers, consecutive decode steps meet it: the step before
 * wrote the rows of the same layer one launch per layer earlier. A
 * one-layer model's consecutive fused steps do not: put another kernel
 * between them or leave this flag off.) Off by default. */
#define PKV_FLAG_PDL 1

typedef struct pkv_pool* pkv_pool_t;

/* Validates the geometry and creates a handle on the current device. The
 * handle owns only device scratch: the split-KV partials (two layer-parity
 * copies of max_batch x 32 x max_splits x (64 + 2) floats), one ticket
 * counter per (sequence, kv head) and parity, one layer counter per sequence
 * (pkv_append_attend_layers) and the sticky error flag.
 * It does not own the pools, tables or tensors. A handle's launches share
 * that scratch, so they must be ordered in one stream (calls issued to
 * several streams at once need a handle each). Returns INVALID_ARG for a
 * null argument, UNSUPPORTED for a geometry other than the one above, CUDA
 * if an allocation fails. */
pkv_status pkv_pool_create(const pkv_pool_config* config, pkv_pool_t* out);

/* Frees the handle's device scratch. Waits for the device to finish work
 * that may still use it. NULL is accepted. */
pkv_status pkv_pool_destroy(pkv_pool_t pool);

/* Decode-time append [samir-vllm: Build LLM Inference From Scratch in C++ and
 * CUDA, "Architecture walkthrough", KV cache paragraph; README feature list,
 * shared BF16 KV page pool bullet]: for every sequence b < batch and kv head
 * j, copies k[b][j][:] and v[b][j][:] to
 *   k_pool / v_pool [block_tables[layer][b][p / 16]][j][p % 16][:],
 * p = positions[b]. Bit copy, no arithmetic. A sequence whose position or
 * page id is out of range is skipped and flagged. batch == 0 is a no-op. */
pkv_status pkv_append(pkv_pool_t pool, int layer, const void* k, const void* v, void* k_pool,
                      void* v_pool, const int32_t* block_tables, const int32_t* positions,
                      int batch, void* stream);

/* Paged decode attention for one layer [README feature list, direct paged
 * decode attention bullet]: for every sequence b and query head h,
 *   out[b][h][:] = sum_t softmax_t(q[b][h] . K_t / 8) V_t,  t < seq_lens[b],
 * K_t, V_t read from the pools through block_tables[layer][b] (kv head h/4).
 * One thread block per (sequence, kv head, split) serves the 4 query heads of
 * the kv head, so every page tile is read once. num_splits = S > 0 splits
 * each sequence's np = ceil(len / 16) pages into ranges of ceil(np / S)
 * pages, computed separately and merged by log-sum-exp inside the same
 * launch: for 2 <= S <= 16 (where the device schedules such clusters) the S
 * blocks of a (sequence, kv head) form a thread-block cluster and merge
 * through distributed shared memory; otherwise through the handle's global
 * partials and a ticket (the last block to finish merges). num_splits = 0
 * lets the library choose: for up to 32 sequences a cluster split and a
 * block shape (page stages per warp, blocks per SM) from plans measured on
 * GB300, for larger batches the ticket merge over page ranges sized in the
 * launch from the batch's lengths (whole sequences past two waves of
 * blocks), longest sequences first (pkv_plan_decode below).
 * S must not exceed max_splits. The
 * output does not depend on which physical pages hold the data. A sequence
 * with an invalid seq_len is skipped (its out rows are left untouched) and
 * flagged; an invalid page id is skipped and flagged. */
pkv_status pkv_decode_attention(pkv_pool_t pool, int layer, const void* q, const void* k_pool,
                                const void* v_pool, const int32_t* block_tables,
                                const int32_t* seq_lens, float* out, int batch, int num_splits,
                                void* stream);

/* Append and attend fused into one launch: the same results as pkv_append
 * with positions[b] = seq_lens[b] - 1 followed by pkv_decode_attention. The
 * block that owns the sequence's last page writes the new token's K/V into
 * the pool and uses it from on-chip memory; no other block reads that slot. */
pkv_status pkv_append_attend(pkv_pool_t pool, int layer, const void* q, const void* k,
                             const void* v, void* k_pool, void* v_pool,
                             const int32_t* block_tables, const int32_t* seq_lens, float* out,
                             int batch, int num_splits, void* stream);

/* Rotary position embedding applied on the decode path. The pages have decode
 * write the new token at its absolute rotary position [samir-vllm: Build LLM
 * Inference From Scratch in C++ and CUDA, "Architecture walkthrough", KV
 * cache paragraph; 6 Hours of YouTube and 85 handtyped pages of notes on LLM
 * Inference - Start here, README feature list, shared BF16 KV page pool
 * bullet] and the prefill stack applies RoPE to Q and K; they do not print the
 * rotation, so it is the rotate-half form: dim i < 32 pairs with dim i + 32,
 *   x'[i] = x[i] cos(a) - x[i+32] sin(a),  x'[i+32] = x[i+32] cos(a) + x[i] sin(a),
 * a = angle (p, i) for position p.
 *
 * rope_cos, rope_sin: device FP32 tables [max_seq_len][32] (cos and sin of
 * the angle of pair i at position p; row p at offset 32 p), 16-byte aligned,
 * owned by the caller, read-only here; the base and any frequency scaling are
 * the caller's choice. A null or misaligned table returns INVALID_ARG.
 *
 * Keys are rotated in FP32 with each product and the sum rounded separately
 * (no fused multiply-add) and stored as BF16 rounded to nearest even, so the
 * pool content is bit-defined. Queries are rotated in FP32 and never stored.
 *
 * pkv_append_rope: pkv_append with each key rotated to positions[b].
 * pkv_decode_attention_rope: pkv_decode_attention with each query rotated to
 *   position seq_lens[b] - 1 (the cached keys are expected to be rotated).
 * pkv_append_attend_rope: pkv_append_attend with both: the same results as
 *   pkv_append_rope then pkv_decode_attention_rope, in one launch. */
pkv_status pkv_append_rope(pkv_pool_t pool, int layer, const void* k, const void* v,
                           void* k_pool, void* v_pool, const int32_t* block_tables,
                           const int32_t* positions, const float* rope_cos,
                           const float* rope_sin, int batch, void* stream);
pkv_status pkv_decode_attention_rope(pkv_pool_t pool, int layer, const void* q,
                                     const void* k_pool, const void* v_pool,
                                     const int32_t* block_tables, const int32_t* seq_lens,
                                     const float* rope_cos, const float* rope_sin, float* out,
                                     int batch, int num_splits, void* stream);
pkv_status pkv_append_attend_rope(pkv_pool_t pool, int layer, const void* q, const void* k,
                                  const void* v, void* k_pool, void* v_pool,
                                  const int32_t* block_tables, const int32_t* seq_lens,
                                  const float* rope_cos, const float* rope_sin, float* out,
                                  int batch, int num_splits, void* stream);

/* Several consecutive layers of the fused step in one launch. A decode step
 * runs the attention of every one of the model's 16 layers for each new
 * token [6 Hours of YouTube and 85 handtyped pages of notes on LLM Inference
 * - Start here, README feature list: the fixed 16-layer Llama 3.2 1B layout
 * and the batched decode bullet]; at small batches each layer's work is a few
 * microseconds, so the per-layer launch and the wait for the previous
 * layer's completion dominate, and one persistent launch removes them.
 *
 * For j = 0 .. num_layers - 1 the same results (pool contents and out) as
 *   pkv_append_attend(pool, layer_begin + j, q_j, k_j, v_j, k_pool, v_pool,
 *                     block_tables, seq_lens, out_j, batch, 0, stream)
 * in order of j, where q is [num_layers][batch][32][64] BF16 (q_j its j-th
 * slab), k and v [num_layers][batch][8][64] BF16 and out
 * [num_layers][batch][32][64] FP32; seq_lens (the post-append length) holds
 * for every layer. Layers keep their order per sequence: the blocks of
 * sequence b read q_j, k_j, v_j and write the appended slot of layer j only
 * after every output row of b at layer j - 1 has been written, the order a
 * model imposes between layers; pages of cached tokens, which no layer of
 * the call writes, are read ahead across the layer boundary.
 *
 * Plan: one thread-block cluster of S blocks per (sequence, kv head), S the
 * largest of 16, 8, 4, 2 for which every cluster of the grid is resident at
 * once; the blocks of a sequence then wait for one another between layers
 * (bounded: a wait that gives up flags PKV_ERR_DEVICE_TIMEOUT and the block
 * carries on without waiting). A launch covers at most 256 / ceil(128 / S)
 * layers (32 at S = 16, 4 at S = 2); longer calls are split into several. A
 * batch for which even S = 2 does not fit runs as one pkv_append_attend launch
 * per layer. Uses a per-sequence counter in the handle (zeroed on the stream
 * before each launch), so one handle serves one such call at a time.
 * Residency is checked against an idle device: the launch must not overlap
 * other work on the device (another stream's kernels holding SMs can keep
 * some clusters from becoming resident; the blocks of a sequence then wait
 * for blocks that cannot start, every such wait gives up after about two
 * seconds, PKV_ERR_DEVICE_TIMEOUT is flagged and that launch's outputs carry
 * no layer-order guarantee). A caller that shares the device with other
 * streams uses pkv_append_attend per layer instead.
 * Errors as for pkv_append_attend; layer_begin + num_layers must not exceed
 * num_layers of the handle. num_layers == 0 or batch == 0 is a no-op. */
pkv_status pkv_append_attend_layers(pkv_pool_t pool, int layer_begin, int num_layers,
                                    const void* q, const void* k, const void* v, void* k_pool,
                                    void* v_pool, const int32_t* block_tables,
                                    const int32_t* seq_lens, float* out, int batch,
                                    void* stream);

/* Test hook for failure detection: the same launch as
 * pkv_append_attend_layers with every between-layer wait made unreachable
 * (its target raised by one), so each block's first wait runs out after about
 * two seconds; the block flags PKV_ERR_DEVICE_TIMEOUT, stops waiting and
 * finishes (outputs then carry no layer-order guarantee). No GPU fault; the
 * context stays usable. Returns UNSUPPORTED for a batch that would run as
 * per-layer launches. */
pkv_status pkv_test_layers_wait_timeout(pkv_pool_t pool, int layer_begin, int num_layers,
                                        const void* q, const void* k, const void* v,
                                        void* k_pool, void* v_pool, const int32_t* block_tables,
                                        const int32_t* seq_lens, float* out, int batch,
                                        void* stream);

/* The launch plan of pkv_decode_attention and pkv_append_attend (and their
 * rotary variants) for a batch, from the device figures a handle records.
 * pkv_plan_decode is plain host arithmetic (no GPU needed), the same function
 * the launches call.
 *
 * Plans (num_splits = 0): for up to 32 sequences a thread-block cluster of S
 * blocks per (sequence, kv head): the narrow shape (3 page stages per warp)
 * with S = 16 or 12 while the blocks of two consecutive launches fit its
 * resident slots, else the wide shape (2 stages, 4 blocks per SM) with S = 8
 * while two launches fit its slots, else the narrow shape with S = 8 while
 * one launch's blocks take at most 9/16 of its slots, else the wide shape
 * with the largest S <= 8 whose blocks take at most 27/32 of its slots;
 * larger batches take the ticket merge with ranges of at least chunk_pages
 * = max(16, ceil(max_seq_len / 16 / max_splits)) pages. When the blocks of
 * full-length sequences would exceed one wave of resident ticket blocks,
 * the launch has the grid (1, 8, grid_units), its blocks taking (sequence,
 * range) units longest sequence first. Up to two waves of sequences
 * (batch x 8 <= 2 x resident ticket blocks) it sizes the ranges from the
 * lengths it reads: max(chunk_pages, min(128, ceil(T / range_div))) pages,
 * T the batch's total page count (one kv head), range_div = resident
 * ticket blocks x 3 / 40, rounded (about 1.65 times the pages per resident
 * block slot), grid_units = batch + range_div. Past two waves every sequence is
 * one unit (chunk_pages = max_seq_len / 16, grid_units = batch). Otherwise
 * the grid is (grid_splits, 8, batch). A chosen
 * num_splits = S takes a cluster for 2 <= S <= max_cluster (narrow while its
 * blocks fit one wave of it, else wide), the ticket merge otherwise. */
typedef struct {
  int num_sms;                /* streaming multiprocessors */
  int ticket_blocks_per_sm;   /* resident blocks per SM of the ticket-merge shape */
  int narrow_blocks_per_sm;   /* ... of the narrow cluster shape */
  int wide_blocks_per_sm;     /* ... of the wide cluster shape */
  int max_cluster;            /* largest cluster (power of two <= 16) the device schedules; 0: none */
  int max_splits;             /* the handle's max_splits (after the default) */
  int max_seq_len;            /* the handle's max_seq_len */
} pkv_device_figures;

#define PKV_SHAPE_TICKET 0
#define PKV_SHAPE_NARROW 1
#define PKV_SHAPE_WIDE 2

typedef struct {
  int shape;          /* PKV_SHAPE_* */
  int cluster;        /* blocks per cluster (the split count) for the cluster shapes, else 0 */
  int num_splits;     /* splits per sequence (cluster plans, chosen counts), else 0 */
  int chunk_pages;    /* pages per range when num_splits == 0 (the least, with range_div), else 0 */
  int range_div;      /* longest first: ranges of max(chunk_pages, min(128, ceil(T / range_div)))
                         pages, T the batch's pages; else 0 */
  int grid_splits;    /* blocks per (sequence, kv head) in the grid (longest first: the most
                         ranges a sequence can have) */
  int grid_units;     /* longest first: (sequence, range) units in the grid (its z), each
                         8 blocks (one per kv head); else 0 */
  int longest_first;  /* several waves of ticket blocks: units taken longest sequence first */
} pkv_plan;

/* INVALID_ARG for null pointers, figures out of range (num_sms, blocks per
 * SM < 1; max_splits outside [1, 128]; max_seq_len not a multiple of 16 in
 * [16, 2048]; max_cluster outside [0, 16]), batch < 1 or num_splits outside
 * [0, max_splits]. */
pkv_status pkv_plan_decode(const pkv_device_figures* dev, int batch, int num_splits,
                           pkv_plan* out);

/* The figures of the handle's device and geometry (no GPU work). */
pkv_status pkv_pool_device_figures(pkv_pool_t pool, pkv_device_figures* out);

/* Synchronises `stream`, then returns and clears the sticky device error
 * flag: PKV_OK, PKV_ERR_OUT_OF_RANGE or PKV_ERR_DEVICE_TIMEOUT (or CUDA if
 * the synchronisation itself failed). */
pkv_status pkv_get_error(pkv_pool_t pool, void* stream);

/* Decode attention that allocates no device memory. This entry point has no
 * counterpart in the pages; it exists for callers that may not allocate:
 * code running under another component's memory allocator (a framework or
 * server that owns every device allocation and forbids direct cudaMalloc),
 * latency-critical loops that cannot afford the implicit synchronisation and
 * possible failure of an allocation, and hosts that must never hit
 * out-of-memory after start-up. It needs no pool handle.
 *
 * It computes what pkv_decode_attention computes, with the same argument
 * meanings and layouts, and always merges splits through partials and
 * tickets. Those live in one file-scope device array of this library,
 * about 2.1 MiB, which every GPU that loads the library holds until the
 * process exits. Limits: 1 <= num_splits <= 16, batch <= 256 and
 * batch x num_splits <= 256; larger requests return PKV_ERR_STATIC_LIMIT
 * and launch nothing. Geometry arguments describe the caller's pool and
 * tables (num_layers, num_pages, max_batch = block-table rows per layer,
 * max_seq_len = 16 x block-table row length).
 *
 * error_bits: optional device int the caller allocates and zeroes; device
 * index errors (page id, seq_len) are OR-ed into it. NULL: not reported.
 *
 * The first call on each device does a one-time set-up (looks up the
 * array's device address and sets the kernel's shared-memory limit); make
 * that first call before any stream capture. The ticket counters are
 * cleared on the stream at every call. All calls share the one array, so
 * calls that may overlap on the GPU (on different streams, or from several
 * host threads) race and must be serialised by the caller. */
pkv_status pkv_decode_attention_noalloc(int layer, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* block_tables,
                                        const int32_t* seq_lens, float* out, int num_layers,
                                        int num_pages, int max_batch, int max_seq_len,
                                        int batch, int num_splits, int* error_bits,
                                        void* stream);

/* Static text for a status code. */
const char* pkv_status_string(pkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
