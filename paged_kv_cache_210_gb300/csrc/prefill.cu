// Prefill over the shared KV page pool for GB300 (sm_103a): the chunk's K/V
// are written into their pages, then causal attention of the chunk's tokens
// over the pages runs on the fifth-generation tensor cores. The C ABI is
// declared in include/pkv_prefill.h.
//
// Method: prefill fills a prompt's pages with its K/V and every prompt token
// attends causally to the tokens up to itself [samir-vllm: Build LLM
// Inference From Scratch in C++ and CUDA, "Architecture walkthrough",
// Prefill and KV cache paragraphs; 6 Hours of YouTube and 85 handtyped
// pages of notes on LLM Inference - Start here, README feature list, dense
// causal prefill bullet]. The pages' engine runs prefill as dense causal
// attention; here it reads keys through the block table, so a chunk can
// continue a prompt whose earlier pages are already cached.
//
// Attention kernel, one CTA per (sequence, kv head, 64-token query tile),
// warp-specialised:
//  * the 256 rows of the tile are its 64 tokens x the 4 query heads of the
//    kv head (row = token * 4 + head), so every K/V page tile is shared by
//    the group, as in decode; they are two row halves of 128, each the M of
//    its own tensor-core products (M 128 is the largest a single CTA issues);
//  * two loader warps bring Q (32 KiB) and per step 4 pages of K and of V
//    (64 keys, 8 KiB each) by TMA tensor copies (cp.async.bulk.tensor) with
//    the 128-byte swizzle, K in a 6-stage and V in a 5-stage ring; each warp
//    copies one tensor, a step's 4 pages in one round (one wait for the free
//    stage, one copy instruction across lanes 0..3); a page's tile is
//    addressed by its id in the block table, nothing is gathered into a
//    contiguous buffer;
//  * a score warp (one thread) issues S = Q K^T (two M 128 x N 64 x K 64
//    products, one per row half, their K 16 slices interleaved) up to three
//    steps ahead into three pairs of tensor-memory tiles, and two value
//    warps (one thread each, one per row half) issue O += P V (M 128 x N 64
//    x K 64, high and low parts) into FP32 accumulators that stay in tensor
//    memory, as tcgen05.mma kind::f16 completed on mbarriers through
//    tcgen05.commit, which also tell the loader when a stage is free and the
//    score warp when a tile is (the value barriers count both halves);
//  * eight softmax warps, one per (tensor-memory lane quarter, row half):
//    each thread owns one row and reads all 64 keys of the step, so no
//    thread needs another's maximum or sum and the step loop has no block
//    barrier; online softmax in base 2 whose max moves only when the row's
//    max grows by more than 2^8 (O is then rescaled in tensor memory by that
//    thread); the probabilities go back into tensor memory over the scores
//    they came from, as a BF16 high part (truncated) and a BF16 low part,
//    and the value product reads them from there (A operand in tensor
//    memory; ~16 significant bits for P from two MMAs). With three score
//    tiles P is triple-buffered too: the softmax warps wait for a value
//    product only to rescale O. An mbarrier with one arrival per softmax
//    thread hands P over;
//  * one CTA per SM (it holds all 512 tensor-memory columns); tiles run
//    heaviest first (the last tile of a prompt sees the most keys).
//
// What bounds it (measured with clock counters in an instrumented copy):
// with one loader warp for both tensors a step took ~1,850 cycles, a copy
// round costing that warp ~1,800 (the free-stage waits ~400, the 8-lane copy
// instruction ~1,300), so K(j) landed just as the score product wanted it.
// With the tensors split over two loader warps the copies keep ahead, and
// the step (~1,650 cycles) is set by the hand-offs between the warps: each
// mbarrier wait that ends a dependency costs its waiter ~200-500 cycles;
// the softmax threads need ~1,350 cycles of a step.
//
// Every mbarrier wait is bounded (about two seconds of SM clock); a timeout
// sets the error flag, the CTA waits (bounded) for its own copies and
// products in flight, frees its tensor memory and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv.h"
#include "pkv_prefill.h"
#include "device_common.cuh"
#include "pool_internal.h"

using namespace pkv_dev;

namespace {

constexpr int kRowHalves = 2;                        // MMAs of M = 128 rows per CTA
constexpr int kHalfRows = 128;                       // rows of one MMA (its M): 32 tokens
constexpr int kRows = kRowHalves * kHalfRows;        // 256 rows: token x head
constexpr int kTileTokens = kRows / kGroup;          // 64 query tokens per CTA
constexpr int kCtasPerSm = 2 / kRowHalves;           // tensor memory: 256 columns per row half
constexpr int kStepKeys = 64;                        // keys per step: the S MMA's N
constexpr int kStepPages = kStepKeys / kPage;        // 4
constexpr int kSoftmaxWarps = 4 * kRowHalves;        // one per (lane quarter, row half)
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kLoadWarp = kSoftmaxWarps;             // TMA copies: Q and K, then V (+ 1)
constexpr int kScoreWarp = kSoftmaxWarps + 2;        // S = Q K^T products
constexpr int kValueWarp0 = kSoftmaxWarps + 3;       // O += P V products, one warp per row half
constexpr int kThreads = kSoftmaxThreads + 96 + 32 * kRowHalves;
constexpr int kKStages = kRowHalves == 2 ? 6 : 4;     // K ring
constexpr int kVStages = kRowHalves == 2 ? 5 : 3;     // V ring
constexpr int kSTiles = 3;                           // score (then P) tiles in tensor memory
constexpr uint32_t kTmemCols = 256 * kRowHalves;     // S/P tiles, then O
constexpr uint32_t kTmemO = kSTiles * kRowHalves * kStepKeys;   // O of row half h at + 64 h
constexpr float kRescaleLog2 = 8.f;                  // lazy max: p <= 2^8

struct PrefillSmem {                                 // every tile 1024-byte aligned
  uint8_t q[kRows * kRowBytes];                      // 32 KiB
  uint8_t k[kKStages][kStepKeys * kRowBytes];        // 6 x 8 KiB
  uint8_t v[kVStages][kStepKeys * kRowBytes];        // 5 x 8 KiB
  unsigned long long bar_q, bar_k[kKStages], bar_v[kVStages], bar_s[kSTiles], bar_p[kSTiles];
  unsigned long long bar_o[kSTiles];   // P(j) V(j) (and every earlier product) done, per tile
  unsigned long long p_free[kSTiles];                // tile (S, then P) read by its value product
  unsigned long long k_free[kKStages], v_free[kVStages];   // stage read by its product
  uint32_t tmem_base;
  int abort_flag;
  int pages[kMaxPages];                              // block-table row, -1 = not loadable
};
static_assert(offsetof(PrefillSmem, k) % 1024 == 0 && offsetof(PrefillSmem, v) % 1024 == 0 &&
                  (kHalfRows * kRowBytes) % 1024 == 0,
              "swizzled tiles (and Q's second row half) start on 1024-byte boundaries");
// kCtasPerSm CTAs share an SM's 512 tensor-memory columns (the registers
// of their threads admit no more)
static_assert(kCtasPerSm * (sizeof(PrefillSmem) + 2048) <= 228 * 1024,
              "shared memory holds kCtasPerSm prefill CTAs per SM");
constexpr size_t kSmemBytes = sizeof(PrefillSmem) + 1024;   // + room to align the base

struct PrefillParams {
  const int32_t* table;       // this layer's block tables [max_batch][table_stride]
  const int32_t* cu_tokens;   // [batch + 1]
  const int32_t* start_pos;   // [batch]
  float* out;                 // [total][32][64]
  int* err;
  int num_pages;
  int table_stride;
  int max_seq_len;
  int tiles_max;              // gridDim.y: tiles per sequence the launch covers
  int total_tokens;           // rows of q and out
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ int lane_of(int tid) { return tid & 31; }

// Generic-proxy writes to shared memory become visible to the tensor cores
// and the copy engine (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA tensor copies, global -> shared, completion in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
        "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
        "r"(smem_u32(bar))
      : "memory");
}

// Tensor memory: allocation by one whole warp, address written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, BF16 operands, FP32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A's 128 rows are the tensor-memory lanes,
// its K elements packed two BF16 per 32-bit column (element 2c in the low half).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrive on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane, written
// (completion awaited separately with tmem_wait_st).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (>> 4), descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: FP32 D, BF16 A and B, A K-major, B K-
// or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}


// ---------------------------------------------------------------- fill
// One block of 128 threads per chunk token (blockIdx.x = token of the chunk,
// blockIdx.y = sequence): thread t copies 16-byte chunk (t % 64) % 8 of kv
// head (t % 64) / 8, of K for t < 64 and of V otherwise.
__global__ void __launch_bounds__(128) prefill_fill_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, uint16_t* __restrict__ k_pool,
    uint16_t* __restrict__ v_pool, const int32_t* __restrict__ table,
    const int32_t* __restrict__ cu_tokens, const int32_t* __restrict__ start_pos,
    int table_stride, int num_pages, int max_seq_len, int max_chunk, int total_tokens, int* err) {
  const int i = blockIdx.x;
  const int b = blockIdx.y;
  const int t = threadIdx.x;
  const int row0 = cu_tokens[b];
  const int n = cu_tokens[b + 1] - row0;
  if (row0 < 0 || n < 0 || row0 + n > total_tokens) {   // rows outside the caller's buffers
    if (i == 0 && t == 0) set_error(err, PKV_DEV_ERR_SEQ_LEN);
    return;
  }
  if (i == 0 && t == 0 && n > max_chunk) set_error(err, PKV_DEV_ERR_SEQ_LEN);
  if (i >= n) return;
  const int pos = start_pos[b] + i;
  if (pos < 0 || pos >= max_seq_len) {
    if (t == 0) set_error(err, PKV_DEV_ERR_POSITION);
    return;
  }
  const int page = table[static_cast<size_t>(b) * table_stride + pos / kPage];
  if (page < 0 || page >= num_pages) {
    if (t == 0) set_error(err, PKV_DEV_ERR_PAGE);
    return;
  }
  const int r = t & 63;
  const int head = r >> 3;
  const int chunk = r & 7;
  const size_t row = static_cast<size_t>(row0 + i);
  const uint16_t* src = (t < 64 ? k : v) + (row * kHkv + head) * kDim + chunk * 8;
  uint16_t* dst = (t < 64 ? k_pool : v_pool) +
                  ((static_cast<size_t>(page) * kHkv + head) * kPage + pos % kPage) * kDim +
                  chunk * 8;
  *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
}

// ---------------------------------------------------------------- attention
__global__ void __launch_bounds__(kThreads, kCtasPerSm) prefill_attention_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v, const PrefillParams prm) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw + pad);

  // CTAs are dispatched in linear block order (x fastest): the kv head in x
  // and the tile, counted from the last, in y make that order heaviest first
  const int tile = prm.tiles_max - 1 - static_cast<int>(blockIdx.y);
  const int g = blockIdx.x;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  const int row0 = prm.cu_tokens[b];
  const int n = prm.cu_tokens[b + 1] - row0;
  const int start = prm.start_pos[b];
  if (row0 < 0 || n < 0 || row0 + n > prm.total_tokens) {   // rows outside the caller's buffers
    if (blockIdx.y == 0 && g == 0 && tid == 0) set_error(prm.err, PKV_DEV_ERR_SEQ_LEN);
    return;
  }
  if (blockIdx.y == 0 && g == 0 && tid == 0 && n > prm.tiles_max * kTileTokens)
    set_error(prm.err, PKV_DEV_ERR_SEQ_LEN);
  if (tile * kTileTokens >= n) return;                 // the whole CTA, before any allocation
  if (start < 0 || start + n > prm.max_seq_len) {
    if (tid == 0) set_error(prm.err, PKV_DEV_ERR_POSITION);
    return;
  }
  const int t_valid = min(kTileTokens, n - tile * kTileTokens);
  const int p_first = start + tile * kTileTokens;      // position of the tile's token 0
  const int n_keys = p_first + t_valid;                // keys the tile's last token sees
  const int n_steps = (n_keys + kStepKeys - 1) / kStepKeys;
  const int n_pages = (n_keys + kPage - 1) / kPage;

  // block-table row; ids outside the pool are flagged and not loaded
  const int32_t* trow = prm.table + static_cast<size_t>(b) * prm.table_stride;
  bool bad_page = false;
  for (int i = tid; i < n_pages; i += kThreads) {
    const int id = trow[i];
    const bool ok = id >= 0 && id < prm.num_pages;
    sm.pages[i] = ok ? id : -1;
    bad_page |= !ok;
  }
  if (bad_page) set_error(prm.err, PKV_DEV_ERR_PAGE);

  if (tid == 0) {
    mbar_init(&sm.bar_q, 1);
    for (int i = 0; i < kKStages; ++i) mbar_init(&sm.bar_k[i], 1);
    for (int i = 0; i < kVStages; ++i) mbar_init(&sm.bar_v[i], 1);
    for (int i = 0; i < kSTiles; ++i) mbar_init(&sm.bar_s[i], 1);
    // P(j) ready, one barrier per tile: the softmax warps may run up to two
    // steps ahead of the value products, and a parity wait must never see
    // two completed phases of one barrier
    for (int i = 0; i < kSTiles; ++i) mbar_init(&sm.bar_p[i], kSoftmaxThreads);
    // one per tile as well: the softmax warps may be two value products
    // ahead, and a parity wait on a single barrier could then return for an
    // older product
    // the value barriers complete once both row halves' issuers committed
    for (int i = 0; i < kSTiles; ++i) mbar_init(&sm.bar_o[i], kRowHalves);
    for (int i = 0; i < kSTiles; ++i) mbar_init(&sm.p_free[i], kRowHalves);
    for (int i = 0; i < kKStages; ++i) mbar_init(&sm.k_free[i], 1);
    for (int i = 0; i < kVStages; ++i) mbar_init(&sm.v_free[i], kRowHalves);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  const bool any_bad_page = __syncthreads_or(bad_page);   // also publishes sm.pages
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kLoadWarp || warp == kLoadWarp + 1) {
    // ------------------------------------------------------------ copy engine
    // Two loader warps, one for K (and Q), one for V: a copy round costs its
    // warp a few hundred cycles whatever it copies, so the two tensors' rounds
    // run side by side. Each round: lane 0 waits until the step's stage is
    // free (its products committed) and sets the expected bytes, then lanes
    // 0..3 copy the step's 4 pages in one instruction.
    const int lane = lane_of(tid);
    const bool is_v = warp != kLoadWarp;
    const CUtensorMap* map = is_v ? &tmap_v : &tmap_k;
    const int stages = is_v ? kVStages : kKStages;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
      if (!is_v) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
        mbar_arrive_expect_tx(&sm.bar_q, kRows * kRowBytes);
        tma_load_3d(sm.q, &tmap_q, 0, g * kGroup, row0 + tile * kTileTokens, &sm.bar_q);
      }
    }
    int issued = 0;
    bool ok = true;
    for (int j = 0; j < n_steps; ++j) {
      const int st = j % stages;
      unsigned long long* full = is_v ? &sm.bar_v[st] : &sm.bar_k[st];
      bool good = true;
      if (lane == 0) {
        good = *abort_flag == 0;
        if (good && j >= stages)
          good = mbar_wait(is_v ? &sm.v_free[st] : &sm.k_free[st], ((j - stages) / stages) & 1);
        if (good) {
          int valid = 0;
          for (int q = 0; q < kStepPages; ++q) {
            const int lp = j * kStepPages + q;
            valid += (lp < n_pages && sm.pages[lp] >= 0) ? 1 : 0;
          }
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(valid) * kPage * kRowBytes);
        }
      }
      if (!__shfl_sync(0xffffffffu, good ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      if (lane < kStepPages) {
        const int lp = j * kStepPages + lane;
        const int page = lp < n_pages ? sm.pages[lp] : -1;
        // the pool seen as rows of 64 dims: (page, kv head, token) -> row
        if (page >= 0)
          tma_load_2d((is_v ? sm.v[st] : sm.k[st]) + lane * kPage * kRowBytes, map, 0,
                      (page * kHkv + g) * kPage, full);
      }
      __syncwarp();
      ++issued;
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        set_error(prm.err, PKV_DEV_ERR_TIMEOUT);
      }
      // every copy issued lands before the CTA frees its memory (last phase
      // of each barrier; every wait bounded)
      if (!is_v) mbar_wait(&sm.bar_q, 0);
      for (int s = 0; s < stages; ++s) {
        const int uses = (issued - s + stages - 1) / stages;
        if (uses > 0) mbar_wait(is_v ? &sm.bar_v[s] : &sm.bar_k[s], (uses - 1) & 1);
      }
    }
  } else if (warp == kScoreWarp || (warp >= kValueWarp0 && warp < kValueWarp0 + kRowHalves)) {
    // ------------------------------------------------------------ tensor cores
    // Three issuing threads: one for the score products and one per row half
    // for the value products (a tcgen05.commit tracks the products of its
    // own thread), so scores can run ahead while the value products wait for
    // P, and the two halves' value products, each a chain of accumulations
    // into its own O, overlap in the tensor pipe.
    if (lane_of(tid) == 0) {
      const bool scores = warp == kScoreWarp;
      const int half = warp - kValueWarp0;   // the value issuer's row half
      int issued = 0;
      bool ok = true;
      if (scores) {
        const uint32_t idesc_s = instr_desc(kHalfRows, kStepKeys, false);
        const uint64_t q_desc = smem_desc_sw128(smem_u32(sm.q), 16, 1024);
        ok = mbar_wait(&sm.bar_q, 0);
        for (int j = 0; ok && j < n_steps; ++j) {
          // S(j) = Q K(j)^T into tile j % 3, once K(j) landed and the value
          // product of P(j - 3), written over S(j - 3) in that tile, is done
          if (*abort_flag || !mbar_wait(&sm.bar_k[j % kKStages], (j / kKStages) & 1) ||
              (j >= kSTiles &&
               !mbar_wait(&sm.p_free[j % kSTiles], ((j - kSTiles) / kSTiles) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t k_desc = smem_desc_sw128(smem_u32(sm.k[j % kKStages]), 16, 1024);
          // the descriptor's start address counts 16-byte units: + bytes >> 4;
          // row half h reads Q rows 128 h .. 128 h + 127 into its own S tile
          // the row halves' accumulations interleaved: two independent
          // chains keep the tensor pipe busy while one waits on its operand
          #pragma unroll
          for (int kk = 0; kk < kDim / 16; ++kk) {
            #pragma unroll
            for (int h = 0; h < kRowHalves; ++h)
              mma_bf16(tmem + ((j % kSTiles) * kRowHalves + h) * kStepKeys,
                       q_desc + h * (kHalfRows * kRowBytes >> 4) + kk * 2, k_desc + kk * 2,
                       idesc_s, kk > 0);
          }
          mma_commit(&sm.bar_s[j % kSTiles]);
          mma_commit(&sm.k_free[j % kKStages]);
          ++issued;
        }
      } else {
        const uint32_t idesc_o = instr_desc(kHalfRows, kDim, true);
        for (int j = 0; ok && j < n_steps; ++j) {
          // O += P(j) V(j): P from tensor memory (tile j % 3: high part in
          // columns 0..31, low part in 32..63, 16 keys per 8 columns), once
          // the softmax warps handed it over and V(j) landed
          if (*abort_flag || !mbar_wait(&sm.bar_p[j % kSTiles], (j / kSTiles) & 1) ||
              !mbar_wait(&sm.bar_v[j % kVStages], (j / kVStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t v_desc = smem_desc_sw128(smem_u32(sm.v[j % kVStages]), 8192, 1024);
          // this issuer's row half: P tile columns 0..31 high parts, 32..63 low
          const uint32_t p_tile = tmem + ((j % kSTiles) * kRowHalves + half) * kStepKeys;
          const uint32_t o_tile = tmem + kTmemO + half * kDim;
          #pragma unroll
          for (int kk = 0; kk < kStepKeys / 16; ++kk)
            mma_bf16_tmem_a(o_tile, p_tile + kk * 8, v_desc + kk * (16 * kRowBytes >> 4),
                            idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          #pragma unroll
          for (int kk = 0; kk < kStepKeys / 16; ++kk)
            mma_bf16_tmem_a(o_tile, p_tile + 32 + kk * 8,
                            v_desc + kk * (16 * kRowBytes >> 4), idesc_o, 1u);
          mma_commit(&sm.bar_o[j % kSTiles]);
          mma_commit(&sm.v_free[j % kVStages]);
          mma_commit(&sm.p_free[j % kSTiles]);
          ++issued;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(prm.err, PKV_DEV_ERR_TIMEOUT);
      }
      // every product this thread issued completes before the CTA frees its memory
      if (scores) {
        for (int t = 0; t < kSTiles; ++t) {
          const int uses = (issued - t + kSTiles - 1) / kSTiles;
          if (uses > 0) mbar_wait(&sm.bar_s[t], (uses - 1) & 1);
        }
      } else if (issued > 0) {
        // the last product's commit covers every earlier one of this thread
        mbar_wait(&sm.bar_o[(issued - 1) % kSTiles], ((issued - 1) / kSTiles) & 1);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // One thread per row: warp w reads tensor-memory lanes 32 (w % 4) ..
    // + 31 of row half w / 4, all 64 keys of the step, so no thread needs
    // another's maximum or sum and the step loop has no block barrier.
    const int rh = warp >> 2;                           // row half: tokens 32 rh .. 32 rh + 31
    const int r = (warp & 3) * 32 + (tid & 31);         // its MMA row = tensor-memory lane
    const int tok = (rh * kHalfRows + r) >> 2;          // token of the tile, head r & 3
    const uint32_t s_col = rh * kStepKeys;              // the row half's S/P tile columns
    const uint32_t o_col = kTmemO + rh * kDim;          // ... and its O columns
    const int pos = p_first + min(tok, t_valid - 1);    // rows past the chunk mirror its last token
    const float c = 1.4426950408889634f * 0.125f;       // log2(e) / sqrt(64)
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_steps; ++j) {
      // one verdict per warp (the tensor-memory accesses below are warp-wide)
      if (!__all_sync(0xffffffffu, *abort_flag == 0 &&
                                       mbar_wait(&sm.bar_s[j % kSTiles], (j / kSTiles) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t st_tile = tmem + lane_addr + (j % kSTiles) * kRowHalves * kStepKeys + s_col;
      uint32_t sv[64];                                   // the row's 64 keys of the step
      {
        uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tmem_ld32(st_tile, a);
        tmem_ld32(st_tile + 32, b);
      }
      const int key0 = j * kStepKeys;
      if (key0 + kStepKeys - 1 > p_first) {              // some key hidden from some row
        #pragma unroll
        for (int i = 0; i < 64; ++i)
          if (key0 + i > pos) sv[i] = __float_as_uint(-INFINITY);
      }
      float mx8[8];
      #pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = __uint_as_float(sv[e]);
      #pragma unroll
      for (int i = 8; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sv[i]));
      const float m_step = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * c;
      // The max used for the exponentials moves only when the row's max
      // grows by more than 2^8 (so every p <= 2^8).
      float alpha = 1.f;
      const bool grow = m_step > m_run + kRescaleLog2;
      if (grow) {
        alpha = fast_exp2(m_run - m_step);
        m_run = m_step;
        l_run *= alpha;
      }
      // the 64 probabilities, their sum, BF16 high / low parts, in two
      // halves of 32 keys written over the scores they came from (high
      // parts in columns 0..31, low parts in 32..63)
      {
        const float2 c2 = make_float2(c, c);
        const float2 nm2 = make_float2(-m_run, -m_run);
        const float2 neg1 = make_float2(-1.f, -1.f);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        #pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          uint32_t hi[16], lo[16];
          #pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int k = kh * 32 + i;
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), c2, nm2);
            const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            acc[(i >> 1) & 3] = __fadd2_rn(acc[(i >> 1) & 3], pp);
            const uint32_t b0 = __float_as_uint(pp.x), b1 = __float_as_uint(pp.y);
            hi[i / 2] = __byte_perm(b0, b1, 0x7632);
            const float2 h = make_float2(__uint_as_float(b0 & 0xffff0000u),
                                         __uint_as_float(b1 & 0xffff0000u));
            const float2 rest = __ffma2_rn(h, neg1, pp);
            lo[i / 2] = float2_to_bf16x2(rest.x, rest.y);
          }
          // the scores of both halves are in registers already: P may overwrite them
          tmem_st16(st_tile + kh * 16, hi);
          tmem_st16(st_tile + 32 + kh * 16, lo);
        }
        const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        l_run += a.x + a.y;
      }

      // a row that grew its max rescales its O, once P(j - 1) V(j - 1) is
      // done (P(j) V(j) cannot start before this thread hands over P(j))
      bool failed = false;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        failed = !__all_sync(0xffffffffu,
                             mbar_wait(&sm.bar_o[(j - 1) % kSTiles], ((j - 1) / kSTiles) & 1));
        tc_fence_after();
        if (!failed) {
          #pragma unroll
          for (int dh = 0; dh < 2; ++dh) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_addr + o_col + dh * 32, ov);
            #pragma unroll
            for (int d = 0; d < 32; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
            tmem_st32(tmem + lane_addr + o_col + dh * 32, ov);
          }
        }
      }
      // V rows the product must not see: keys past the tile's last token and
      // pages not loaded (zero, so that p = 0 times them stays 0); every
      // softmax thread zeroes its share before it hands over P(j)
      if (!failed && (any_bad_page || (j + 1) * kStepKeys > n_keys)) {
        if (__all_sync(0xffffffffu, mbar_wait(&sm.bar_v[j % kVStages], (j / kVStages) & 1))) {
          for (int idx = tid; idx < kStepKeys * 8; idx += kSoftmaxThreads) {
            const int key_row = idx >> 3;
            const int key = j * kStepKeys + key_row;
            const int lp = key / kPage;
            if (key >= n_keys || lp >= n_pages || sm.pages[lp] < 0)
              *reinterpret_cast<uint4*>(sm.v[j % kVStages] + key_row * kRowBytes + (idx & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        } else {
          failed = true;
        }
      }
      if (failed) {
        ok = false;
        break;
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.bar_p[j % kSTiles]);
    }
    if (!ok) {
      *abort_flag = 1;
      set_error(prm.err, PKV_DEV_ERR_TIMEOUT);
    }
    if (ok && !*abort_flag &&
        mbar_wait(&sm.bar_o[(n_steps - 1) % kSTiles], ((n_steps - 1) / kSTiles) & 1)) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      float* dst = prm.out + ((static_cast<size_t>(row0) + tile * kTileTokens + tok) * kHq +
                              g * kGroup + (r & 3)) * kDim;
      #pragma unroll
      for (int dh = 0; dh < 2; ++dh) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_addr + o_col + dh * 32, ov);
        if (tok < t_valid) {
          #pragma unroll
          for (int d = 0; d < 32; d += 4)
            *reinterpret_cast<float4*>(dst + dh * 32 + d) =
                make_float4(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv,
                            __uint_as_float(ov[d + 2]) * inv, __uint_as_float(ov[d + 3]) * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major BF16 tensor, dims innermost first, 128-byte swizzle.
bool encode_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                 const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t elem[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
            strides_bytes, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool set_smem_attribute(int device) {
  constexpr int kMaxDevices = 64;
  static std::mutex lock;
  static bool done[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return false;
  std::lock_guard<std::mutex> guard(lock);
  if (!done[device]) {
    if (cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return false;
    done[device] = true;
  }
  return true;
}

pkv_status check_common(pkv_pool_t pool, int layer, int batch, int max_chunk_tokens,
                        const int32_t* block_tables, const int32_t* cu_tokens,
                        const int32_t* start_pos) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  if (layer < 0 || layer >= c.num_layers || batch < 0 || batch > c.max_batch)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (max_chunk_tokens < 1 || max_chunk_tokens > c.max_seq_len) return PKV_ERR_INVALID_ARG;
  if (!block_tables || !cu_tokens || !start_pos || !pkv_aligned16(block_tables) ||
      !pkv_aligned16(cu_tokens) || !pkv_aligned16(start_pos))
    return PKV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

pkv_status launch_fill(pkv_pool_t pool, int layer, const void* k, const void* v, void* k_pool,
                       void* v_pool, const int32_t* block_tables, const int32_t* cu_tokens,
                       const int32_t* start_pos, int batch, int total_tokens,
                       int max_chunk_tokens, void* stream) {
  pkv_status st = check_common(pool, layer, batch, max_chunk_tokens, block_tables, cu_tokens,
                               start_pos);
  if (st != PKV_OK || batch == 0) return st;
  if (total_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (total_tokens == 0) return PKV_OK;
  if (!k || !v || !k_pool || !v_pool || !pkv_aligned16(k) || !pkv_aligned16(v) ||
      !pkv_aligned16(k_pool) || !pkv_aligned16(v_pool))
    return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  const int stride = c.max_seq_len / kPage;
  prefill_fill_kernel<<<dim3(max_chunk_tokens, batch), 128, 0,
                        static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
      static_cast<uint16_t*>(k_pool), static_cast<uint16_t*>(v_pool),
      block_tables + static_cast<size_t>(layer) * c.max_batch * stride, cu_tokens, start_pos,
      stride, c.num_pages, c.max_seq_len, max_chunk_tokens, total_tokens, pool->err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status launch_attention(pkv_pool_t pool, int layer, const void* q, const void* k_pool,
                            const void* v_pool, const int32_t* block_tables,
                            const int32_t* cu_tokens, const int32_t* start_pos, float* out,
                            int batch, int total_tokens, int max_chunk_tokens, void* stream) {
  pkv_status st = check_common(pool, layer, batch, max_chunk_tokens, block_tables, cu_tokens,
                               start_pos);
  if (st != PKV_OK || batch == 0) return st;
  if (total_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (total_tokens == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !out || !pkv_aligned16(q) || !pkv_aligned16(k_pool) ||
      !pkv_aligned16(v_pool) || !pkv_aligned16(out))
    return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  if (!set_smem_attribute(pool->device)) return PKV_ERR_CUDA;

  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[3] = {kDim, kHq, static_cast<cuuint64_t>(total_tokens)};
    const cuuint64_t strides[2] = {kRowBytes, static_cast<cuuint64_t>(kHq) * kRowBytes};
    const cuuint32_t box[3] = {kDim, kGroup, kTileTokens};
    if (!encode_bf16(&tq, q, 3, dims, strides, box)) return PKV_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {kDim, static_cast<cuuint64_t>(c.num_pages) * kHkv * kPage};
    const cuuint64_t strides[1] = {kRowBytes};
    const cuuint32_t box[2] = {kDim, kPage};
    if (!encode_bf16(&tk, k_pool, 2, dims, strides, box)) return PKV_ERR_CUDA;
    if (!encode_bf16(&tv, v_pool, 2, dims, strides, box)) return PKV_ERR_CUDA;
  }
  const int stride = c.max_seq_len / kPage;
  PrefillParams prm;
  prm.table = block_tables + static_cast<size_t>(layer) * c.max_batch * stride;
  prm.cu_tokens = cu_tokens;
  prm.start_pos = start_pos;
  prm.out = out;
  prm.err = pool->err;
  prm.num_pages = c.num_pages;
  prm.table_stride = stride;
  prm.max_seq_len = c.max_seq_len;
  prm.tiles_max = (max_chunk_tokens + kTileTokens - 1) / kTileTokens;
  prm.total_tokens = total_tokens;
  prefill_attention_kernel<<<dim3(kHkv, prm.tiles_max, batch), kThreads, kSmemBytes,
                             static_cast<cudaStream_t>(stream)>>>(tq, tk, tv, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_prefill_fill(pkv_pool_t pool, int layer, const void* k, const void* v,
                            void* k_pool, void* v_pool, const int32_t* block_tables,
                            const int32_t* cu_tokens, const int32_t* start_pos, int batch,
                            int total_tokens, int max_chunk_tokens, void* stream) {
  return launch_fill(pool, layer, k, v, k_pool, v_pool, block_tables, cu_tokens, start_pos, batch,
                     total_tokens, max_chunk_tokens, stream);
}

pkv_status pkv_prefill_attention(pkv_pool_t pool, int layer, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables,
                                 const int32_t* cu_tokens, const int32_t* start_pos, float* out,
                                 int batch, int total_tokens, int max_chunk_tokens,
                                 void* stream) {
  return launch_attention(pool, layer, q, k_pool, v_pool, block_tables, cu_tokens, start_pos, out,
                          batch, total_tokens, max_chunk_tokens, stream);
}

pkv_status pkv_prefill(pkv_pool_t pool, int layer, const void* q, const void* k, const void* v,
                       void* k_pool, void* v_pool, const int32_t* block_tables,
                       const int32_t* cu_tokens, const int32_t* start_pos, float* out,
                       int batch, int total_tokens, int max_chunk_tokens, void* stream) {
  pkv_status st = launch_fill(pool, layer, k, v, k_pool, v_pool, block_tables, cu_tokens,
                              start_pos, batch, total_tokens, max_chunk_tokens, stream);
  if (st != PKV_OK) return st;
  return launch_attention(pool, layer, q, k_pool, v_pool, block_tables, cu_tokens, start_pos, out,
                          batch, total_tokens, max_chunk_tokens, stream);
}

}  // extern "C"
