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
// Attention kernel, one CTA of 4 warps per (sequence, kv head, 32-token
// query tile):
//  * the 128 rows of the MMA are the tile's 32 tokens x the 4 query heads
//    of the kv head (row = token * 4 + head), so every K/V page tile is
//    shared by the group, as in decode;
//  * Q (16 KiB) and per step 4 pages of K and of V (64 keys, 8 KiB each)
//    arrive by TMA tensor copies (cp.async.bulk.tensor) with the 128-byte
//    swizzle, K/V double-buffered; a page's tile is addressed by its id in
//    the block table, so nothing is gathered into a contiguous buffer;
//  * S = Q K^T (M 128, N 64, K 64) and the value product O_step = P V
//    (M 128, N 64, K 64) run as tcgen05.mma kind::f16 with FP32
//    accumulators in tensor memory, issued by one thread and completed on
//    mbarriers through tcgen05.commit;
//  * each thread owns one row: it reads its S row from tensor memory,
//    keeps the running max and sum (online softmax in base 2), writes the
//    probabilities to shared memory as a BF16 high part and a BF16 low
//    part (two MMAs, so P carries ~16 significant bits), and accumulates
//    O_step into 64 FP32 registers with the rescale factor;
//  * tiles run heaviest first (the last tile of a prompt sees the most keys).
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
#include "pool_internal.h"

namespace {

constexpr int kPage = 16;
constexpr int kHq = 32;
constexpr int kHkv = 8;
constexpr int kGroup = kHq / kHkv;
constexpr int kDim = 64;
constexpr int kMaxSeqLen = 2048;
constexpr int kMaxPages = kMaxSeqLen / kPage;
constexpr int kRowBytes = kDim * 2;                  // 128 B: one swizzle row
constexpr int kTileTokens = 32;                      // query tokens per CTA
constexpr int kRows = kTileTokens * kGroup;          // 128: the MMA's M
constexpr int kStepKeys = 64;                        // keys per step: the S MMA's N
constexpr int kStepPages = kStepKeys / kPage;        // 4
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 128;                  // S: columns 0..63, O_step: 64..127
constexpr long long kWaitCycles = 4000000000LL;      // about two seconds

struct PrefillSmem {                                 // every tile 1024-byte aligned
  uint8_t q[kRows * kRowBytes];                      // 16 KiB
  uint8_t k[2][kStepKeys * kRowBytes];               // 2 x 8 KiB
  uint8_t v[2][kStepKeys * kRowBytes];               // 2 x 8 KiB
  uint8_t p_hi[kRows * kRowBytes];                   // 16 KiB
  uint8_t p_lo[kRows * kRowBytes];                   // 16 KiB
  unsigned long long bar_q, bar_kv[2], bar_s, bar_o;
  uint32_t tmem_base;
  int pages[kMaxPages];                              // block-table row, -1 = not loadable
};
static_assert(offsetof(PrefillSmem, k) % 1024 == 0 && offsetof(PrefillSmem, v) % 1024 == 0 &&
                  offsetof(PrefillSmem, p_hi) % 1024 == 0 && offsetof(PrefillSmem, p_lo) % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
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
  int tiles_max;              // gridDim.x: tiles per sequence the launch covers
  int total_tokens;           // rows of q and out
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_error(int* err, int bits) { atomicOr(err, bits); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  constexpr uint32_t kSuspendHintNs = 10000000;
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return done != 0;
}

// Bounded wait on an mbarrier phase: false after about two seconds.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > kWaitCycles) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

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

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3), "r"(smem_u32(bar))
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

// One arrive on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar))
               : "memory");
}

// 64 consecutive FP32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
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

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}

__device__ __forceinline__ float bf16_lo_to_float(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_to_float(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
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
__global__ void __launch_bounds__(kThreads, 1) prefill_attention_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v, const PrefillParams prm) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw + pad);

  const int tile = prm.tiles_max - 1 - static_cast<int>(blockIdx.x);   // heaviest first
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  const int row0 = prm.cu_tokens[b];
  const int n = prm.cu_tokens[b + 1] - row0;
  const int start = prm.start_pos[b];
  if (row0 < 0 || n < 0 || row0 + n > prm.total_tokens) {   // rows outside the caller's buffers
    if (blockIdx.x == 0 && g == 0 && tid == 0) set_error(prm.err, PKV_DEV_ERR_SEQ_LEN);
    return;
  }
  if (blockIdx.x == 0 && g == 0 && tid == 0 && n > prm.tiles_max * kTileTokens)
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
    mbar_init(&sm.bar_kv[0], 1);
    mbar_init(&sm.bar_kv[1], 1);
    mbar_init(&sm.bar_s, 1);
    mbar_init(&sm.bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  const bool any_bad_page = __syncthreads_or(bad_page);   // also publishes sm.pages
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // K/V of step j (pages 4j .. 4j+3) into stage j & 1: thread 0 issues
  auto issue_kv = [&](int j) {
    const int stage = j & 1;
    int valid = 0;
    for (int q = 0; q < kStepPages; ++q) {
      const int lp = j * kStepPages + q;
      valid += (lp < n_pages && sm.pages[lp] >= 0) ? 1 : 0;
    }
    mbar_arrive_expect_tx(&sm.bar_kv[stage], static_cast<uint32_t>(valid) * 2 * kPage * kRowBytes);
    for (int q = 0; q < kStepPages; ++q) {
      const int lp = j * kStepPages + q;
      if (lp < n_pages && sm.pages[lp] >= 0) {
        tma_load_4d(sm.k[stage] + q * kPage * kRowBytes, &tmap_k, 0, 0, g, sm.pages[lp],
                    &sm.bar_kv[stage]);
        tma_load_4d(sm.v[stage] + q * kPage * kRowBytes, &tmap_v, 0, 0, g, sm.pages[lp],
                    &sm.bar_kv[stage]);
      }
    }
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(&sm.bar_q, kRows * kRowBytes);
    tma_load_3d(sm.q, &tmap_q, 0, g * kGroup, row0 + tile * kTileTokens, &sm.bar_q);
    issue_kv(0);
    if (n_steps > 1) issue_kv(1);
  }

  // this thread's row: token tok of the tile, head (tid & 3) of the group
  const int tok = tid >> 2;
  const int pos = p_first + min(tok, t_valid - 1);     // rows past the chunk mirror its last token
  const float c = 1.4426950408889634f * 0.125f;        // log2(e) / sqrt(64)
  const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t idesc_s = instr_desc(kRows, kStepKeys, false);
  const uint32_t idesc_o = instr_desc(kRows, kDim, true);
  const uint32_t q_addr = smem_u32(sm.q);
  const uint32_t phi_addr = smem_u32(sm.p_hi);
  const uint32_t plo_addr = smem_u32(sm.p_lo);

  float o[kDim];
  #pragma unroll
  for (int d = 0; d < kDim; ++d) o[d] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  bool failed = !mbar_wait(&sm.bar_q, 0);
  int kv_waited = 0;          // steps whose K/V this CTA has waited for
  int kv_issued = min(n_steps, 2);
  bool s_pending = false, o_pending = false;
  int j = 0;
  for (; j < n_steps; ++j) {
    const int stage = j & 1;
    bool ok = mbar_wait(&sm.bar_kv[stage], (j >> 1) & 1);
    if (ok) kv_waited = j + 1;
    // V rows the product must not see: keys past the tile's last token and
    // pages not loaded (zero, so that p = 0 times them stays 0)
    if (ok && (any_bad_page || (j + 1) * kStepKeys > n_keys)) {
      for (int idx = tid; idx < kStepKeys * 8; idx += kThreads) {
        const int key_row = idx >> 3;
        const int key = j * kStepKeys + key_row;
        const int lp = key / kPage;
        if (key >= n_keys || lp >= n_pages || sm.pages[lp] < 0)
          *reinterpret_cast<uint4*>(sm.v[stage] + key_row * kRowBytes + (idx & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    if (__syncthreads_or(failed || !ok)) {
      failed = true;
      break;
    }

    // S = Q K^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t k_addr = smem_u32(sm.k[stage]);
      #pragma unroll
      for (int kk = 0; kk < kDim / 16; ++kk)
        mma_bf16(tmem, smem_desc_sw128(q_addr + kk * 32, 16, 1024),
                 smem_desc_sw128(k_addr + kk * 32, 16, 1024), idesc_s, kk > 0);
      mma_commit(&sm.bar_s);
    }
    s_pending = true;
    ok = mbar_wait(&sm.bar_s, j & 1);
    s_pending = !ok;
    tc_fence_after();
    uint32_t sraw[kStepKeys];
    tmem_ld64(tmem + lane_addr, sraw);

    // online softmax over this step's keys (base 2)
    const int key0 = j * kStepKeys;
    float m_step = -INFINITY;
    #pragma unroll
    for (int i = 0; i < kStepKeys; ++i) {
      const float s = key0 + i <= pos ? __uint_as_float(sraw[i]) * c : -INFINITY;
      sraw[i] = __float_as_uint(s);
      m_step = fmaxf(m_step, s);
    }
    const float m_new = fmaxf(m_run, m_step);
    const float alpha = fast_exp2(m_run - m_new);
    float sum = 0.f;
    #pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t hi[4], lo[4];
      #pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = fast_exp2(__uint_as_float(sraw[ch * 8 + 2 * e]) - m_new);
        const float p1 = fast_exp2(__uint_as_float(sraw[ch * 8 + 2 * e + 1]) - m_new);
        sum += p0 + p1;
        hi[e] = pack_bf16x2(p0, p1);
        lo[e] = pack_bf16x2(p0 - bf16_lo_to_float(hi[e]), p1 - bf16_hi_to_float(hi[e]));
      }
      const uint32_t off = static_cast<uint32_t>(tid * kRowBytes + ((ch ^ (tid & 7)) << 4));
      *reinterpret_cast<uint4*>(sm.p_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sm.p_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    l_run = l_run * alpha + sum;
    m_run = m_new;
    #pragma unroll
    for (int d = 0; d < kDim; ++d) o[d] *= alpha;
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }

    // O_step = P_hi V + P_lo V
    if (tid == 0) {
      tc_fence_after();
      const uint32_t v_addr = smem_u32(sm.v[stage]);
      #pragma unroll
      for (int kk = 0; kk < kStepKeys / 16; ++kk)
        mma_bf16(tmem + kDim, smem_desc_sw128(phi_addr + kk * 32, 16, 1024),
                 smem_desc_sw128(v_addr + kk * 16 * kRowBytes, 8192, 1024), idesc_o, kk > 0);
      #pragma unroll
      for (int kk = 0; kk < kStepKeys / 16; ++kk)
        mma_bf16(tmem + kDim, smem_desc_sw128(plo_addr + kk * 32, 16, 1024),
                 smem_desc_sw128(v_addr + kk * 16 * kRowBytes, 8192, 1024), idesc_o, 1);
      mma_commit(&sm.bar_o);
    }
    o_pending = true;
    ok = mbar_wait(&sm.bar_o, j & 1);
    o_pending = !ok;
    tc_fence_after();
    uint32_t oraw[kDim];
    tmem_ld64(tmem + lane_addr + kDim, oraw);
    #pragma unroll
    for (int d = 0; d < kDim; ++d) o[d] += __uint_as_float(oraw[d]);

    // both products of this step are done: its K/V stage can be refilled
    if (ok && tid == 0 && j + 2 < n_steps) {
      issue_kv(j + 2);
      kv_issued = j + 3;
    }
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
  }

  if (failed) {
    if (tid == 0) set_error(prm.err, PKV_DEV_ERR_TIMEOUT);
    // let this CTA's copies and products in flight land (each wait bounded)
    for (int w = kv_waited; w < kv_issued; ++w) mbar_wait(&sm.bar_kv[w & 1], (w >> 1) & 1);
    if (s_pending) mbar_wait(&sm.bar_s, j & 1);
    if (o_pending) mbar_wait(&sm.bar_o, j & 1);
  } else if (tok < t_valid) {
    const float inv = 1.f / l_run;
    float* dst = prm.out + ((static_cast<size_t>(row0) + tile * kTileTokens + tok) * kHq +
                            g * kGroup + (tid & 3)) * kDim;
    #pragma unroll
    for (int d = 0; d < kDim; d += 4)
      *reinterpret_cast<float4*>(dst + d) =
          make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
  if (!block_tables || !cu_tokens || !start_pos || !aligned16(block_tables) ||
      !aligned16(cu_tokens) || !aligned16(start_pos))
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
  if (!k || !v || !k_pool || !v_pool || !aligned16(k) || !aligned16(v) || !aligned16(k_pool) ||
      !aligned16(v_pool))
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
  if (!q || !k_pool || !v_pool || !out || !aligned16(q) || !aligned16(k_pool) ||
      !aligned16(v_pool) || !aligned16(out))
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
    const cuuint64_t dims[4] = {kDim, kPage, kHkv, static_cast<cuuint64_t>(c.num_pages)};
    const cuuint64_t strides[3] = {kRowBytes, static_cast<cuuint64_t>(kPage) * kRowBytes,
                                   static_cast<cuuint64_t>(kHkv) * kPage * kRowBytes};
    const cuuint32_t box[4] = {kDim, kPage, 1, 1};
    if (!encode_bf16(&tk, k_pool, 4, dims, strides, box)) return PKV_ERR_CUDA;
    if (!encode_bf16(&tv, v_pool, 4, dims, strides, box)) return PKV_ERR_CUDA;
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
  prefill_attention_kernel<<<dim3(prm.tiles_max, kHkv, batch), kThreads, kSmemBytes,
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
