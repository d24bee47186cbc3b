// Paged KV cache decode path for GB300 (sm_103a): append scatter, paged
// decode attention with split-KV and an in-launch log-sum-exp merge, and the
// fused append-then-attend step. The C ABI is declared in include/pkv.h.
//
// Method: decode appends one token's K/V at its absolute position into the
// page its block table names, then streams the sequence's pages in place
// with an FP32 online softmax, with no contiguous gather and no stored
// scores [samir-vllm: Build LLM Inference From Scratch in C++ and CUDA,
// "Architecture walkthrough", KV cache paragraph; 6 Hours of YouTube and 85
// handtyped pages of notes on LLM Inference - Start here, README feature
// list, direct paged decode attention bullet].
//
// Design for sm_103a (what differs from the pages' engine, which streams
// pages once per query head):
//  * one thread block per (sequence, kv head, split) serves the 4 query heads
//    of the group, so each 2 KiB (page, kv head) tile of K and of V is read
//    from HBM exactly once;
//  * each of the block's 4 warps owns every 4th page of the split and its own
//    ring of page stages in shared memory, filled by the bulk-copy engine
//    (cp.async.bulk, completion counted on an mbarrier), so bytes in flight
//    do not depend on registers and warps never wait on each other inside
//    the page loop;
//  * QK: a lane owns 2 tokens x 16 dims for all 4 heads; packed FP32 FMA
//    (two lanes of FP32 per instruction) over dim pairs; a 2-step
//    reduce-scatter leaves each lane with one head's scores for its 2 tokens;
//  * online softmax per page in base 2 (q is pre-scaled by log2(e)/8);
//  * PV: a lane owns 4 dims x every other token for all 4 heads; the
//    probabilities go through a per-warp shared-memory slot, duplicated so
//    that packed FMAs read them as pairs;
//  * warps merge in shared memory; splits merge in the same launch: every
//    split block writes its (o, m, l) partial and takes a ticket, and the
//    last to arrive merges (no spinning);
//  * the score scale 1/8 and log2(e) are folded into q once per block.

#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace {

constexpr int kPage = 16;
constexpr int kHq = 32;
constexpr int kHkv = 8;
constexpr int kGroup = kHq / kHkv;
constexpr int kDim = 64;
constexpr int kMaxSeqLen = 2048;
constexpr int kRowBytes = kDim * 2;             // one token of one kv head: 128 B
constexpr int kTileBytes = kPage * kRowBytes;   // one (page, kv head) tile: 2 KiB
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;                       // page stages per warp
constexpr int kDefaultMaxSplits = 64;
constexpr int kMaxSplitsLimit = 128;

// device error flag bits
constexpr int kErrPage = 1;
constexpr int kErrPosition = 2;
constexpr int kErrSeqLen = 4;
constexpr int kErrTimeout = 8;

// about two seconds at the maximum SM clock
constexpr long long kWaitCycles = 4000000000LL;

struct WarpSmem {
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  float2 p[kPage][kGroup];   // (p, p) per token and head
  float2 alpha[kGroup];      // (alpha, alpha) per head
  unsigned long long bar[kStages];
};

struct BlockSmem {
  WarpSmem warp[kWarps];
  float m[kWarps][kGroup];
  float l[kWarps][kGroup];
  float acc[kWarps][kGroup][kDim];
  int last;
};

static_assert(sizeof(WarpSmem) % 16 == 0, "warp slab must keep 16-byte alignment");

struct DecodeParams {
  const uint16_t* q;          // [B][32][64]
  const uint16_t* k_new;      // [B][8][64]   (fused only)
  const uint16_t* v_new;
  uint16_t* k_pool;           // [num_pages][8][16][64]
  uint16_t* v_pool;
  const int32_t* table;       // this layer's block tables: [max_batch][table_stride]
  const int32_t* seq_lens;    // [B]
  float* out;                 // [B][32][64]
  float* part_o;              // [max_batch][32][max_splits][64] (this layer's parity)
  float2* part_ml;            // [max_batch][32][max_splits]
  int* tickets;               // [max_batch][8]
  int* err;
  int num_pages;
  int table_stride;
  int max_seq_len;
  int max_splits;
  int num_splits;             // > 0: S ranges per sequence
  int chunk_pages;            // > 0: ranges of this many pages (used when num_splits == 0)
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
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

// Bulk copy global -> shared (the copy engine), completion counted in bytes
// on `bar`. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// BF16 pair (low half = element 0) -> two FP32 values, exact.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  return __ffma2_rn(a, b, c);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ void set_error(int* err, int bits) { atomicOr(err, bits); }

// ---------------------------------------------------------------- append
// One block of 128 threads per sequence: thread t copies 16-byte chunk
// (t % 64) % 8 of kv head (t % 64) / 8, of K for t < 64 and of V otherwise.
__global__ void __launch_bounds__(128) append_kernel(const uint16_t* __restrict__ k,
                                                     const uint16_t* __restrict__ v,
                                                     uint16_t* __restrict__ k_pool,
                                                     uint16_t* __restrict__ v_pool,
                                                     const int32_t* __restrict__ table,
                                                     const int32_t* __restrict__ positions,
                                                     int table_stride, int num_pages,
                                                     int max_seq_len, int* err) {
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  const int pos = positions[b];
  if (pos < 0 || pos >= max_seq_len) {
    if (t == 0) set_error(err, kErrPosition);
    return;
  }
  const int page = table[static_cast<size_t>(b) * table_stride + pos / kPage];
  if (page < 0 || page >= num_pages) {
    if (t == 0) set_error(err, kErrPage);
    return;
  }
  const int slot = pos % kPage;
  const int r = t & 63;
  const int head = r >> 3;
  const int chunk = r & 7;
  const uint16_t* src = (t < 64 ? k : v) + (static_cast<size_t>(b) * kHkv + head) * kDim + chunk * 8;
  uint16_t* dst = (t < 64 ? k_pool : v_pool) +
                  ((static_cast<size_t>(page) * kHkv + head) * kPage + slot) * kDim + chunk * 8;
  *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
}

// ---------------------------------------------------------------- decode
template <bool kFused>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(const DecodeParams prm) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  BlockSmem& sm = *reinterpret_cast<BlockSmem*>(smem_raw);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int len = prm.seq_lens[b];
  if (len < 1 || len > prm.max_seq_len) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) set_error(prm.err, kErrSeqLen);
    return;
  }
  const int n_pages = (len + kPage - 1) / kPage;
  const int chunk = prm.num_splits > 0 ? (n_pages + prm.num_splits - 1) / prm.num_splits
                                       : prm.chunk_pages;
  const int n_splits = (n_pages + chunk - 1) / chunk;   // non-empty splits of this sequence
  if (split >= n_splits) return;
  const int page_begin = split * chunk;
  const int page_end = min(n_pages, page_begin + chunk);
  const int last_page = n_pages - 1;
  const int new_slot = (len - 1) % kPage;               // slot of the appended token
  const int32_t* row = prm.table + static_cast<size_t>(b) * prm.table_stride;

  WarpSmem& ws = sm.warp[warp];
  // pages of this warp: page_begin + warp + 4 i
  const int mine = page_begin + warp < page_end
                       ? (page_end - (page_begin + warp) + kWarps - 1) / kWarps
                       : 0;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&ws.bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Issue the copies of this warp's i-th page into stage i % kStages. Every
  // lane calls it; lane 0 drives the copy engine, lanes 0..15 place the
  // appended token in the fused step.
  auto issue = [&](int i) {
    const int stage = i % kStages;
    const int lp = page_begin + warp + kWarps * i;
    const int phys = row[lp];
    const bool ok = phys >= 0 && phys < prm.num_pages;
    int rows = lp == last_page ? len - lp * kPage : kPage;
    if (kFused && lp == last_page) rows = new_slot;     // the new row comes from k/v
    if (lane == 0) {
      if (!ok) set_error(prm.err, kErrPage);
      if (ok && rows > 0) {
        const uint32_t bytes = static_cast<uint32_t>(rows) * kRowBytes;
        const size_t tile = (static_cast<size_t>(phys) * kHkv + kvh) * (kPage * kDim);
        mbar_arrive_expect_tx(&ws.bar[stage], 2 * bytes);
        bulk_load(ws.k[stage], prm.k_pool + tile, bytes, &ws.bar[stage]);
        bulk_load(ws.v[stage], prm.v_pool + tile, bytes, &ws.bar[stage]);
      } else {
        mbar_arrive(&ws.bar[stage]);
      }
    }
    if (kFused && lp == last_page && ok && lane < 16) {
      const bool is_v = lane >= 8;
      const int c = lane & 7;
      const uint16_t* src = (is_v ? prm.v_new : prm.k_new) +
                            (static_cast<size_t>(b) * kHkv + kvh) * kDim + c * 8;
      const uint4 val = __ldg(reinterpret_cast<const uint4*>(src));
      uint16_t* pool = is_v ? prm.v_pool : prm.k_pool;
      *reinterpret_cast<uint4*>(pool + ((static_cast<size_t>(phys) * kHkv + kvh) * kPage +
                                        new_slot) * kDim + c * 8) = val;
      uint8_t* tile = is_v ? ws.v[stage] : ws.k[stage];
      *reinterpret_cast<uint4*>(tile + new_slot * kRowBytes + c * 16) = val;
    }
  };

  const int n_prefetch = min(mine, kStages);
  for (int i = 0; i < n_prefetch; ++i) issue(i);
  int issued = n_prefetch;
  __syncwarp();   // the appended row written by lanes 0..15 is read by every lane

  // ---- lane roles
  const int tp = lane >> 2;            // QK: tokens tp and tp + 8
  const int qd = lane & 3;             // QK: 16-byte chunks qd and qd + 4
  const int par = tp & 1;
  const int cA = qd + 4 * par;         // chunk read first (bank-conflict-free order)
  const int cB = qd + 4 * (1 - par);
  const int gh = 2 * (qd & 1) + ((qd >> 1) & 1);   // head owned after reduce-scatter
  const int dq = lane & 15;            // PV: dims 4 dq .. 4 dq + 3
  const int tpar = lane >> 4;          // PV: tokens 2 i + tpar

  // q of the 4 heads for this lane's chunks, scaled by log2(e) / sqrt(64)
  const float qscale = 1.4426950408889634f * 0.125f;
  float2 qa[kGroup][4], qb[kGroup][4];
  {
    const uint16_t* qrow = prm.q + (static_cast<size_t>(b) * kHq + kvh * kGroup) * kDim;
    #pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const uint4 ra = __ldg(reinterpret_cast<const uint4*>(qrow + g * kDim + cA * 8));
      const uint4 rb = __ldg(reinterpret_cast<const uint4*>(qrow + g * kDim + cB * 8));
      const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
      const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
      #pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fa = bf16x2_to_float2(wa[j]);
        const float2 fb = bf16x2_to_float2(wb[j]);
        qa[g][j] = make_float2(fa.x * qscale, fa.y * qscale);
        qb[g][j] = make_float2(fb.x * qscale, fb.y * qscale);
      }
    }
  }

  float m_run = -INFINITY;   // running max (base 2) of head gh
  float l_run = 0.f;         // this lane's share of the running sum of head gh
  float2 acc[kGroup][2];     // PV accumulators: dims (4dq, 4dq+1), (4dq+2, 4dq+3)
  #pragma unroll
  for (int g = 0; g < kGroup; ++g) acc[g][0] = acc[g][1] = make_float2(0.f, 0.f);

  bool timed_out = false;
  int consumed = 0;
  for (int i = 0; i < mine; ++i) {
    const int stage = i % kStages;
    const int lp = page_begin + warp + kWarps * i;
    const int valid = lp == last_page ? len - lp * kPage : kPage;   // tokens in this page
    const int phys = row[lp];
    const bool ok = phys >= 0 && phys < prm.num_pages;
    if (!mbar_wait(&ws.bar[stage], (i / kStages) & 1)) {
      timed_out = true;
      break;
    }
    consumed = i + 1;
    const int live = ok ? valid : 0;
    const uint8_t* kt = ws.k[stage];
    const uint8_t* vt = ws.v[stage];

    // ---- scores for tokens tp and tp + 8, all 4 heads, this lane's 16 dims
    float s[kGroup][2];
    #pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint8_t* krow = kt + (tp + 8 * j) * kRowBytes;
      const uint4 ka = *reinterpret_cast<const uint4*>(krow + cA * 16);
      const uint4 kb = *reinterpret_cast<const uint4*>(krow + cB * 16);
      const float2 fa[4] = {bf16x2_to_float2(ka.x), bf16x2_to_float2(ka.y),
                            bf16x2_to_float2(ka.z), bf16x2_to_float2(ka.w)};
      const float2 fb[4] = {bf16x2_to_float2(kb.x), bf16x2_to_float2(kb.y),
                            bf16x2_to_float2(kb.z), bf16x2_to_float2(kb.w)};
      #pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        float2 d = make_float2(0.f, 0.f);
        #pragma unroll
        for (int c = 0; c < 4; ++c) d = ffma2(qa[g][c], fa[c], d);
        #pragma unroll
        for (int c = 0; c < 4; ++c) d = ffma2(qb[g][c], fb[c], d);
        s[g][j] = d.x + d.y;
      }
    }
    // ---- reduce-scatter over the 4 lanes of a token pair: lane keeps head gh
    float sc[2];
    {
      const bool hi1 = qd & 1;
      const bool hi2 = qd & 2;
      #pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float send0 = hi1 ? s[0][j] : s[2][j];
        const float send1 = hi1 ? s[1][j] : s[3][j];
        float keep0 = hi1 ? s[2][j] : s[0][j];
        float keep1 = hi1 ? s[3][j] : s[1][j];
        keep0 += __shfl_xor_sync(0xffffffffu, send0, 1);
        keep1 += __shfl_xor_sync(0xffffffffu, send1, 1);
        const float send = hi2 ? keep0 : keep1;
        float kept = hi2 ? keep1 : keep0;
        kept += __shfl_xor_sync(0xffffffffu, send, 2);
        sc[j] = kept;
      }
    }
    // mask tokens past the sequence end (select, so stale or NaN data never leaks)
    sc[0] = tp < live ? sc[0] : -INFINITY;
    sc[1] = tp + 8 < live ? sc[1] : -INFINITY;

    // ---- online softmax, base 2, per head over the page's 16 tokens
    float pm = fmaxf(sc[0], sc[1]);
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
    const float m_new = fmaxf(m_run, pm);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);
    const float p0 = exp2f(sc[0] - m_use);
    const float p1 = exp2f(sc[1] - m_use);
    l_run = l_run * alpha + p0 + p1;
    m_run = m_new;
    ws.p[tp][gh] = make_float2(p0, p0);
    ws.p[tp + 8][gh] = make_float2(p1, p1);
    if (tp == 0) ws.alpha[gh] = make_float2(alpha, alpha);
    __syncwarp();

    // ---- PV: rescale, then accumulate this lane's tokens
    {
      const float4 a01 = *reinterpret_cast<const float4*>(&ws.alpha[0]);
      const float4 a23 = *reinterpret_cast<const float4*>(&ws.alpha[2]);
      const float2 al[kGroup] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w),
                                 make_float2(a23.x, a23.y), make_float2(a23.z, a23.w)};
      #pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        acc[g][0] = fmul2(acc[g][0], al[g]);
        acc[g][1] = fmul2(acc[g][1], al[g]);
      }
    }
    auto pv_token = [&](int r) {
      const uint2 vv = *reinterpret_cast<const uint2*>(vt + r * kRowBytes + dq * 8);
      const float2 v01 = bf16x2_to_float2(vv.x);
      const float2 v23 = bf16x2_to_float2(vv.y);
      const float4 pa = *reinterpret_cast<const float4*>(&ws.p[r][0]);
      const float4 pb = *reinterpret_cast<const float4*>(&ws.p[r][2]);
      const float2 pg[kGroup] = {make_float2(pa.x, pa.y), make_float2(pa.z, pa.w),
                                 make_float2(pb.x, pb.y), make_float2(pb.z, pb.w)};
      #pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        acc[g][0] = ffma2(pg[g], v01, acc[g][0]);
        acc[g][1] = ffma2(pg[g], v23, acc[g][1]);
      }
    };
    if (live == kPage) {
      #pragma unroll
      for (int r2 = 0; r2 < kPage / 2; ++r2) pv_token(2 * r2 + tpar);
    } else {
      #pragma unroll
      for (int r2 = 0; r2 < kPage / 2; ++r2) {
        if (2 * r2 + tpar < live) pv_token(2 * r2 + tpar);
      }
    }
    __syncwarp();
    if (i + kStages < mine) {
      issue(i + kStages);
      issued = i + kStages + 1;
    }
  }
  if (timed_out) {
    // let this warp's copies still in flight land before the block exits
    // (each wait bounded again)
    for (int j = consumed; j < issued; ++j) mbar_wait(&ws.bar[j % kStages], (j / kStages) & 1);
  }

  // ---- warp state -> shared memory
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 4);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 8);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
  #pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    #pragma unroll
    for (int h = 0; h < 2; ++h) {
      acc[g][h].x += __shfl_xor_sync(0xffffffffu, acc[g][h].x, 16);
      acc[g][h].y += __shfl_xor_sync(0xffffffffu, acc[g][h].y, 16);
    }
  }
  if (timed_out) {
    if (lane == 0) set_error(prm.err, kErrTimeout);
    m_run = -INFINITY;
    l_run = 0.f;
  }
  if (tp == 0) {
    sm.m[warp][gh] = m_run;
    sm.l[warp][gh] = l_run;
  }
  if (tpar == 0) {
    #pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      *reinterpret_cast<float4*>(&sm.acc[warp][g][4 * dq]) =
          make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
    }
  }
  __syncthreads();

  // ---- merge the 4 warps: thread -> (head g, dims d0, d0 + 1)
  const int g = threadIdx.x >> 5;
  const int d0 = 2 * (threadIdx.x & 31);
  float M = -INFINITY;
  #pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][g]);
  float L = 0.f;
  float2 O = make_float2(0.f, 0.f);
  #pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float mw = sm.m[w][g];
    if (mw == -INFINITY) continue;
    const float f = exp2f(mw - M);
    L += f * sm.l[w][g];
    O.x += f * sm.acc[w][g][d0];
    O.y += f * sm.acc[w][g][d0 + 1];
  }
  const int head = kvh * kGroup + g;
  const size_t out_row = (static_cast<size_t>(b) * kHq + head) * kDim;
  if (n_splits == 1) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<float2*>(prm.out + out_row + d0) = make_float2(O.x * inv, O.y * inv);
    return;
  }

  // ---- split partial, ticket, and the last block's log-sum-exp merge
  const size_t prow = (static_cast<size_t>(b) * kHq + head) * prm.max_splits;
  *reinterpret_cast<float2*>(prm.part_o + (prow + split) * kDim + d0) = O;
  if (d0 == 0) prm.part_ml[prow + split] = make_float2(M, L);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* ticket = prm.tickets + static_cast<size_t>(b) * kHkv + kvh;
    const int arrived = atomicAdd(ticket, 1);
    const int last = arrived == n_splits - 1;
    if (last) *ticket = 0;   // every split has arrived: reset for the next launch
    sm.last = last;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  float MM = -INFINITY;
  for (int s = 0; s < n_splits; ++s) MM = fmaxf(MM, __ldcg(&prm.part_ml[prow + s]).x);
  float LL = 0.f;
  float2 OO = make_float2(0.f, 0.f);
  for (int s = 0; s < n_splits; ++s) {
    const float2 ml = __ldcg(&prm.part_ml[prow + s]);
    if (ml.x == -INFINITY) continue;
    const float f = exp2f(ml.x - MM);
    const float2 o = __ldcg(reinterpret_cast<const float2*>(prm.part_o + (prow + s) * kDim + d0));
    LL += f * ml.y;
    OO.x += f * o.x;
    OO.y += f * o.y;
  }
  const float inv = LL > 0.f ? 1.f / LL : 0.f;
  *reinterpret_cast<float2*>(prm.out + out_row + d0) = make_float2(OO.x * inv, OO.y * inv);
}

}  // namespace

// ================================================================= host side

struct pkv_pool {
  pkv_pool_config cfg;
  int device;
  int num_sms;
  float* part_o;     // [2][max_batch][32][max_splits][64]
  float2* part_ml;   // [2][max_batch][32][max_splits]
  int* tickets;      // [2][max_batch][8]
  int* err;          // sticky error bits
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t smem_bytes() { return sizeof(BlockSmem); }

pkv_status check_launch() {
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Pages per split when the caller leaves the choice to the library: enough
// blocks to keep every SM busy when all sequences are at full length,
// capped so that one block's range stays short.
int auto_chunk_pages(const pkv_pool* pool, int batch) {
  const int max_pages = pool->cfg.max_seq_len / kPage;
  const long long tiles = static_cast<long long>(batch) * kHkv * max_pages;
  const long long target_blocks = 4LL * pool->num_sms;
  long long chunk = (tiles + target_blocks - 1) / target_blocks;
  const int min_chunk = (max_pages + pool->cfg.max_splits - 1) / pool->cfg.max_splits;
  if (chunk < 2) chunk = 2;
  if (chunk > 16) chunk = 16;
  if (chunk < min_chunk) chunk = min_chunk;
  return static_cast<int>(chunk);
}

template <bool kFused>
pkv_status launch_decode(pkv_pool_t pool, int layer, const void* q, const void* k,
                         const void* v, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* seq_lens, float* out,
                         int batch, int num_splits, void* stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  if (layer < 0 || layer >= c.num_layers || batch < 0 || batch > c.max_batch)
    return PKV_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > c.max_splits) return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARG;
  if (kFused && (!k || !v)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(block_tables) ||
      !aligned16(seq_lens) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  if (kFused && (!aligned16(k) || !aligned16(v))) return PKV_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_ERR_INVALID_ARG;

  const int max_pages = c.max_seq_len / kPage;
  const int parity = layer & 1;
  DecodeParams prm;
  prm.q = static_cast<const uint16_t*>(q);
  prm.k_new = static_cast<const uint16_t*>(k);
  prm.v_new = static_cast<const uint16_t*>(v);
  prm.k_pool = const_cast<uint16_t*>(static_cast<const uint16_t*>(k_pool));
  prm.v_pool = const_cast<uint16_t*>(static_cast<const uint16_t*>(v_pool));
  prm.table = block_tables + static_cast<size_t>(layer) * c.max_batch * max_pages;
  prm.seq_lens = seq_lens;
  prm.out = out;
  prm.part_o = pool->part_o + static_cast<size_t>(parity) * c.max_batch * kHq * c.max_splits * kDim;
  prm.part_ml = pool->part_ml + static_cast<size_t>(parity) * c.max_batch * kHq * c.max_splits;
  prm.tickets = pool->tickets + static_cast<size_t>(parity) * c.max_batch * kHkv;
  prm.err = pool->err;
  prm.num_pages = c.num_pages;
  prm.table_stride = max_pages;
  prm.max_seq_len = c.max_seq_len;
  prm.max_splits = c.max_splits;
  prm.num_splits = num_splits;
  prm.chunk_pages = num_splits > 0 ? 0 : auto_chunk_pages(pool, batch);
  const int grid_splits = num_splits > 0 ? num_splits
                                         : (max_pages + prm.chunk_pages - 1) / prm.chunk_pages;
  dim3 grid(grid_splits, kHkv, batch);
  decode_kernel<kFused><<<grid, kThreads, smem_bytes(), static_cast<cudaStream_t>(stream)>>>(prm);
  return check_launch();
}

}  // namespace

extern "C" {

const char* pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_OUT_OF_RANGE: return "index out of range in device data";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_UNSUPPORTED: return "unsupported geometry";
    case PKV_ERR_DEVICE_TIMEOUT: return "bounded device wait timed out";
  }
  return "unknown status";
}

pkv_status pkv_pool_create(const pkv_pool_config* config, pkv_pool_t* out) {
  if (!config || !out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  pkv_pool_config c = *config;
  if (c.page_size != kPage || c.num_q_heads != kHq || c.num_kv_heads != kHkv ||
      c.head_dim != kDim)
    return PKV_ERR_UNSUPPORTED;
  if (c.num_layers < 1 || c.num_pages < 1 || c.max_batch < 1 || c.max_seq_len < kPage ||
      c.max_seq_len > kMaxSeqLen || c.max_seq_len % kPage != 0 || c.max_splits < 0 ||
      c.max_splits > kMaxSplitsLimit || c.max_batch > 65535)
    return PKV_ERR_INVALID_ARG;
  if (c.max_splits == 0) c.max_splits = kDefaultMaxSplits;

  pkv_pool* pool = new pkv_pool();
  pool->cfg = c;
  if (cudaGetDevice(&pool->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&pool->num_sms, cudaDevAttrMultiProcessorCount, pool->device) !=
          cudaSuccess) {
    delete pool;
    return PKV_ERR_CUDA;
  }
  const size_t rows = static_cast<size_t>(2) * c.max_batch * kHq * c.max_splits;
  bool ok = cudaMalloc(&pool->part_o, rows * kDim * sizeof(float)) == cudaSuccess;
  ok = ok && cudaMalloc(&pool->part_ml, rows * sizeof(float2)) == cudaSuccess;
  ok = ok && cudaMalloc(&pool->tickets, 2 * static_cast<size_t>(c.max_batch) * kHkv * sizeof(int)) ==
                 cudaSuccess;
  ok = ok && cudaMalloc(&pool->err, sizeof(int)) == cudaSuccess;
  ok = ok && cudaMemset(pool->tickets, 0, 2 * static_cast<size_t>(c.max_batch) * kHkv * sizeof(int)) ==
                 cudaSuccess;
  ok = ok && cudaMemset(pool->err, 0, sizeof(int)) == cudaSuccess;
  ok = ok && cudaFuncSetAttribute(decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem_bytes())) == cudaSuccess;
  ok = ok && cudaFuncSetAttribute(decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem_bytes())) == cudaSuccess;
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    pkv_pool_destroy(pool);
    return PKV_ERR_CUDA;
  }
  *out = pool;
  return PKV_OK;
}

pkv_status pkv_pool_destroy(pkv_pool_t pool) {
  if (!pool) return PKV_OK;
  pkv_status st = cudaDeviceSynchronize() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  cudaFree(pool->part_o);
  cudaFree(pool->part_ml);
  cudaFree(pool->tickets);
  cudaFree(pool->err);
  delete pool;
  return st;
}

pkv_status pkv_append(pkv_pool_t pool, int layer, const void* k, const void* v, void* k_pool,
                      void* v_pool, const int32_t* block_tables, const int32_t* positions,
                      int batch, void* stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  if (layer < 0 || layer >= c.num_layers || batch < 0 || batch > c.max_batch)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!k || !v || !k_pool || !v_pool || !block_tables || !positions) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(block_tables) || !aligned16(positions))
    return PKV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_ERR_INVALID_ARG;
  const int max_pages = c.max_seq_len / kPage;
  append_kernel<<<batch, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
      static_cast<uint16_t*>(k_pool), static_cast<uint16_t*>(v_pool),
      block_tables + static_cast<size_t>(layer) * c.max_batch * max_pages, positions, max_pages,
      c.num_pages, c.max_seq_len, pool->err);
  return check_launch();
}

pkv_status pkv_decode_attention(pkv_pool_t pool, int layer, const void* q, const void* k_pool,
                                const void* v_pool, const int32_t* block_tables,
                                const int32_t* seq_lens, float* out, int batch, int num_splits,
                                void* stream) {
  return launch_decode<false>(pool, layer, q, nullptr, nullptr, k_pool, v_pool, block_tables,
                              seq_lens, out, batch, num_splits, stream);
}

pkv_status pkv_append_attend(pkv_pool_t pool, int layer, const void* q, const void* k,
                             const void* v, void* k_pool, void* v_pool,
                             const int32_t* block_tables, const int32_t* seq_lens, float* out,
                             int batch, int num_splits, void* stream) {
  return launch_decode<true>(pool, layer, q, k, v, k_pool, v_pool, block_tables, seq_lens, out,
                             batch, num_splits, stream);
}

pkv_status pkv_get_error(pkv_pool_t pool, void* stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int bits = 0;
  if (cudaMemcpyAsync(&bits, pool->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (bits == 0) return PKV_OK;
  if (cudaMemsetAsync(pool->err, 0, sizeof(int), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return PKV_ERR_CUDA;
  return (bits & kErrTimeout) ? PKV_ERR_DEVICE_TIMEOUT : PKV_ERR_OUT_OF_RANGE;
}

}  // extern "C"
