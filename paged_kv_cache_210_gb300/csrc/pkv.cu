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

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "device_common.cuh"
#include "pool_internal.h"

using namespace pkv_dev;

namespace {

constexpr int kTileBytes = kPage * kRowBytes;   // one (page, kv head) tile: 2 KiB

// Block shapes, all 4 warps with a ring of page stages per warp:
//  * ticket merge (large batches): 3 stages, 4 blocks per SM (128 registers);
//  * narrow cluster (batches up to about 4): 3 stages, 3 blocks per SM, so up
//    to 168 registers; about 256 blocks a launch leave room for the next
//    launch's blocks to become resident and prefetch while this one finishes;
//  * wide cluster (batches of about 5 to 32): 2 stages, 4 blocks per SM
//    (128 registers), so twice the splits fit one wave.
// (8-warp cluster blocks, 2 per SM, measured slower for 2 sequences because
// the next layer could not start early.)
constexpr int kTicketWarps = 4;
constexpr int kTicketStages = 3;
constexpr int kClusterWarps = 4;
constexpr int kNarrowStages = 3;
constexpr int kWideStages = 2;
constexpr int kMergeThreads = 128;               // one thread per (head, dim pair)
constexpr int kDefaultMaxSplits = 64;
constexpr int kMaxSplitsLimit = 128;
constexpr int kMaxClusterSize = 16;                // non-portable cluster size limit

// device error flag bits
constexpr int kErrPage = PKV_DEV_ERR_PAGE;
constexpr int kErrPosition = PKV_DEV_ERR_POSITION;
constexpr int kErrSeqLen = PKV_DEV_ERR_SEQ_LEN;
constexpr int kErrTimeout = PKV_DEV_ERR_TIMEOUT;


template <int kStages>
struct alignas(16) WarpSmem {
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  float2 p[kPage][kGroup];   // (p, p) per token and head
  float2 alpha[kGroup];      // (alpha, alpha) per head
  unsigned long long bar[kStages];
};

// A head leader's inbox (placed after BlockSmem, cluster kernels only): every
// block of the cluster stores its (m, l, o) for the heads this block leads.
// Slot of block r for head g: (g / S) * S + r (at most 16 slots for S <= 16).
constexpr int kInboxSlots = kMaxClusterSize;
struct ClusterInbox {
  float o[kInboxSlots][kDim];
  float m[kInboxSlots];
  float l[kInboxSlots];
};

template <int kWarps, int kStages>
struct alignas(16) BlockSmem {
  WarpSmem<kStages> warp[kWarps];
  float m[kWarps][kGroup];
  float l[kWarps][kGroup];
  union {
    float acc[kWarps][kGroup][kDim];   // the warps' partial outputs (block merge)
    struct {                           // longest-first order (prologue only)
      int hist[kMaxPages + 1];
      int wsum[kWarps];
      int pick[3];
    } order;
  };
  int pages[kMaxPages];      // this sequence's block-table row
  int last;
};

using TicketSmem = BlockSmem<kTicketWarps, kTicketStages>;
using NarrowSmem = BlockSmem<kClusterWarps, kNarrowStages>;
using WideSmem = BlockSmem<kClusterWarps, kWideStages>;
static_assert(sizeof(WarpSmem<kTicketStages>) % 16 == 0 &&
                  sizeof(WarpSmem<kWideStages>) % 16 == 0,
              "warp slabs keep 16-byte alignment");
static_assert(sizeof(NarrowSmem) % 16 == 0 && sizeof(WideSmem) % 16 == 0,
              "the cluster inbox follows BlockSmem 16-byte aligned");
static_assert(sizeof(ClusterInbox) % 16 == 0, "inbox size keeps 16-byte alignment");
// residency the kernels are shaped for: 228 KiB of shared memory per SM, 1 KiB
// of it reserved per block; 4 ticket blocks or 3 cluster blocks per SM
constexpr size_t kSmemPerSm = 228 * 1024;
static_assert(4 * (sizeof(TicketSmem) + 1024) <= kSmemPerSm, "4 ticket blocks per SM");
static_assert(3 * (sizeof(NarrowSmem) + sizeof(ClusterInbox) + 1024) <= kSmemPerSm,
              "3 narrow cluster blocks per SM");
static_assert(4 * (sizeof(WideSmem) + sizeof(ClusterInbox) + 1024) <= kSmemPerSm,
              "4 wide cluster blocks per SM");

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
  int early_trigger;          // let the next launch start right after the prefetch (one wave)
  int longest_first;          // blockIdx.z is a rank by length, not a sequence index
  const float* rope_cos;      // rotary angles [max_seq_len][32] FP32, or null: no rotation
  const float* rope_sin;
};

// ---------------------------------------------------------------- PTX helpers
// Thread-block cluster barrier, split: arrive (release) and wait (acquire).
// A wait completes once every non-exited thread of the cluster has arrived.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store to the same shared-memory offset in cluster block `rank`.
__device__ __forceinline__ void st_cluster(float* p, uint32_t rank, float v) {
  uint32_t addr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster2(float* p, uint32_t rank, float2 v) {
  uint32_t addr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
               : "memory");
}

// Pull a 128-byte line into L2 (no register result; L2 is coherent, so this
// cannot return stale data to a later load).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// own prologue, and wait until the previous kernel's results are visible.
// Both are no-ops when the launch did not opt in.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// cos (or sin) of the 8 rotary angles 8 c4 .. 8 c4 + 7 of one position row.
__device__ __forceinline__ void load_angles(const float* row, int c4, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(row + 8 * c4));
  const float4 b = __ldg(reinterpret_cast<const float4*>(row + 8 * c4 + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Rotary embedding of one 16-byte chunk (8 dims) of the appended key. Dim i of
// the low half pairs with dim i + 32 (rotate-half): low' = low cos - high sin,
// high' = high cos + low sin. `own` is chunk c (dims 8c .. 8c+7), `partner` the
// chunk 4 away, `high` says own is in the upper half; cs/sn hold the angles of
// pairs 8 (c mod 4) .. +7. Products and sum are each rounded in FP32 (no fused
// multiply-add), then to BF16, so the stored key has one defined value.
__device__ __forceinline__ uint4 rope_key_chunk(uint4 own, uint4 partner, bool high,
                                               const float (&cs)[8], const float (&sn)[8]) {
  const uint32_t a[4] = {own.x, own.y, own.z, own.w};
  const uint32_t b[4] = {partner.x, partner.y, partner.z, partner.w};
  uint32_t o[4];
  #pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 fa = bf16x2_to_float2(a[j]);
    const float2 fb = bf16x2_to_float2(b[j]);
    const float ac0 = __fmul_rn(fa.x, cs[2 * j]), bs0 = __fmul_rn(fb.x, sn[2 * j]);
    const float ac1 = __fmul_rn(fa.y, cs[2 * j + 1]), bs1 = __fmul_rn(fb.y, sn[2 * j + 1]);
    const float e0 = high ? __fadd_rn(ac0, bs0) : __fsub_rn(ac0, bs0);
    const float e1 = high ? __fadd_rn(ac1, bs1) : __fsub_rn(ac1, bs1);
    o[j] = float2_to_bf16x2(e0, e1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 shfl_xor_uint4(uint4 v, int m) {
  return make_uint4(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m),
                    __shfl_xor_sync(0xffffffffu, v.z, m), __shfl_xor_sync(0xffffffffu, v.w, m));
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  return __ffma2_rn(a, b, c);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// ---------------------------------------------------------------- append
// One block of 128 threads per sequence: thread t copies 16-byte chunk
// (t % 64) % 8 of kv head (t % 64) / 8, of K for t < 64 and of V otherwise.
// With rotary tables the key is rotated to its position on the way (the
// partner chunk sits in lane t ^ 4 of the same warp).
__global__ void __launch_bounds__(128) append_kernel(const uint16_t* __restrict__ k,
                                                     const uint16_t* __restrict__ v,
                                                     uint16_t* __restrict__ k_pool,
                                                     uint16_t* __restrict__ v_pool,
                                                     const int32_t* __restrict__ table,
                                                     const int32_t* __restrict__ positions,
                                                     int table_stride, int num_pages,
                                                     int max_seq_len, int* err,
                                                     const float* __restrict__ rope_cos,
                                                     const float* __restrict__ rope_sin) {
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
  uint4 val = __ldg(reinterpret_cast<const uint4*>(src));
  if (rope_cos) {   // the same for every thread of the block
    const uint4 partner = shfl_xor_uint4(val, 4);
    if (t < 64) {
      float cs[8], sn[8];
      load_angles(rope_cos + static_cast<size_t>(pos) * (kDim / 2), chunk & 3, cs);
      load_angles(rope_sin + static_cast<size_t>(pos) * (kDim / 2), chunk & 3, sn);
      val = rope_key_chunk(val, partner, chunk >= 4, cs, sn);
    }
  }
  *reinterpret_cast<uint4*>(dst) = val;
}

// ---------------------------------------------------------------- page computation
// Lane roles, fixed per lane. QK: a lane owns tokens tp and tp + 8 and the
// 16-byte dim chunks qd and qd + 4 (read in a row-parity-dependent order so
// the shared loads are bank-conflict-free); after the reduce-scatter it owns
// head gh. PV: a lane owns dims 4 dq .. 4 dq + 3 of the tokens 2 i + tpar.
struct LaneRoles {
  int tp, qd, cA, cB, gh, dq, tpar;
  __device__ explicit LaneRoles(int lane) {
    tp = lane >> 2;
    qd = lane & 3;
    const int par = tp & 1;
    cA = qd + 4 * par;
    cB = qd + 4 * (1 - par);
    gh = 2 * (qd & 1) + ((qd >> 1) & 1);
    dq = lane & 15;
    tpar = lane >> 4;
  }
};

// Online-softmax state of one warp for the 4 heads of a kv head.
struct WarpState {
  float m_run;              // running max (base 2) of head gh
  float l_run;              // this lane's share of the running sum of head gh
  float2 acc[kGroup][2];    // PV accumulators: dims (4dq, 4dq+1), (4dq+2, 4dq+3)
  __device__ void reset() {
    m_run = -INFINITY;
    l_run = 0.f;
    #pragma unroll
    for (int g = 0; g < kGroup; ++g) acc[g][0] = acc[g][1] = make_float2(0.f, 0.f);
  }
};

// q of the 4 heads at qrow ([4][64] BF16) for this lane's chunks, scaled by
// log2(e) / sqrt(64) so that scores come out in base 2. kRope: q is first
// rotated in FP32 by the angles cs, sn of pairs 8 qd .. 8 qd + 7 at the
// query's position; the lane's chunks qd and qd + 4 are exactly the two
// halves of those pairs. With the scale folded into the angles and the sign
// of the rotation folded into sin (chunk A is the low half when cA < 4):
//   A' = A c' + B s_A,  B' = B c' - A s_A,  c' = c scale, s_A = -/+ s scale.
template <bool kRope>
__device__ __forceinline__ void load_q(const uint16_t* qrow, const LaneRoles& r,
                                       float2 (&qa)[kGroup][4], float2 (&qb)[kGroup][4],
                                       const float (&cs)[8], const float (&sn)[8]) {
  const float qscale = 1.4426950408889634f * 0.125f;
  float2 cq[4], sa[4], sb[4];
  if (kRope) {
    const float sgn = r.cA < 4 ? -qscale : qscale;
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      cq[j] = make_float2(cs[2 * j] * qscale, cs[2 * j + 1] * qscale);
      sa[j] = make_float2(sn[2 * j] * sgn, sn[2 * j + 1] * sgn);
      sb[j] = make_float2(-sa[j].x, -sa[j].y);
    }
  }
  #pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    const uint4* pa = reinterpret_cast<const uint4*>(qrow + g * kDim + r.cA * 8);
    const uint4* pb = reinterpret_cast<const uint4*>(qrow + g * kDim + r.cB * 8);
    const uint4 ra = __ldg(pa);
    const uint4 rb = __ldg(pb);
    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
    const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 fa = bf16x2_to_float2(wa[j]);
      const float2 fb = bf16x2_to_float2(wb[j]);
      if (kRope) {
        qa[g][j] = ffma2(fb, sa[j], fmul2(fa, cq[j]));
        qb[g][j] = ffma2(fa, sb[j], fmul2(fb, cq[j]));
      } else {
        qa[g][j] = make_float2(fa.x * qscale, fa.y * qscale);
        qb[g][j] = make_float2(fb.x * qscale, fb.y * qscale);
      }
    }
  }
}

// Scores of one page for this lane: tokens tp and tp + 8 of K tile kt, all 4
// heads over the lane's 16 dims, then a reduce-scatter over the 4 lanes of a
// token pair so that the lane keeps head gh's full scores (base 2, scaled).
// Tokens at or past `live` get -inf.
__device__ __forceinline__ void page_scores(const uint8_t* kt, int live,
                                            const float2 (&qa)[kGroup][4],
                                            const float2 (&qb)[kGroup][4], const LaneRoles& r,
                                            float (&sc)[2]) {
  float s[kGroup][2];
  #pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint8_t* krow = kt + (r.tp + 8 * j) * kRowBytes;
    const uint4 ka = *reinterpret_cast<const uint4*>(krow + r.cA * 16);
    const uint4 kb = *reinterpret_cast<const uint4*>(krow + r.cB * 16);
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
  const bool hi1 = r.qd & 1;
  const bool hi2 = r.qd & 2;
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
  sc[0] = r.tp < live ? sc[0] : -INFINITY;
  sc[1] = r.tp + 8 < live ? sc[1] : -INFINITY;
}

// Rescale of the accumulators by the per-head factors in alpha_s.
__device__ __forceinline__ void rescale_acc(const float2* alpha_s, WarpState& st) {
  const float4 a01 = *reinterpret_cast<const float4*>(&alpha_s[0]);
  const float4 a23 = *reinterpret_cast<const float4*>(&alpha_s[2]);
  const float2 al[kGroup] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w),
                             make_float2(a23.x, a23.y), make_float2(a23.z, a23.w)};
  #pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    st.acc[g][0] = fmul2(st.acc[g][0], al[g]);
    st.acc[g][1] = fmul2(st.acc[g][1], al[g]);
  }
}

// P V of one page: this lane's 4 dims over its tokens 2 i + tpar of V tile vt
// (the first `live`), with the probabilities of the 4 heads from p ([16][4],
// each duplicated as a pair).
__device__ __forceinline__ void page_pv(const uint8_t* vt, int live, const float2 (*p)[kGroup],
                                        const LaneRoles& r, WarpState& st) {
  auto pv_token = [&](int t) {
    const uint2 vv = *reinterpret_cast<const uint2*>(vt + t * kRowBytes + r.dq * 8);
    const float2 v01 = bf16x2_to_float2(vv.x);
    const float2 v23 = bf16x2_to_float2(vv.y);
    const float4 pa = *reinterpret_cast<const float4*>(&p[t][0]);
    const float4 pb = *reinterpret_cast<const float4*>(&p[t][2]);
    const float2 pg[kGroup] = {make_float2(pa.x, pa.y), make_float2(pa.z, pa.w),
                               make_float2(pb.x, pb.y), make_float2(pb.z, pb.w)};
    #pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      st.acc[g][0] = ffma2(pg[g], v01, st.acc[g][0]);
      st.acc[g][1] = ffma2(pg[g], v23, st.acc[g][1]);
    }
  };
  if (live == kPage) {
    #pragma unroll
    for (int t2 = 0; t2 < kPage / 2; ++t2) pv_token(2 * t2 + r.tpar);
  } else {
    #pragma unroll
    for (int t2 = 0; t2 < kPage / 2; ++t2) {
      if (2 * t2 + r.tpar < live) pv_token(2 * t2 + r.tpar);
    }
  }
}

// One page: K tile kt and V tile vt in shared memory, `live` valid tokens
// (the rest are masked by select, so stale data never leaks). p and alpha
// are the warp's shared slots for the probabilities and the rescale factors.
__device__ __forceinline__ void attend_page(const uint8_t* kt, const uint8_t* vt, int live,
                                            const float2 (&qa)[kGroup][4],
                                            const float2 (&qb)[kGroup][4],
                                            float2 (*p)[kGroup], float2* alpha_s,
                                            const LaneRoles& r, WarpState& st) {
  float sc[2];
  page_scores(kt, live, qa, qb, r, sc);

  // online softmax, base 2, per head over the page's 16 tokens
  float pm = fmaxf(sc[0], sc[1]);
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
  const float m_new = fmaxf(st.m_run, pm);
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float alpha = fast_exp2(st.m_run - m_use);
  const float p0 = fast_exp2(sc[0] - m_use);
  const float p1 = fast_exp2(sc[1] - m_use);
  st.l_run = st.l_run * alpha + p0 + p1;
  st.m_run = m_new;
  p[r.tp][r.gh] = make_float2(p0, p0);
  p[r.tp + 8][r.gh] = make_float2(p1, p1);
  if (r.tp == 0) alpha_s[r.gh] = make_float2(alpha, alpha);
  __syncwarp();

  // PV: rescale, then accumulate this lane's tokens
  rescale_acc(alpha_s, st);
  page_pv(vt, live, p, r, st);
  __syncwarp();
}

// End of a warp's pages: the running sum over the 8 token-pair lanes of each
// head, the accumulators over the two token-parity halves.
__device__ __forceinline__ void reduce_warp_state(WarpState& st) {
  st.l_run += __shfl_xor_sync(0xffffffffu, st.l_run, 4);
  st.l_run += __shfl_xor_sync(0xffffffffu, st.l_run, 8);
  st.l_run += __shfl_xor_sync(0xffffffffu, st.l_run, 16);
  #pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    #pragma unroll
    for (int h = 0; h < 2; ++h) {
      st.acc[g][h].x += __shfl_xor_sync(0xffffffffu, st.acc[g][h].x, 16);
      st.acc[g][h].y += __shfl_xor_sync(0xffffffffu, st.acc[g][h].y, 16);
    }
  }
}

// ---------------------------------------------------------------- merges
// The block's warps merged in shared memory: thread t < 128 gets the
// log-sum-exp state of head g = (t / 32) % 4 for dims d0 = 2 (t % 32), d0 + 1
// (M: max, L: sum, O: unnormalised output); the rest of an 8-warp block
// computes an alias.
template <int kWarps, int kStages>
__device__ __forceinline__ void block_merge(BlockSmem<kWarps, kStages>& sm, const WarpState& st,
                                            const LaneRoles& rl, int warp, float& M, float& L,
                                            float2& O) {
  if (rl.tp == 0) {
    sm.m[warp][rl.gh] = st.m_run;
    sm.l[warp][rl.gh] = st.l_run;
  }
  if (rl.tpar == 0) {
    #pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      *reinterpret_cast<float4*>(&sm.acc[warp][g][4 * rl.dq]) =
          make_float4(st.acc[g][0].x, st.acc[g][0].y, st.acc[g][1].x, st.acc[g][1].y);
    }
  }
  __syncthreads();
  const int g = (threadIdx.x >> 5) & (kGroup - 1);
  const int d0 = 2 * (threadIdx.x & 31);
  M = -INFINITY;
  #pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][g]);
  L = 0.f;
  O = make_float2(0.f, 0.f);
  #pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float mw = sm.m[w][g];
    if (mw == -INFINITY) continue;
    const float f = fast_exp2(mw - M);
    L += f * sm.l[w][g];
    O.x += f * sm.acc[w][g][d0];
    O.y += f * sm.acc[w][g][d0 + 1];
  }
}

// Cluster merge of the S blocks of one (sequence, kv head) (S = the cluster
// size): each block first merges its warps (block_merge), then sends one
// (m, l, o) part per head straight into the inbox of the head's leader,
// block g mod S of the cluster; every thread arrives on the cluster barrier,
// and in each leader warp w combines the S parts of head rank + w S into
// out_kv ([4][64], the kv head's query heads). A block that leads no head
// returns after its arrival, or, with `wait_always` (blocks that go on to use
// the cluster barrier again), after the wait as well.
template <int kWarps, int kStages>
__device__ __forceinline__ void cluster_merge(BlockSmem<kWarps, kStages>& sm,
                                              ClusterInbox& inbox, const WarpState& st,
                                              const LaneRoles& rl, int warp, int lane,
                                              float* out_kv, bool wait_always) {
  static_assert(kWarps == kGroup, "one merging thread per (head, dim pair)");
  float M, L;
  float2 O;
  block_merge(sm, st, rl, warp, M, L, O);
  const int S = gridDim.x;
  const int rank = static_cast<int>(cluster_rank());
  const int g = warp;               // thread t: head t / 32, dims 2 (t % 32), + 1
  const int d0 = 2 * lane;
  const int at = (g / S) * S + rank;
  st_cluster2(&inbox.o[at][d0], g % S, O);
  if (lane == 0) {
    st_cluster(&inbox.m[at], g % S, M);
    st_cluster(&inbox.l[at], g % S, L);
  }
  cluster_arrive_release();
  if (rank >= kGroup) {   // leads no head
    if (wait_always) cluster_wait_acquire();
    return;
  }
  cluster_wait_acquire();
  const int hg = rank + warp * S;   // head of this leader warp
  if (hg < kGroup) {
    const int base = warp * S;      // its parts: slots base .. base + S - 1, part p from rank p
    const float mp = lane < S ? inbox.m[base + lane] : -INFINITY;
    float mx = mp;
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float w = mp == -INFINITY ? 0.f : fast_exp2(mp - mx);
    float lw = lane < S ? w * inbox.l[base + lane] : 0.f;
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    float2 acc = make_float2(0.f, 0.f);
    #pragma unroll
    for (int p = 0; p < kMaxClusterSize; ++p) {
      if (p < S) {
        const float wp = __shfl_sync(0xffffffffu, w, p);
        const float2 op = *reinterpret_cast<const float2*>(&inbox.o[base + p][d0]);
        acc.x += wp * op.x;
        acc.y += wp * op.y;
      }
    }
    const float inv = lw > 0.f ? 1.f / lw : 0.f;
    *reinterpret_cast<float2*>(out_kv + hg * kDim + d0) = make_float2(acc.x * inv, acc.y * inv);
  }
}

// ---------------------------------------------------------------- dispatch order
// Blocks start in linear block order (x fastest, z slowest). With mixed
// lengths, handing out the longest sequences first shortens the launch's
// tail (the longest-processing-time-first rule), so a ticket-mode launch
// reads blockIdx.z as a rank: rank z is the z-th sequence by page count,
// most pages first, ties by index. Each block finds its own sequence with a
// counting sort of the page counts in shared memory: O(batch / threads +
// 128) work and four block barriers, reading only seq_lens (which may be
// read before the wait for the previous launch).
__device__ __forceinline__ int page_count(int len) {
  return min(max((len + kPage - 1) / kPage, 0), kMaxPages);
}

// Returns -1 without the second pass when `useful(pages)` says a block of
// that rank has no work (split slots past the sequence's last range).
template <int kWarps, int kStages, class Useful>
__device__ int longest_first_sequence(int z, int batch, const int32_t* seq_lens,
                                      BlockSmem<kWarps, kStages>& sm, Useful useful) {
  constexpr int kThreads = kWarps * 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kHeld = 4;                 // page counts kept in registers per thread
  int held[kHeld];
  #pragma unroll
  for (int e = 0; e < kHeld; ++e) {
    const int s = static_cast<int>(threadIdx.x) + e * kThreads;
    held[e] = s < batch ? page_count(seq_lens[s]) : -1;
  }
  for (int i = threadIdx.x; i <= kMaxPages; i += kThreads) sm.order.hist[i] = 0;
  __syncthreads();
  #pragma unroll
  for (int e = 0; e < kHeld; ++e)
    if (held[e] >= 0) atomicAdd(&sm.order.hist[held[e]], 1);
  for (int s = static_cast<int>(threadIdx.x) + kHeld * kThreads; s < batch; s += kThreads)
    atomicAdd(&sm.order.hist[page_count(seq_lens[s])], 1);
  __syncthreads();
  // bucket of rank z: lane l owns the buckets kMaxPages - 4l - e (e < 4),
  // most pages first; bucket 0 comes last
  if (warp == 0) {
    int cnt[4], sum = 0;
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
      cnt[e] = sm.order.hist[kMaxPages - 4 * lane - e];
      sum += cnt[e];
    }
    int incl = sum;
    #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int excl = incl - sum;
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (z >= excl && z < excl + cnt[e]) {
        sm.order.pick[0] = kMaxPages - 4 * lane - e;
        sm.order.pick[1] = z - excl;
      }
      excl += cnt[e];
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0 && z >= total) {
      sm.order.pick[0] = 0;
      sm.order.pick[1] = z - total;
    }
  }
  __syncthreads();
  const int p = sm.order.pick[0];
  const int k = sm.order.pick[1];
  if (!useful(p)) return -1;                // the same decision in every thread
  // the k-th sequence (by index) with p pages
  int seen = 0;
  auto scan = [&](int s, int pc) {          // one pass over kThreads sequences
    const bool hit = s < batch && pc == p;
    const uint32_t ballot = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) sm.order.wsum[warp] = __popc(ballot);
    __syncthreads();
    int before = seen, total = 0;
    #pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      before += w < warp ? sm.order.wsum[w] : 0;
      total += sm.order.wsum[w];
    }
    if (hit && before + __popc(ballot & ((1u << lane) - 1u)) == k) sm.order.pick[2] = s;
    seen += total;
    __syncthreads();
  };
  #pragma unroll
  for (int e = 0; e < kHeld; ++e) {
    if (e * kThreads >= batch || seen > k) break;   // the same decision in every thread
    scan(e * kThreads + static_cast<int>(threadIdx.x), held[e]);
  }
  for (int base = kHeld * kThreads; base < batch && seen <= k; base += kThreads) {
    const int s = base + static_cast<int>(threadIdx.x);
    scan(s, s < batch ? page_count(seq_lens[s]) : -1);
  }
  return sm.order.pick[2];
}

// ---------------------------------------------------------------- ticket merge
// A split's partial (M, L, O from block_merge: thread t of the 4-warp block
// owns head t / 32, dims 2 (t % 32), + 1) into the handle's partials, one
// ticket per (sequence, kv head), and the last split's log-sum-exp merge of
// all n_splits partials into out. Called by every thread of the block.
template <class Smem>
__device__ __forceinline__ void ticket_merge(Smem& sm, float* part_o, float2* part_ml,
                                             int* tickets, int max_splits, float* out, int b,
                                             int kvh, int split, int n_splits, float M, float L,
                                             float2 O, int warp, int lane) {
  const int g = (threadIdx.x >> 5) & (kGroup - 1);
  const int d0 = 2 * (threadIdx.x & 31);
  // ---- split partial, ticket, and the last block's log-sum-exp merge
  const size_t head0 = (static_cast<size_t>(b) * kHq + kvh * kGroup) * max_splits;
  const size_t prow = head0 + static_cast<size_t>(g) * max_splits;
  *reinterpret_cast<float2*>(part_o + (prow + split) * kDim + d0) = O;
  if (d0 == 0) part_ml[prow + split] = make_float2(M, L);
  __syncthreads();
  if (threadIdx.x == 0) {
    // One acquire-release atomic after the barrier: its release publishes the
    // partials every thread of this block wrote; for the last block its
    // acquire makes the other blocks' partials visible (the barrier below
    // passes that on to the block's other threads).
    int* ticket = tickets + static_cast<size_t>(b) * kHkv + kvh;
    int arrived;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(arrived)
                 : "l"(ticket)
                 : "memory");
    const int last = arrived == n_splits - 1;
    if (last) *ticket = 0;   // every split has arrived: reset for the next launch
    sm.last = last;
  }
  __syncthreads();
  if (!sm.last) return;

  // Warp hg merges head hg; lane (quad, half) owns dims 4 quad .. 4 quad + 3
  // over the splits s = half, half + 2, ...: an online log-sum-exp merge of
  // (m_s, l_s, o_s) loaded straight from L2 (bypassing L1, which may hold
  // lines of an earlier launch), then the two halves combine by shuffle.
  {
    const int hg = warp;
    const int quad = lane & 15;
    const int half = lane >> 4;
    const size_t hrow = head0 + static_cast<size_t>(hg) * max_splits;
    float mrun = -INFINITY, lrun = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = half; s0 < n_splits; s0 += 16) {
      float2 ml[8];
      float4 v[8];
      #pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int s = s0 + 2 * j;
        ml[j] = s < n_splits ? __ldcg(&part_ml[hrow + s]) : make_float2(-INFINITY, 0.f);
        v[j] = s < n_splits
                   ? __ldcg(reinterpret_cast<const float4*>(part_o + (hrow + s) * kDim + 4 * quad))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mnew = mrun;
      #pragma unroll
      for (int j = 0; j < 8; ++j) mnew = fmaxf(mnew, ml[j].x);
      if (mnew == -INFINITY) continue;
      const float a = fast_exp2(mrun - mnew);   // 0 while nothing was merged
      lrun *= a;
      o = make_float4(o.x * a, o.y * a, o.z * a, o.w * a);
      #pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = fast_exp2(ml[j].x - mnew);   // 0 for an absent split
        lrun += w * ml[j].y;
        o.x += w * v[j].x;
        o.y += w * v[j].y;
        o.z += w * v[j].z;
        o.w += w * v[j].w;
      }
      mrun = mnew;
    }
    // combine with the other half (lane ^ 16)
    const float mo = __shfl_xor_sync(0xffffffffu, mrun, 16);
    const float lo = __shfl_xor_sync(0xffffffffu, lrun, 16);
    const float4 oo = make_float4(__shfl_xor_sync(0xffffffffu, o.x, 16),
                                  __shfl_xor_sync(0xffffffffu, o.y, 16),
                                  __shfl_xor_sync(0xffffffffu, o.z, 16),
                                  __shfl_xor_sync(0xffffffffu, o.w, 16));
    const float mx = fmaxf(mrun, mo);
    const float wa = mrun == -INFINITY ? 0.f : fast_exp2(mrun - mx);
    const float wb = mo == -INFINITY ? 0.f : fast_exp2(mo - mx);
    const float LL = wa * lrun + wb * lo;
    if (half == 0) {
      const float inv = LL > 0.f ? 1.f / LL : 0.f;
      *reinterpret_cast<float4*>(out + (static_cast<size_t>(b) * kHq + kvh * kGroup + hg) *
                                               kDim + 4 * quad) =
          make_float4((wa * o.x + wb * oo.x) * inv, (wa * o.y + wb * oo.y) * inv,
                      (wa * o.z + wb * oo.z) * inv, (wa * o.w + wb * oo.w) * inv);
    }
  }
}

// ---------------------------------------------------------------- decode
// kCluster: the splits of one (sequence, kv head) form one thread-block
// cluster (gridDim.x == cluster size) and merge through distributed shared
// memory; otherwise splits merge through global partials and a ticket.
template <bool kFused, bool kCluster, int kWarps, int kStages, bool kRope>
__global__ void __launch_bounds__(kWarps * 32, kCluster && kStages == kNarrowStages ? 3 : 16 / kWarps)
decode_kernel(const DecodeParams prm) {
  constexpr int kThreads = kWarps * 32;
  using Smem = BlockSmem<kWarps, kStages>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (!kCluster && prm.longest_first) {
    // a split slot past the last range of a sequence with this many pages
    // has nothing to do (split 0 always goes on: it reports invalid lengths)
    auto useful = [&](int pages) {
      if (split == 0) return true;
      const int chunk = prm.num_splits > 0 ? (pages + prm.num_splits - 1) / prm.num_splits
                                           : prm.chunk_pages;
      return pages > 0 && split < (pages + chunk - 1) / chunk;
    };
    b = longest_first_sequence(static_cast<int>(blockIdx.z), static_cast<int>(gridDim.z),
                               prm.seq_lens, sm, useful);
    if (b < 0) return;
  }

  // Before griddepcontrol.wait (programmatic dependent launch) this block
  // reads only seq_lens, the block table and pool rows below the appended
  // position; q, the new k/v, the appended slot and out come after it.
  const int32_t* row = prm.table + static_cast<size_t>(b) * prm.table_stride;
  // the whole block-table row (at most 512 B) is read alongside seq_len, so
  // no global read waits on another
  for (int i = threadIdx.x; i < prm.table_stride; i += kThreads) sm.pages[i] = row[i];
  const int len = prm.seq_lens[b];
  if (len < 1 || len > prm.max_seq_len) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) set_error(prm.err, kErrSeqLen);
    return;
  }
  const int n_pages = (len + kPage - 1) / kPage;
  const int chunk = prm.num_splits > 0 ? (n_pages + prm.num_splits - 1) / prm.num_splits
                                       : prm.chunk_pages;
  const int n_splits = (n_pages + chunk - 1) / chunk;   // non-empty splits of this sequence
  if (kCluster) {
    if (n_splits == 1 && split > 0) return;   // the same decision in every block of the cluster
  } else {
    if (split >= n_splits) return;
  }
  const bool active = split < n_splits;       // an idle cluster block only joins the merge
  const int page_begin = active ? split * chunk : 0;
  const int page_end = active ? min(n_pages, page_begin + chunk) : 0;
  const int last_page = n_pages - 1;
  const int new_slot = (len - 1) % kPage;               // slot of the appended token

  WarpSmem<kStages>& ws = sm.warp[warp];
  // pages of this warp: page_begin + warp + 4 i
  const int mine = page_begin + warp < page_end
                       ? (page_end - (page_begin + warp) + kWarps - 1) / kWarps
                       : 0;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&ws.bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();   // the block-table row is in shared memory

  // Physical page of this warp's i-th page (i < mine <= 32) sits in lane i:
  // one parallel read of the block table instead of one per page.
  int my_phys = -1;
  if (lane < mine) my_phys = sm.pages[page_begin + warp + kWarps * lane];

  // Copy engine: rows of this warp's i-th page into stage i % kStages (lane 0
  // issues). In the fused step the appended row is not copied from the pool.
  auto issue_copy = [&](int i, int stage, int phys) {
    if (lane != 0) return;
    const int lp = page_begin + warp + kWarps * i;
    const bool ok = phys >= 0 && phys < prm.num_pages;
    int rows = lp == last_page ? len - lp * kPage : kPage;
    if (kFused && lp == last_page) rows = new_slot;     // the new row comes from k/v
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
  };
  // Rotary angles of the position len - 1 for pairs 8 (lane & 3) .. + 7: the
  // query rotation uses them, and so does the key rotation in lanes 0..7
  // (chunk c = lane, c & 3 == lane & 3). The tables are constant inputs, read
  // ahead of the wait for the previous launch.
  float rcs[8], rsn[8];
  if (kRope) {
    load_angles(prm.rope_cos + static_cast<size_t>(len - 1) * (kDim / 2), lane & 3, rcs);
    load_angles(prm.rope_sin + static_cast<size_t>(len - 1) * (kDim / 2), lane & 3, rsn);
  }

  // Fused step: the warp whose i_new-th page is the sequence's last page
  // writes the appended token's K/V row to the pool and to the stage tile.
  // Lanes 0..15 load one 16-byte chunk each (K for lanes 0..7, V for 8..15),
  // only after the wait: k/v may come from the previous kernel.
  const int new_off = last_page - page_begin - warp;
  const int i_new = kFused && new_off >= 0 && new_off % kWarps == 0 && new_off / kWarps < mine
                        ? new_off / kWarps
                        : -1;
  auto load_new_row = [&]() {
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 16) {
      const uint16_t* src = (lane >= 8 ? prm.v_new : prm.k_new) +
                            (static_cast<size_t>(b) * kHkv + kvh) * kDim + (lane & 7) * 8;
      val = __ldg(reinterpret_cast<const uint4*>(src));
    }
    return val;
  };
  // Stores the loaded chunk `val` (page i_new, in stage `stage`). With rotary
  // tables lanes 0..7 rotate the key first, the partner chunk coming from
  // lane ^ 4, with the angles above (`preloaded`) or loaded again (in the
  // page loop, where rcs/rsn are no longer kept). Called by the whole warp.
  auto place_new_row = [&](int stage, int phys, bool preloaded, uint4 val) {
    if (phys < 0 || phys >= prm.num_pages) return;
    const bool is_v = lane >= 8;
    const int c = lane & 7;
    if (kRope) {
      const uint4 partner = shfl_xor_uint4(val, 4);
      if (lane < 8) {
        float cs[8], sn[8];
        if (preloaded) {
          #pragma unroll
          for (int e = 0; e < 8; ++e) {
            cs[e] = rcs[e];
            sn[e] = rsn[e];
          }
        } else {
          load_angles(prm.rope_cos + static_cast<size_t>(len - 1) * (kDim / 2), c & 3, cs);
          load_angles(prm.rope_sin + static_cast<size_t>(len - 1) * (kDim / 2), c & 3, sn);
        }
        val = rope_key_chunk(val, partner, c >= 4, cs, sn);
      }
    }
    if (lane >= 16) return;
    uint16_t* pool = is_v ? prm.v_pool : prm.k_pool;
    *reinterpret_cast<uint4*>(pool + ((static_cast<size_t>(phys) * kHkv + kvh) * kPage +
                                      new_slot) * kDim + c * 8) = val;
    uint8_t* tile = is_v ? ws.v[stage] : ws.k[stage];
    *reinterpret_cast<uint4*>(tile + new_slot * kRowBytes + c * 16) = val;
  };

  // prefetch; the unfused kernel defers the page holding the appended slot,
  // which the preceding append kernel may still be writing
  const int n_prefetch = min(mine, kStages);
  int deferred = -1;
  for (int i = 0; i < n_prefetch; ++i) {
    const int phys = __shfl_sync(0xffffffffu, my_phys, i);
    if (!kFused && page_begin + warp + kWarps * i == last_page) {
      deferred = i;
    } else {
      issue_copy(i, i, phys);
    }
  }
  // q of the 4 heads (512 B) and, fused, the new k/v rows into L2 ahead of the wait
  if (warp == 0 && lane < 6 && active) {
    const uint16_t* line = nullptr;
    if (lane < 4) {
      line = prm.q + (static_cast<size_t>(b) * kHq + kvh * kGroup + lane) * kDim;
    } else if (kFused) {
      line = (lane == 4 ? prm.k_new : prm.v_new) + (static_cast<size_t>(b) * kHkv + kvh) * kDim;
    }
    if (line) prefetch_l2(line);
  }
  // A launch that fits in one wave of resident blocks lets the next launch
  // start now, so its blocks prefetch while this one computes; a larger
  // launch triggers after its page loop, so waiting blocks of the next
  // launch do not take slots this launch's later blocks need.
  if (prm.early_trigger) pdl_launch_dependents();
  pdl_wait();
  // the new row's load goes out before q's, so the two latencies overlap
  const bool new_in_prologue = i_new >= 0 && i_new < n_prefetch;
  uint4 new_val = make_uint4(0u, 0u, 0u, 0u);
  if (new_in_prologue) new_val = load_new_row();
  if (deferred >= 0) issue_copy(deferred, deferred, __shfl_sync(0xffffffffu, my_phys, deferred));
  int issued = n_prefetch;

  const LaneRoles rl(lane);
  float2 qa[kGroup][4], qb[kGroup][4];
  load_q<kRope>(prm.q + (static_cast<size_t>(b) * kHq + kvh * kGroup) * kDim, rl, qa, qb, rcs,
                rsn);
  if (new_in_prologue) place_new_row(i_new, __shfl_sync(0xffffffffu, my_phys, i_new), true, new_val);
  __syncwarp();   // the appended row written by lanes 0..15 is read by every lane

  WarpState st;
  st.reset();

  bool timed_out = false;
  int consumed = 0;
  // tokens of the warp's i-th page that count (0 for a page id out of range)
  auto live_of = [&](int i, int phys) {
    const int lp = page_begin + warp + kWarps * i;
    const int valid = lp == last_page ? len - lp * kPage : kPage;
    return phys >= 0 && phys < prm.num_pages ? valid : 0;
  };
  // after page i is consumed: the copy of page i + kStages into its stage
  auto refill = [&](int i, int stage) {
    if (i + kStages < mine) {
      const int next_phys = __shfl_sync(0xffffffffu, my_phys, i + kStages);
      issue_copy(i + kStages, stage, next_phys);
      if (i + kStages == i_new) place_new_row(stage, next_phys, false, load_new_row());
      __syncwarp();
      issued = i + kStages + 1;
    }
  };
  int stage = 0;            // i % kStages
  uint32_t phase = 0;       // (i / kStages) & 1
  for (int i = 0; i < mine; ++i) {
    const int phys = __shfl_sync(0xffffffffu, my_phys, i);
    // one verdict per warp: the page work below shuffles across all lanes
    if (!__all_sync(0xffffffffu, mbar_wait(&ws.bar[stage], phase))) {
      timed_out = true;
      break;
    }
    consumed = i + 1;
    attend_page(ws.k[stage], ws.v[stage], live_of(i, phys), qa, qb, ws.p, ws.alpha, rl, st);
    refill(i, stage);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  if (timed_out) {
    // let this warp's copies still in flight land before the block exits
    // (each wait bounded again)
    for (int j = consumed; j < issued; ++j) mbar_wait(&ws.bar[j % kStages], (j / kStages) & 1);
  }

  if (!prm.early_trigger) pdl_launch_dependents();

  // ---- warp state
  reduce_warp_state(st);
  if (timed_out) {
    if (lane == 0) set_error(prm.err, kErrTimeout);
    st.m_run = -INFINITY;
    st.l_run = 0.f;
  }
  if constexpr (kCluster) {
    if (n_splits > 1) {
      cluster_merge(sm, *reinterpret_cast<ClusterInbox*>(smem_raw + sizeof(Smem)), st, rl, warp,
                    lane, prm.out + (static_cast<size_t>(b) * kHq + kvh * kGroup) * kDim, false);
      return;
    }
  }

  // ---- block merge (every ticket-mode block; a cluster whose sequence has
  // a single split)
  float M, L;
  float2 O;
  block_merge(sm, st, rl, warp, M, L, O);
  const bool merger = threadIdx.x < kMergeThreads;
  const int g = (threadIdx.x >> 5) & (kGroup - 1);
  const int d0 = 2 * (threadIdx.x & 31);
  const int head = kvh * kGroup + g;
  const size_t out_row = (static_cast<size_t>(b) * kHq + head) * kDim;
  if (n_splits == 1) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (merger)
      *reinterpret_cast<float2*>(prm.out + out_row + d0) = make_float2(O.x * inv, O.y * inv);
    return;
  }

  if constexpr (!kCluster) {
    static_assert(kWarps == kGroup, "the ticket merge maps one warp to each head");
    ticket_merge(sm, prm.part_o, prm.part_ml, prm.tickets, prm.max_splits, prm.out, b, kvh, split,
                 n_splits, M, L, O, warp, lane);
  }
}

// ---------------------------------------------------------------- layer stack
// Consecutive layers of the fused step in one launch: the grid of the
// cluster kernel (S blocks of 4 warps per (sequence, kv head), merged through
// distributed shared memory), made persistent. Each block loops over the
// layers, and each warp's ring of page stages runs on across the layer
// boundary: the pages of cached tokens of layer l + 1, which nothing of layer
// l writes, are in flight while layer l's merge and the wait below run.
// Layer order per sequence: a block reads layer l's q and new k/v, and writes
// its appended slot, only after every block of its sequence has finished
// layer l - 1 (a per-sequence completion counter in global memory, bounded
// wait), the order a model imposes through the rest of the layer. The blocks
// of a sequence wait for one another, so the host launches this grid only
// when all of its clusters are resident at once.
constexpr int kLayerTab = 256;   // block-table entries a block keeps: layers x its pages

struct LayersParams {
  const uint16_t* q;          // [num_layers][batch][32][64]
  const uint16_t* k_new;      // [num_layers][batch][8][64]
  const uint16_t* v_new;
  uint16_t* k_pool;           // [num_pages][8][16][64]
  uint16_t* v_pool;
  const int32_t* tables;      // block tables from the launch's first layer: [.][max_batch][table_stride]
  const int32_t* seq_lens;    // [batch], the same for every layer
  float* out;                 // [num_layers][batch][32][64]
  int* seq_done;              // [batch]: layer completions of the sequence's blocks (zero at launch)
  int* err;
  int num_pages;
  int table_stride;
  size_t table_layer_stride;  // max_batch * table_stride
  int max_seq_len;
  int batch;
  int num_layers;             // layers of this launch
  int wait_extra;             // added to every wait's target: 0, or 1 from the timeout test hook
};

struct alignas(16) LayersSmem {
  WideSmem blk;
  ClusterInbox inbox;
  int ptab[kLayerTab];        // physical page of (layer j, page o of the block's range): j * span + o
  int flag;                   // thread 0's wait verdict for the block
};

// Bounded wait until *ctr >= target (acquire, GPU scope): false after about
// two seconds.
static_assert(4 * (sizeof(LayersSmem) + 1024) <= kSmemPerSm, "4 multi-layer blocks per SM");

__device__ __forceinline__ bool wait_count(const int* ctr, int target) {
  auto load = [&]() {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const long long start = clock64();
  while (load() < target) {
    if (clock64() - start > kWaitCycles) return false;
  }
  return true;
}

__global__ void __launch_bounds__(kClusterWarps * 32, 4) decode_layers_kernel(const LayersParams prm) {
  constexpr int kWarps = kClusterWarps;
  constexpr int kStages = kWideStages;
  constexpr int kThreads = kWarps * 32;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  LayersSmem& ls = *reinterpret_cast<LayersSmem*>(smem_raw);
  WideSmem& sm = ls.blk;

  const int S = static_cast<int>(gridDim.x);
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int J = prm.num_layers;

  // the plan depends on the length only, so every block of a sequence takes
  // the same exits: no block waits for one that left
  const int len = prm.seq_lens[b];
  if (len < 1 || len > prm.max_seq_len) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) set_error(prm.err, kErrSeqLen);
    return;
  }
  const int n_pages = (len + kPage - 1) / kPage;
  const int chunk = (n_pages + S - 1) / S;
  const int n_splits = (n_pages + chunk - 1) / chunk;
  if (n_splits == 1 && split > 0) return;            // one block serves the sequence
  if (chunk * J > kLayerTab) {                        // the host sizes launches below this
    if (split == 0 && kvh == 0 && threadIdx.x == 0) set_error(prm.err, kErrSeqLen);
    return;
  }
  const int arrivals = kHkv * (n_splits == 1 ? 1 : S);   // blocks of the sequence
  const bool active = split < n_splits;              // an idle cluster block only joins merges
  const int page_begin = active ? split * chunk : 0;
  const int span = active ? min(n_pages, page_begin + chunk) - page_begin : 0;
  const int last_page = n_pages - 1;
  const int new_slot = (len - 1) % kPage;

  for (int e = threadIdx.x; e < span * J; e += kThreads) {
    const int j = e / span;
    ls.ptab[e] = prm.tables[static_cast<size_t>(j) * prm.table_layer_stride +
                            static_cast<size_t>(b) * prm.table_stride + page_begin + (e - j * span)];
  }
  WarpSmem<kStages>& ws = sm.warp[warp];
  // this warp's pages of the range: warp, warp + 4, ...; its items run over
  // the layers: item k is page i = k % mine of layer j = k / mine
  const int mine = warp < span ? (span - warp + kWarps - 1) / kWarps : 0;
  const int total = mine * J;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&ws.bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // the warp's page index (within a layer) that holds the appended slot
  const int new_off = last_page - page_begin - warp;
  const int i_new = active && new_off >= 0 && new_off % kWarps == 0 && new_off / kWarps < mine
                        ? new_off / kWarps
                        : -1;
  auto phys_of = [&](int k) {
    const int j = k / mine;
    return ls.ptab[j * span + warp + kWarps * (k - j * mine)];
  };
  // Copy engine: item k into `stage` (lane 0 issues); the last page's copy
  // stops before the appended row, which comes from k/v after the wait
  auto issue_copy = [&](int k, int stage) {
    if (lane != 0) return;
    const int lp = page_begin + warp + kWarps * (k % mine);
    const int phys = phys_of(k);
    const bool ok = phys >= 0 && phys < prm.num_pages;
    const int rows = lp == last_page ? new_slot : kPage;
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
  };
  // the appended row of layer j: lanes 0..7 K, 8..15 V, one 16-byte chunk each
  auto load_new_row = [&](int j) {
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 16) {
      const uint16_t* src = (lane >= 8 ? prm.v_new : prm.k_new) +
                            ((static_cast<size_t>(j) * prm.batch + b) * kHkv + kvh) * kDim +
                            (lane & 7) * 8;
      val = __ldg(reinterpret_cast<const uint4*>(src));
    }
    return val;
  };
  // ... written to the pool and to the stage tile of its page
  auto place_new_row = [&](int stage, int phys, uint4 val) {
    if (lane >= 16 || phys < 0 || phys >= prm.num_pages) return;
    const bool is_v = lane >= 8;
    const int c = lane & 7;
    uint16_t* pool = is_v ? prm.v_pool : prm.k_pool;
    *reinterpret_cast<uint4*>(pool + ((static_cast<size_t>(phys) * kHkv + kvh) * kPage +
                                      new_slot) * kDim + c * 8) = val;
    uint8_t* tile = is_v ? ws.v[stage] : ws.k[stage];
    *reinterpret_cast<uint4*>(tile + new_slot * kRowBytes + c * 16) = val;
  };

  int issued = min(total, kStages);
  for (int k = 0; k < issued; ++k) issue_copy(k, k);

  const LaneRoles rl(lane);
  const float no_angles[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int k = 0;                 // next item to consume
  int consumed = 0;
  bool broken = false;       // a page wait gave up: this warp copies and computes no more
  bool waits_off = false;    // a sequence wait gave up: the block stops waiting (flagged)
  for (int j = 0; j < J; ++j) {
    if (j > 0 && !waits_off) {
      if (threadIdx.x == 0)
        ls.flag = wait_count(prm.seq_done + b, j * arrivals + prm.wait_extra) ? 0 : 1;
      __syncthreads();
      if (ls.flag) {
        waits_off = true;
        if (threadIdx.x == 0) set_error(prm.err, kErrTimeout);
      }
    }
    // q and the new k/v rows of the next layer into L2 while this one runs
    if (warp == 0 && lane < 6 && active && j + 1 < J) {
      const size_t row = static_cast<size_t>(j + 1) * prm.batch + b;
      const uint16_t* line = lane < 4 ? prm.q + (row * kHq + kvh * kGroup + lane) * kDim
                                      : (lane == 4 ? prm.k_new : prm.v_new) +
                                            (row * kHkv + kvh) * kDim;
      prefetch_l2(line);
    }
    const int item_new = i_new >= 0 ? j * mine + i_new : -1;   // this layer's appended-row item
    const bool place_now = item_new >= 0 && item_new < issued && !broken;
    uint4 new_val = make_uint4(0u, 0u, 0u, 0u);
    if (place_now) new_val = load_new_row(j);
    float2 qa[kGroup][4], qb[kGroup][4];
    load_q<false>(prm.q + ((static_cast<size_t>(j) * prm.batch + b) * kHq + kvh * kGroup) * kDim,
                  rl, qa, qb, no_angles, no_angles);
    if (place_now) place_new_row(item_new % kStages, phys_of(item_new), new_val);
    __syncwarp();

    WarpState st;
    st.reset();
    bool lost = false;       // this layer's pages are incomplete
    // tokens of item k (page i of this layer) that count
    auto live_of = [&](int k, int i) {
      const int lp = page_begin + warp + kWarps * i;
      const int valid = lp == last_page ? len - lp * kPage : kPage;
      const int phys = phys_of(k);
      return phys >= 0 && phys < prm.num_pages ? valid : 0;
    };
    // after item k is consumed: the copy of item k + kStages into its stage
    auto refill = [&](int k) {
      const int kn = k + kStages;
      if (kn < total) {
        issue_copy(kn, k % kStages);
        // a later item of this layer holding the appended slot: its row now
        if (kn == item_new) place_new_row(k % kStages, phys_of(kn), load_new_row(j));
        __syncwarp();
        issued = kn + 1;
      }
    };
    for (int i = 0; i < mine && !broken; ++i, ++k) {
      // one verdict per warp: the page work below shuffles across all lanes
      if (!__all_sync(0xffffffffu, mbar_wait(&ws.bar[k % kStages], (k / kStages) & 1))) {
        broken = true;
        if (lane == 0) set_error(prm.err, kErrTimeout);
        break;
      }
      consumed = k + 1;
      attend_page(ws.k[k % kStages], ws.v[k % kStages], live_of(k, i), qa, qb, ws.p, ws.alpha,
                  rl, st);
      refill(k);
    }
    lost |= broken;
    k = (j + 1) * mine;      // the next layer's first item (also after a break)
    reduce_warp_state(st);
    if (lost) {
      st.m_run = -INFINITY;
      st.l_run = 0.f;
    }
    float* out_kv = prm.out + ((static_cast<size_t>(j) * prm.batch + b) * kHq + kvh * kGroup) * kDim;
    if (n_splits > 1) {
      cluster_merge(sm, ls.inbox, st, rl, warp, lane, out_kv, true);
    } else {
      float M, L;
      float2 O;
      block_merge(sm, st, rl, warp, M, L, O);
      const int g = (threadIdx.x >> 5) & (kGroup - 1);
      const int d0 = 2 * (threadIdx.x & 31);
      const float inv = L > 0.f ? 1.f / L : 0.f;
      *reinterpret_cast<float2*>(out_kv + g * kDim + d0) = make_float2(O.x * inv, O.y * inv);
    }
    // this block is done with layer j: its output rows are written
    __syncthreads();
    if (j + 1 < J && threadIdx.x == 0) {
      __threadfence();
      atomicAdd(prm.seq_done + b, 1);
    }
  }
  if (broken) {
    // let this warp's copies still in flight land before the block exits
    // (each wait bounded again)
    for (int kk = consumed; kk < issued; ++kk) mbar_wait(&ws.bar[kk % kStages], (kk / kStages) & 1);
  }
}

}  // namespace

// ================================================================= host side

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The three kernel shapes (the cluster kernels add the leaders' inbox).
enum Shape { kTicketShape = 0, kNarrowShape = 1, kWideShape = 2 };
template <bool kFused, bool kRope = false>
constexpr auto ticket_kernel = decode_kernel<kFused, false, kTicketWarps, kTicketStages, kRope>;
template <bool kFused, bool kRope = false>
constexpr auto narrow_kernel = decode_kernel<kFused, true, kClusterWarps, kNarrowStages, kRope>;
template <bool kFused, bool kRope = false>
constexpr auto wide_kernel = decode_kernel<kFused, true, kClusterWarps, kWideStages, kRope>;

size_t smem_bytes(Shape shape) {
  switch (shape) {
    case kNarrowShape: return sizeof(NarrowSmem) + sizeof(ClusterInbox);
    case kWideShape: return sizeof(WideSmem) + sizeof(ClusterInbox);
    default: return sizeof(TicketSmem);
  }
}

int block_threads(Shape shape) {
  return 32 * (shape == kTicketShape ? kTicketWarps : kClusterWarps);
}

template <typename Kernel>
bool set_kernel_attributes(Kernel kernel, Shape shape) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes(shape))) != cudaSuccess)
    return false;
  if (shape != kTicketShape &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess)
    return false;
  return true;
}

pkv_status check_launch() {
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}


static_assert(kTicketShape == PKV_SHAPE_TICKET && kNarrowShape == PKV_SHAPE_NARROW &&
                  kWideShape == PKV_SHAPE_WIDE,
              "the plan's shape codes are the kernel shapes");

// Pages per block when the caller leaves the choice to the library and the
// batch is too large for a cluster split: the largest of 128, 64, 32, 16
// pages for which a batch of full-length sequences still yields at least
// three (sequence, kv head, range) blocks per resident block slot. Fewer
// blocks per slot leave SMs idle behind the longest sequences; more, smaller
// ranges pay a partial merge for nothing (measured: 256 sequences run best
// unsplit, 64 log-uniform ones with 32-page ranges).
int auto_chunk_pages(const pkv_device_figures& d, int batch) {
  const int max_pages = d.max_seq_len / kPage;
  const int min_chunk = (max_pages + d.max_splits - 1) / d.max_splits;
  const long long resident = static_cast<long long>(d.ticket_blocks_per_sm) * d.num_sms;
  int chunk = 16;
  for (int c = 128; c >= 16; c /= 2) {
    const long long blocks = static_cast<long long>(batch) * kHkv * ((max_pages + c - 1) / c);
    if (blocks >= 3 * resident) {
      chunk = c;
      break;
    }
  }
  if (chunk > max_pages) chunk = max_pages;
  return chunk < min_chunk ? min_chunk : chunk;
}

// The launch plan for a batch. Cluster plans when the library chooses: the
// split count S (16, 8, 4, 2) and the block shape, from a sweep on a 152-SM
// GB300 with full-length sequences (GB/s per 16-layer step):
//   batch 2:  narrow S = 16 (256 blocks) 1522; wide S = 16 1453; S = 8 1337;
//   batch 4:  narrow S = 8 (256) 2304; narrow S = 16 1404; wide S = 8 2015;
//   batch 8:  wide S = 8 (512) 3462; narrow S = 4 (256) 2680; wide S = 16 2016;
//   batch 16: wide S = 4 (512) 4214; narrow S = 2 (256) 3187; wide S = 8 3443.
// So: the narrow shape with the largest S whose blocks take at most 9/16 of
// its resident slots (256 of 456, leaving room for the next launch), if that
// S is at least 8; else the wide shape with the largest S <= 8 whose blocks
// take at most 27/32 of its slots (512 of 608); else (large batches) the
// ticket merge over page ranges.
pkv_plan plan_decode(const pkv_device_figures& d, int batch, int num_splits) {
  const int max_pages = d.max_seq_len / kPage;
  const long long narrow = static_cast<long long>(d.narrow_blocks_per_sm) * d.num_sms;
  const long long wide = static_cast<long long>(d.wide_blocks_per_sm) * d.num_sms;
  pkv_plan p = {};
  p.shape = kTicketShape;
  if (num_splits == 0) {
    auto usable = [&](int s) {
      return s <= d.max_cluster && s <= d.max_splits && s <= max_pages;
    };
    for (int s = kMaxClusterSize; s >= 8 && !p.cluster; s /= 2) {
      if (usable(s) && 16 * static_cast<long long>(batch) * kHkv * s <= 9 * narrow) {
        p.cluster = s;
        p.shape = kNarrowShape;
      }
    }
    for (int s = 8; s >= 2 && !p.cluster; s /= 2) {
      if (usable(s) && 32 * static_cast<long long>(batch) * kHkv * s <= 27 * wide) {
        p.cluster = s;
        p.shape = kWideShape;
      }
    }
    if (p.cluster) {
      p.num_splits = p.cluster;
    } else {
      p.chunk_pages = auto_chunk_pages(d, batch);
    }
  } else {
    p.num_splits = num_splits;
    if (num_splits >= 2 && num_splits <= d.max_cluster) {
      // a chosen split count takes the narrow shape while its blocks fit one
      // wave of it, the wide shape beyond
      p.cluster = num_splits;
      p.shape = static_cast<long long>(batch) * kHkv * num_splits <= narrow ? kNarrowShape
                                                                           : kWideShape;
    }
  }
  p.grid_splits = p.num_splits > 0 ? p.num_splits
                                   : (max_pages + p.chunk_pages - 1) / p.chunk_pages;
  const long long blocks = static_cast<long long>(p.grid_splits) * kHkv * batch;
  const int per_sm = p.shape == kNarrowShape  ? d.narrow_blocks_per_sm
                     : p.shape == kWideShape ? d.wide_blocks_per_sm
                                             : d.ticket_blocks_per_sm;
  const long long resident = static_cast<long long>(per_sm) * d.num_sms;
  p.early_trigger = blocks <= resident ? 1 : 0;
  // more than one wave of ticket-mode blocks: longest sequences first
  p.longest_first = (!p.cluster && num_splits == 0 && blocks > resident) ? 1 : 0;
  return p;
}

pkv_device_figures figures_of(const pkv_pool* pool) {
  pkv_device_figures d;
  d.num_sms = pool->num_sms;
  d.ticket_blocks_per_sm = pool->blocks_per_sm;
  d.narrow_blocks_per_sm = pool->cluster_blocks_per_sm;
  d.wide_blocks_per_sm = pool->wide_blocks_per_sm;
  d.max_cluster = pool->max_cluster;
  d.max_splits = pool->cfg.max_splits;
  d.max_seq_len = pool->cfg.max_seq_len;
  return d;
}

// Cluster size of the multi-layer launch: the largest S of 16, 8, 4, 2 (within
// the device's cluster limit, max_splits and the pages of a full sequence)
// for which all batch x 8 clusters are resident at once; 0 when none is.
int layers_cluster_splits(const pkv_pool* pool, int batch) {
  const int max_pages = pool->cfg.max_seq_len / kPage;
  for (int e = 4; e >= 1; --e) {
    const int s = 1 << e;
    if (s > pool->max_cluster || s > pool->cfg.max_splits || s > max_pages) continue;
    if (static_cast<long long>(batch) * kHkv <= pool->layer_clusters[e]) return s;
  }
  return 0;
}

template <bool kFused>
pkv_status launch_decode(pkv_pool_t pool, int layer, const void* q, const void* k,
                         const void* v, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* seq_lens, float* out,
                         int batch, int num_splits, void* stream,
                         const float* rope_cos = nullptr, const float* rope_sin = nullptr,
                         bool rope = false) {
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
  if (rope && (!rope_cos || !rope_sin || !aligned16(rope_cos) || !aligned16(rope_sin)))
    return PKV_ERR_INVALID_ARG;

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
  prm.rope_cos = rope ? rope_cos : nullptr;
  prm.rope_sin = rope ? rope_sin : nullptr;

  // Plan: S splits per sequence merged in a cluster when 2 <= S <= the
  // largest cluster this device schedules; otherwise (S = 1, S larger, or a
  // batch too large for one wave of clusters) global partials and a ticket.
  const pkv_plan plan = plan_decode(figures_of(pool), batch, num_splits);
  const Shape shape = static_cast<Shape>(plan.shape);
  const int cluster = plan.cluster;
  const int grid_splits = plan.grid_splits;
  prm.num_splits = plan.num_splits;
  prm.chunk_pages = plan.chunk_pages;
  prm.early_trigger = plan.early_trigger;
  prm.longest_first = plan.longest_first;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_splits, kHkv, batch);
  cfg.blockDim = dim3(block_threads(shape), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes(shape);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[2];
  int n_attrs = 0;
  if (cluster) {
    attrs[n_attrs].id = cudaLaunchAttributeClusterDimension;
    attrs[n_attrs].val.clusterDim.x = cluster;
    attrs[n_attrs].val.clusterDim.y = 1;
    attrs[n_attrs].val.clusterDim.z = 1;
    ++n_attrs;
  }
  if (c.flags & PKV_FLAG_PDL) {
    attrs[n_attrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n_attrs].val.programmaticStreamSerializationAllowed = 1;
    ++n_attrs;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n_attrs;
  cudaError_t e;
  if (rope) {
    e = shape == kNarrowShape ? cudaLaunchKernelEx(&cfg, narrow_kernel<kFused, true>, prm)
        : shape == kWideShape ? cudaLaunchKernelEx(&cfg, wide_kernel<kFused, true>, prm)
                              : cudaLaunchKernelEx(&cfg, ticket_kernel<kFused, true>, prm);
  } else {
    e = shape == kNarrowShape ? cudaLaunchKernelEx(&cfg, narrow_kernel<kFused>, prm)
        : shape == kWideShape ? cudaLaunchKernelEx(&cfg, wide_kernel<kFused>, prm)
                              : cudaLaunchKernelEx(&cfg, ticket_kernel<kFused>, prm);
  }
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return check_launch();
}

// ---------------------------------------------------------------- no-allocation entry point
// Scratch of pkv_decode_attention_noalloc: split partials and tickets for up
// to kStaticRows (sequence, split) pairs, plus a sink for unreported errors.
constexpr int kStaticRows = 256;        // batch x num_splits
constexpr int kStaticMaxSplits = 16;

struct StaticScratch {
  float part_o[kStaticRows * kHq][kDim];
  float2 part_ml[kStaticRows * kHq];
  int tickets[kStaticRows * kHkv];
  int error_sink;
};

static __device__ __align__(256) unsigned char g_static_scratch[sizeof(StaticScratch)];

// Device address of g_static_scratch per device, looked up once (the array's
// name in host code is only a stand-in, not a device address).
pkv_status static_scratch_address(StaticScratch** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex lock;
  static StaticScratch* address[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> guard(lock);
  if (!address[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return PKV_ERR_CUDA;
    if (!set_kernel_attributes(ticket_kernel<false>, kTicketShape)) return PKV_ERR_CUDA;
    address[dev] = static_cast<StaticScratch*>(ptr);
  }
  *out = address[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_attention_noalloc(int layer, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* block_tables,
                                        const int32_t* seq_lens, float* out, int num_layers,
                                        int num_pages, int max_batch, int max_seq_len,
                                        int batch, int num_splits, int* error_bits,
                                        void* stream) {
  if (num_layers < 1 || num_pages < 1 || max_batch < 1 || max_seq_len < kPage ||
      max_seq_len > kMaxSeqLen || max_seq_len % kPage != 0 || max_batch > 65535)
    return PKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= num_layers || batch < 0 || batch > max_batch)
    return PKV_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > kStaticMaxSplits || batch > kStaticRows ||
      static_cast<long long>(batch) * num_splits > kStaticRows)
    return PKV_ERR_STATIC_LIMIT;
  if (batch == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(block_tables) ||
      !aligned16(seq_lens) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(error_bits) & 3u) != 0)
    return PKV_ERR_INVALID_ARG;

  StaticScratch* scratch = nullptr;
  const pkv_status st = static_scratch_address(&scratch);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // tickets must start at zero; the array keeps whatever the last call left
  if (cudaMemsetAsync(scratch->tickets, 0, static_cast<size_t>(batch) * kHkv * sizeof(int), s) !=
      cudaSuccess)
    return PKV_ERR_CUDA;

  const int max_pages = max_seq_len / kPage;
  DecodeParams prm;
  prm.q = static_cast<const uint16_t*>(q);
  prm.k_new = nullptr;
  prm.v_new = nullptr;
  prm.k_pool = const_cast<uint16_t*>(static_cast<const uint16_t*>(k_pool));
  prm.v_pool = const_cast<uint16_t*>(static_cast<const uint16_t*>(v_pool));
  prm.table = block_tables + static_cast<size_t>(layer) * max_batch * max_pages;
  prm.seq_lens = seq_lens;
  prm.out = out;
  prm.part_o = &scratch->part_o[0][0];
  prm.part_ml = scratch->part_ml;
  prm.tickets = scratch->tickets;
  prm.err = error_bits ? error_bits : &scratch->error_sink;
  prm.num_pages = num_pages;
  prm.table_stride = max_pages;
  prm.max_seq_len = max_seq_len;
  prm.max_splits = num_splits;     // partial rows are (sequence, head) x num_splits
  prm.num_splits = num_splits;
  prm.chunk_pages = 0;
  prm.early_trigger = 1;   // launched without programmatic dependent launch: no effect
  prm.longest_first = 0;
  prm.rope_cos = nullptr;
  prm.rope_sin = nullptr;
  ticket_kernel<false><<<dim3(num_splits, kHkv, batch), block_threads(kTicketShape),
                         smem_bytes(kTicketShape),
                         s>>>(prm);
  return check_launch();
}

const char* pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_OUT_OF_RANGE: return "index out of range in device data";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_UNSUPPORTED: return "unsupported geometry";
    case PKV_ERR_DEVICE_TIMEOUT: return "bounded device wait timed out";
    case PKV_ERR_STATIC_LIMIT: return "request exceeds the no-allocation entry point's scratch";
  }
  return "unknown status";
}

pkv_status pkv_plan_decode(const pkv_device_figures* dev, int batch, int num_splits,
                           pkv_plan* out) {
  if (!dev || !out) return PKV_ERR_INVALID_ARG;
  const pkv_device_figures& d = *dev;
  if (d.num_sms < 1 || d.ticket_blocks_per_sm < 1 || d.narrow_blocks_per_sm < 1 ||
      d.wide_blocks_per_sm < 1 || d.max_cluster < 0 || d.max_cluster > kMaxClusterSize ||
      d.max_splits < 1 || d.max_splits > kMaxSplitsLimit || d.max_seq_len < kPage ||
      d.max_seq_len > kMaxSeqLen || d.max_seq_len % kPage != 0)
    return PKV_ERR_INVALID_ARG;
  if (batch < 1 || num_splits < 0 || num_splits > d.max_splits) return PKV_ERR_INVALID_ARG;
  *out = plan_decode(d, batch, num_splits);
  return PKV_OK;
}

pkv_status pkv_pool_device_figures(pkv_pool_t pool, pkv_device_figures* out) {
  if (!pool || !out) return PKV_ERR_INVALID_ARG;
  *out = figures_of(pool);
  return PKV_OK;
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
  ok = ok && cudaMalloc(&pool->seq_done, static_cast<size_t>(c.max_batch) * sizeof(int)) ==
                 cudaSuccess;

  ok = ok && cudaMemset(pool->tickets, 0, 2 * static_cast<size_t>(c.max_batch) * kHkv * sizeof(int)) ==
                 cudaSuccess;
  ok = ok && cudaMemset(pool->err, 0, sizeof(int)) == cudaSuccess;
  ok = ok && set_kernel_attributes(ticket_kernel<false>, kTicketShape);
  ok = ok && set_kernel_attributes(ticket_kernel<true>, kTicketShape);
  ok = ok && set_kernel_attributes(narrow_kernel<false>, kNarrowShape);
  ok = ok && set_kernel_attributes(narrow_kernel<true>, kNarrowShape);
  ok = ok && set_kernel_attributes(wide_kernel<false>, kWideShape);
  ok = ok && set_kernel_attributes(wide_kernel<true>, kWideShape);
  ok = ok && set_kernel_attributes(ticket_kernel<false, true>, kTicketShape);
  ok = ok && set_kernel_attributes(ticket_kernel<true, true>, kTicketShape);
  ok = ok && set_kernel_attributes(narrow_kernel<false, true>, kNarrowShape);
  ok = ok && set_kernel_attributes(narrow_kernel<true, true>, kNarrowShape);
  ok = ok && set_kernel_attributes(wide_kernel<false, true>, kWideShape);
  ok = ok && set_kernel_attributes(wide_kernel<true, true>, kWideShape);
  ok = ok && cudaFuncSetAttribute(decode_layers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sizeof(LayersSmem))) == cudaSuccess;
  ok = ok && cudaFuncSetAttribute(decode_layers_kernel,
                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;

  ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                  &pool->blocks_per_sm, ticket_kernel<true>, block_threads(kTicketShape),
                  smem_bytes(kTicketShape)) == cudaSuccess;
  ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                  &pool->cluster_blocks_per_sm, narrow_kernel<true>, block_threads(kNarrowShape),
                  smem_bytes(kNarrowShape)) == cudaSuccess;
  ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                  &pool->wide_blocks_per_sm, wide_kernel<true>, block_threads(kWideShape),
                  smem_bytes(kWideShape)) == cudaSuccess;
  pool->max_cluster = 0;
  for (int size = kMaxClusterSize; ok && size >= 2 && !pool->max_cluster; size /= 2) {
    cudaLaunchConfig_t probe = {};
    probe.gridDim = dim3(size, kHkv, 1);
    probe.blockDim = dim3(block_threads(kNarrowShape), 1, 1);
    probe.dynamicSmemBytes = smem_bytes(kNarrowShape);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = size;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    probe.attrs = &attr;
    probe.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, narrow_kernel<true>, &probe) ==
            cudaSuccess && clusters > 0)
      pool->max_cluster = size;
    cudaGetLastError();   // a size the device refuses is not an error here
  }
  // how many clusters of the multi-layer kernel the device holds at once,
  // per cluster size: its blocks wait for one another, so it launches only
  // grids that fit
  for (int e = 0; e < 5; ++e) {
    const int size = 1 << e;
    pool->layer_clusters[e] = 0;
    if (!ok) continue;
    cudaLaunchConfig_t probe = {};
    probe.gridDim = dim3(size, kHkv, 1);
    probe.blockDim = dim3(kClusterWarps * 32, 1, 1);
    probe.dynamicSmemBytes = sizeof(LayersSmem);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = size;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    probe.attrs = &attr;
    probe.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, decode_layers_kernel, &probe) == cudaSuccess)
      pool->layer_clusters[e] = clusters;
    cudaGetLastError();   // a size the device refuses is not an error here
  }
  if (ok && pool->blocks_per_sm < 1) pool->blocks_per_sm = 1;
  if (ok && pool->cluster_blocks_per_sm < 1) pool->cluster_blocks_per_sm = 1;
  if (ok && pool->wide_blocks_per_sm < 1) pool->wide_blocks_per_sm = 1;

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
  cudaFree(pool->seq_done);
  delete pool;
  return st;
}

}  // extern "C"

namespace {

pkv_status launch_append(pkv_pool_t pool, int layer, const void* k, const void* v, void* k_pool,
                         void* v_pool, const int32_t* block_tables, const int32_t* positions,
                         const float* rope_cos, const float* rope_sin, bool rope, int batch,
                         void* stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  if (layer < 0 || layer >= c.num_layers || batch < 0 || batch > c.max_batch)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!k || !v || !k_pool || !v_pool || !block_tables || !positions) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(block_tables) || !aligned16(positions))
    return PKV_ERR_INVALID_ARG;
  if (rope && (!rope_cos || !rope_sin || !aligned16(rope_cos) || !aligned16(rope_sin)))
    return PKV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_ERR_INVALID_ARG;
  const int max_pages = c.max_seq_len / kPage;
  append_kernel<<<batch, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
      static_cast<uint16_t*>(k_pool), static_cast<uint16_t*>(v_pool),
      block_tables + static_cast<size_t>(layer) * c.max_batch * max_pages, positions, max_pages,
      c.num_pages, c.max_seq_len, pool->err, rope ? rope_cos : nullptr,
      rope ? rope_sin : nullptr);
  return check_launch();
}

}  // namespace

extern "C" {

pkv_status pkv_append(pkv_pool_t pool, int layer, const void* k, const void* v, void* k_pool,
                      void* v_pool, const int32_t* block_tables, const int32_t* positions,
                      int batch, void* stream) {
  return launch_append(pool, layer, k, v, k_pool, v_pool, block_tables, positions, nullptr,
                       nullptr, false, batch, stream);
}

pkv_status pkv_append_rope(pkv_pool_t pool, int layer, const void* k, const void* v,
                           void* k_pool, void* v_pool, const int32_t* block_tables,
                           const int32_t* positions, const float* rope_cos,
                           const float* rope_sin, int batch, void* stream) {
  return launch_append(pool, layer, k, v, k_pool, v_pool, block_tables, positions, rope_cos,
                       rope_sin, true, batch, stream);
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

}  // extern "C"

namespace {

// The multi-layer step; wait_extra > 0 makes every layer wait unreachable
// (the timeout test hook), and then there is no per-layer fallback.
pkv_status launch_layers(pkv_pool_t pool, int layer_begin, int num_layers, const void* q,
                         const void* k, const void* v, void* k_pool, void* v_pool,
                         const int32_t* block_tables, const int32_t* seq_lens, float* out,
                         int batch, void* stream, int wait_extra) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  const pkv_pool_config& c = pool->cfg;
  if (layer_begin < 0 || num_layers < 0 ||
      static_cast<long long>(layer_begin) + num_layers > c.num_layers || batch < 0 ||
      batch > c.max_batch)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0 || num_layers == 0) return PKV_OK;
  if (!q || !k || !v || !k_pool || !v_pool || !block_tables || !seq_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_pool) ||
      !aligned16(v_pool) || !aligned16(block_tables) || !aligned16(seq_lens) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_ERR_INVALID_ARG;

  const size_t q_layer = static_cast<size_t>(batch) * kHq * kDim;     // elements per layer
  const size_t kv_layer = static_cast<size_t>(batch) * kHkv * kDim;
  const uint16_t* q16 = static_cast<const uint16_t*>(q);
  const uint16_t* k16 = static_cast<const uint16_t*>(k);
  const uint16_t* v16 = static_cast<const uint16_t*>(v);
  const int S = layers_cluster_splits(pool, batch);
  if (S == 0 && wait_extra) return PKV_ERR_UNSUPPORTED;
  if (S == 0) {
    // too many sequences for a resident grid: one fused launch per layer
    for (int j = 0; j < num_layers; ++j) {
      const pkv_status st = launch_decode<true>(pool, layer_begin + j, q16 + j * q_layer,
                                                k16 + j * kv_layer, v16 + j * kv_layer, k_pool,
                                                v_pool, block_tables, seq_lens, out + j * q_layer,
                                                batch, 0, stream);
      if (st != PKV_OK) return st;
    }
    return PKV_OK;
  }

  const int max_pages = c.max_seq_len / kPage;
  const int chunk_max = (max_pages + S - 1) / S;
  const int per_launch = kLayerTab / chunk_max;   // >= 4: chunk_max <= 64
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int j0 = 0; j0 < num_layers; j0 += per_launch) {
    const int J = std::min(per_launch, num_layers - j0);
    if (J > 1 && cudaMemsetAsync(pool->seq_done, 0, static_cast<size_t>(batch) * sizeof(int), s) !=
                     cudaSuccess)
      return PKV_ERR_CUDA;
    LayersParams prm;
    prm.q = q16 + j0 * q_layer;
    prm.k_new = k16 + j0 * kv_layer;
    prm.v_new = v16 + j0 * kv_layer;
    prm.k_pool = static_cast<uint16_t*>(k_pool);
    prm.v_pool = static_cast<uint16_t*>(v_pool);
    prm.table_stride = max_pages;
    prm.table_layer_stride = static_cast<size_t>(c.max_batch) * max_pages;
    prm.tables = block_tables + static_cast<size_t>(layer_begin + j0) * prm.table_layer_stride;
    prm.seq_lens = seq_lens;
    prm.out = out + j0 * q_layer;
    prm.seq_done = pool->seq_done;
    prm.err = pool->err;
    prm.num_pages = c.num_pages;
    prm.max_seq_len = c.max_seq_len;
    prm.batch = batch;
    prm.num_layers = J;
    prm.wait_extra = wait_extra;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, kHkv, batch);
    cfg.blockDim = dim3(kClusterWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = sizeof(LayersSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = S;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_layers_kernel, prm) != cudaSuccess) return PKV_ERR_CUDA;
  }
  return check_launch();
}

}  // namespace

extern "C" {

pkv_status pkv_append_attend_layers(pkv_pool_t pool, int layer_begin, int num_layers,
                                    const void* q, const void* k, const void* v, void* k_pool,
                                    void* v_pool, const int32_t* block_tables,
                                    const int32_t* seq_lens, float* out, int batch,
                                    void* stream) {
  return launch_layers(pool, layer_begin, num_layers, q, k, v, k_pool, v_pool, block_tables,
                       seq_lens, out, batch, stream, 0);
}

pkv_status pkv_test_layers_wait_timeout(pkv_pool_t pool, int layer_begin, int num_layers,
                                        const void* q, const void* k, const void* v,
                                        void* k_pool, void* v_pool, const int32_t* block_tables,
                                        const int32_t* seq_lens, float* out, int batch,
                                        void* stream) {
  return launch_layers(pool, layer_begin, num_layers, q, k, v, k_pool, v_pool, block_tables,
                       seq_lens, out, batch, stream, 1);
}

pkv_status pkv_decode_attention_rope(pkv_pool_t pool, int layer, const void* q,
                                     const void* k_pool, const void* v_pool,
                                     const int32_t* block_tables, const int32_t* seq_lens,
                                     const float* rope_cos, const float* rope_sin, float* out,
                                     int batch, int num_splits, void* stream) {
  return launch_decode<false>(pool, layer, q, nullptr, nullptr, k_pool, v_pool, block_tables,
                              seq_lens, out, batch, num_splits, stream, rope_cos, rope_sin, true);
}

pkv_status pkv_append_attend_rope(pkv_pool_t pool, int layer, const void* q, const void* k,
                                  const void* v, void* k_pool, void* v_pool,
                                  const int32_t* block_tables, const int32_t* seq_lens,
                                  const float* rope_cos, const float* rope_sin, float* out,
                                  int batch, int num_splits, void* stream) {
  return launch_decode<true>(pool, layer, q, k, v, k_pool, v_pool, block_tables, seq_lens, out,
                             batch, num_splits, stream, rope_cos, rope_sin, true);
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
