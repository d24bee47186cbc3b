// Internal to libpkv: the decode kernels' building blocks, shared by the
// per-layer decode kernels (pkv.cu) and the multi-layer kernel (layers.cu):
// block shapes and their shared-memory layouts, the decode parameters, PTX
// helpers (clusters, bulk copies, programmatic dependent launch), the per-page
// math (scores, online softmax, P V), and the warp, cluster and ticket merges
// [samir-vllm: Build LLM Inference From Scratch in C++ and CUDA,
// "Architecture walkthrough", KV cache paragraph; 6 Hours of YouTube and 85
// handtyped pages of notes on LLM Inference - Start here, README feature
// list, direct paged decode attention bullet].
#ifndef PKV_DECODE_DEVICE_CUH
#define PKV_DECODE_DEVICE_CUH

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "device_common.cuh"
#include "pool_internal.h"

namespace pkv_decode {

using namespace pkv_dev;


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
constexpr int kWideWarps = 4;
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

// A head leader's inbox for the asynchronous cluster merge (decode_kernel):
// every block of the cluster delivers its (o, m, l) for the heads this block
// leads with st.async stores that complete on `bar` in transaction bytes, so
// the leader wakes as soon as its parts have landed, with no cluster-wide
// barrier at the end. Slot of block r for head g: (g / S) * S + r.
struct alignas(16) AsyncInbox {
  float o[kInboxSlots][kDim];
  float2 ml[kInboxSlots];
  unsigned long long bar;
};
constexpr uint32_t kPartBytes = (kDim + 2) * sizeof(float);   // one (o, m, l) part: 264 B

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
using WideSmem = BlockSmem<kWideWarps, kWideStages>;
static_assert(sizeof(WarpSmem<kTicketStages>) % 16 == 0 &&
                  sizeof(WarpSmem<kWideStages>) % 16 == 0,
              "warp slabs keep 16-byte alignment");
static_assert(sizeof(NarrowSmem) % 16 == 0 && sizeof(WideSmem) % 16 == 0,
              "the cluster inbox follows BlockSmem 16-byte aligned");
static_assert(sizeof(ClusterInbox) % 16 == 0 && sizeof(AsyncInbox) % 16 == 0,
              "inbox sizes keep 16-byte alignment");
static_assert(sizeof(AsyncInbox) <= sizeof(ClusterInbox) + 16, "the inboxes take the same room");
// residency the kernels are shaped for: 228 KiB of shared memory per SM, 1 KiB
// of it reserved per block; 4 ticket blocks or 3 cluster blocks per SM
constexpr size_t kSmemPerSm = 228 * 1024;
static_assert(4 * (sizeof(TicketSmem) + 1024) <= kSmemPerSm, "4 ticket blocks per SM");
static_assert(3 * (sizeof(NarrowSmem) + sizeof(AsyncInbox) + 1024) <= kSmemPerSm,
              "3 narrow cluster blocks per SM");
static_assert((16 / kWideWarps) * (sizeof(WideSmem) + sizeof(AsyncInbox) + 1024) <=
                  kSmemPerSm,
              "16 warps of wide cluster blocks per SM");

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

// Shared-memory address of the same offset in cluster block `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t addr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(p)), "r"(rank));
  return addr;
}

// Asynchronous store of two floats into another block's shared memory,
// completing 8 transaction bytes on that block's mbarrier `rbar`.
__device__ __forceinline__ void st_async2(uint32_t raddr, float2 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
      ::"r"(raddr), "f"(v.x), "f"(v.y), "r"(rbar)
      : "memory");
}

// Bounded wait on an mbarrier phase whose transactions come from other
// blocks of the cluster (acquire at cluster scope): false after ~2 s.
__device__ __forceinline__ bool mbar_wait_cluster(unsigned long long* bar, uint32_t parity) {
  constexpr uint32_t kSuspendHintNs = 10000000;
  auto try_once = [&]() {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return done != 0;
  };
  if (try_once()) return true;
  const long long start = clock64();
  while (!try_once()) {
    if (clock64() - start > kWaitCycles) return false;
  }
  return true;
}

// Heads g < 4 that cluster block `rank` leads (g mod S == rank).
__device__ __forceinline__ int heads_led(int rank, int S) {
  int n = 0;
  #pragma unroll
  for (int g = 0; g < kGroup; ++g) n += g % S == rank ? 1 : 0;
  return n;
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
  static_assert(kWarps % kGroup == 0, "threads 0..127 hold one (head, dim pair) each");
  float M, L;
  float2 O;
  block_merge(sm, st, rl, warp, M, L, O);
  const int S = gridDim.x;
  const int rank = static_cast<int>(cluster_rank());
  const int g = warp;               // thread t < 128: head t / 32, dims 2 (t % 32), + 1
  const int d0 = 2 * lane;
  if (g < kGroup) {
    const int at = (g / S) * S + rank;
    st_cluster2(&inbox.o[at][d0], g % S, O);
    if (lane == 0) {
      st_cluster(&inbox.m[at], g % S, M);
      st_cluster(&inbox.l[at], g % S, L);
    }
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

// The leader's inbox barrier, before any block of the cluster sends: thread 0
// of a leader initialises it and arms it for the S parts of every head it
// leads; then every thread of the cluster meets on the cluster barrier, so
// no part can arrive at an uninitialised barrier. Called by every thread.
__device__ __forceinline__ void async_inbox_setup(AsyncInbox& inbox) {
  const int S = static_cast<int>(gridDim.x);
  const int rank = static_cast<int>(cluster_rank());
  const int led = heads_led(rank, S);
  if (threadIdx.x == 0 && led > 0) {
    mbar_init(&inbox.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&inbox.bar, static_cast<uint32_t>(led * S) * kPartBytes);
  }
  cluster_arrive_release();
  cluster_wait_acquire();
}

// Cluster merge without a closing cluster barrier: each block merges its
// warps (block_merge), then threads 0..127 send the block's (o, m, l) part of
// head t / 32 to the head's leader (block g mod S) with st.async stores; a
// block that leads no head is then done. In a leader, warp w waits until the
// parts of head rank + w S have landed and combines them into out_kv.
template <int kWarps, int kStages>
__device__ __forceinline__ void cluster_merge_async(BlockSmem<kWarps, kStages>& sm,
                                                    AsyncInbox& inbox, const WarpState& st,
                                                    const LaneRoles& rl, int warp, int lane,
                                                    float* out_kv, int* err) {
  static_assert(kWarps % kGroup == 0, "threads 0..127 hold one (head, dim pair) each");
  float M, L;
  float2 O;
  block_merge(sm, st, rl, warp, M, L, O);
  const int S = gridDim.x;
  const int rank = static_cast<int>(cluster_rank());
  const int d0 = 2 * lane;
  if (warp < kGroup) {
    const int g = warp;
    const uint32_t dst = static_cast<uint32_t>(g % S);
    const int at = (g / S) * S + rank;
    const uint32_t rbar = cluster_addr(&inbox.bar, dst);
    st_async2(cluster_addr(&inbox.o[at][d0], dst), O, rbar);
    if (lane == 0) st_async2(cluster_addr(&inbox.ml[at], dst), make_float2(M, L), rbar);
  }
  if (rank >= kGroup) return;                  // leads no head
  const int hg = rank + warp * S;             // head of this leader warp
  if (hg >= kGroup) return;
  if (!__all_sync(0xffffffffu, mbar_wait_cluster(&inbox.bar, 0))) {
    if (lane == 0) set_error(err, kErrTimeout);
    return;
  }
  const int base = warp * S;                  // its parts: slots base .. base + S - 1
  const float2 mlp = lane < S ? inbox.ml[base + lane] : make_float2(-INFINITY, 0.f);
  float mx = mlp.x;
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float w = mlp.x == -INFINITY ? 0.f : fast_exp2(mlp.x - mx);
  float lw = w * mlp.y;
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

}  // namespace pkv_decode

#endif  // PKV_DECODE_DEVICE_CUH
