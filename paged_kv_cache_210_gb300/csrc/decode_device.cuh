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

#include <cuda.h>
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


// A head leader's inbox (placed after the block's shared memory, cluster kernels only): every
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

// Shared memory of decode_kernel. Each warp's ring of K and V page tiles
// comes first, as the copy engine writes them with the 128-byte swizzle
// (16-byte chunk c of row r at chunk c ^ (r mod 8); every tile is
// 1024-byte aligned, so the rule holds for each tile's own rows), then one
// mbarrier per stage, then the block merge's slots (aliased by the
// longest-first order of the prologue) and the block-table row.
template <int kStages>
struct alignas(1024) PageRing {
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
};

template <int kWarps, int kStages>
struct alignas(1024) DecodeSmem {
  PageRing<kStages> warp[kWarps];
  unsigned long long bar[kWarps][kStages];
  float m[kWarps][kGroup];
  float l[kWarps][kGroup];
  union {
    float acc[kWarps][kGroup][kDim];   // the warps' partial outputs (block merge)
    struct {                           // longest-first order (prologue only)
      int hist[kMaxPages + 1];
      int wsum[kWarps];
      int pick[5];                     // bucket, rank in it, sequence, range, range size
    } order;
  };
  int pages[kMaxPages];      // this sequence's block-table row
  int last;
};

static_assert(sizeof(ClusterInbox) % 16 == 0 && sizeof(AsyncInbox) % 16 == 0,
              "inbox sizes keep 16-byte alignment");
static_assert(sizeof(AsyncInbox) <= sizeof(ClusterInbox) + 16, "the inboxes take the same room");
// residency the kernels are shaped for: 228 KiB of shared memory per SM, 1 KiB
// of it reserved per block; 4 ticket blocks or 3 cluster blocks per SM
constexpr size_t kSmemPerSm = 228 * 1024;
using TicketDecodeSmem = DecodeSmem<kTicketWarps, kTicketStages>;
using NarrowDecodeSmem = DecodeSmem<kClusterWarps, kNarrowStages>;
using WideDecodeSmem = DecodeSmem<kWideWarps, kWideStages>;
static_assert(sizeof(NarrowDecodeSmem) % 16 == 0 && sizeof(WideDecodeSmem) % 16 == 0,
              "the cluster inbox follows DecodeSmem 16-byte aligned");
// + 1 KiB: the dynamic shared memory base is rounded up to 1024 bytes
static_assert(4 * (sizeof(TicketDecodeSmem) + 1024 + 1024) <= kSmemPerSm,
              "4 ticket blocks per SM");
static_assert(3 * (sizeof(NarrowDecodeSmem) + sizeof(AsyncInbox) + 1024 + 1024) <= kSmemPerSm,
              "3 narrow cluster blocks per SM");
static_assert((16 / kWideWarps) * (sizeof(WideDecodeSmem) + sizeof(AsyncInbox) + 1024 + 1024) <=
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
  int range_div;              // longest first: ranges of at least ceil(batch pages / range_div)
  int batch;
  long long resident_blocks;  // resident blocks of the launch's shape (0: no block counts as late)
  int longest_first;          // grid (1, kv heads, units), units longest sequence first
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

// ---------------------------------------------------------------- page computation on tensor cores
// decode_kernel's page math: warp-wide mma.sync m16n8k16 (BF16 operands,
// FP32 accumulate). The rows of every product are the 4 query heads of the
// kv head, padded to 16 with zero rows, so lane L sees head g = L / 4 in its
// row fragments (lanes 16..31: padding rows 4..7) and column pair 2 q, 2 q + 1
// with q = L % 4.
//   scores: S = Q K^T, columns = the page's 16 tokens (two 8-token tiles),
//           contraction over the 64 dims in 4 slices of 16;
//   values: O += P V, columns = the 64 dims (eight 8-dim tiles), contraction
//           over the 16 tokens, P as a BF16 high part (truncated) plus a
//           BF16 low part (two products, ~16 significant bits of P).
// The order of the dims inside a contraction slice does not change the sum
// as long as Q and K agree on it: slice s, lane q takes dims 16 q + 4 s ..
// + 3, so each lane's K fragments come from one 32-byte span of one token
// row (two 16-byte loads, bank-conflict free on the swizzled tile).

constexpr float kRescaleLog2 = 8.f;   // lazy max: a head's p stay <= 2^8

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a2,
                                               uint32_t b0, uint32_t b1) {
  // rows 8..15 of A (a1, a3) are the zero padding
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Copy of one (page, kv head) tile by the tensor copy engine: 16 token rows
// of 64 dims from a pool seen as [page][kv head * 16 + token][dim] (the
// tensor map), with the 128-byte swizzle, completion counted on `bar`.
__device__ __forceinline__ void tma_load_tile(void* dst, const CUtensorMap* map, int row,
                                              int page, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(page),
        "r"(smem_u32(bar))
      : "memory");
}

// The tensor map's descriptor into the cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// This thread's earlier generic-proxy writes to shared memory are ordered
// before later copy-engine (async proxy) accesses to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four transposed 8x8 BF16 matrices from shared memory, one row address per lane.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// Online-softmax state of one warp on tensor cores (head g = lane / 4).
struct MmaState {
  float o[8][4];   // O tile j: [0..1] = O[g][8 j + 2 q, + 1]; [2..3] padding rows (zero)
  float m_run;     // base-2 max the exponentials of head g are taken against
  float l_run;     // this lane's share of head g's sum (its 4 columns)
  __device__ void reset() {
    #pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    m_run = -INFINITY;
    l_run = 0.f;
  }
};

// q of the 4 heads as the A fragments of the score products: lane L < 16
// holds head L / 4, dims 16 (L % 4) .. + 15 as 8 BF16 pairs; slice s uses
// pairs 2 s and 2 s + 1. Lanes 16..31 hold zeros. kRope: q is first rotated
// in FP32 by the angles of its position (cos_row, sin_row: the 32 pair
// angles; dim d < 32 pairs with d + 32, the partner half coming from lane
// L ^ 2) and kept as a BF16 high part in rows 0..3 and a BF16 low part in
// the otherwise empty rows 4..7 (lanes 16..31), so one set of products
// gives both halves' scores; otherwise q is exact in BF16. ql is zero
// (kept for the signature).
template <bool kRope>
__device__ __forceinline__ void load_q_mma(const uint16_t* qrow, int lane, const float* cos_row,
                                           const float* sin_row, uint32_t (&qh)[8],
                                           uint32_t (&ql)[8]) {
  const int g = lane >> 2;
  const int qq = lane & 3;
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
  if (lane < 16) {
    const uint4* src = reinterpret_cast<const uint4*>(qrow + g * kDim + 16 * qq);
    a = __ldg(src);
    b = __ldg(src + 1);
  }
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  if constexpr (!kRope) {
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
      qh[i] = w[i];
      ql[i] = 0u;
    }
  } else {
  float cs[16], sn[16];
  #pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 c4 = __ldg(reinterpret_cast<const float4*>(cos_row + 16 * (qq & 1)) + i);
    const float4 s4 = __ldg(reinterpret_cast<const float4*>(sin_row + 16 * (qq & 1)) + i);
    cs[4 * i] = c4.x; cs[4 * i + 1] = c4.y; cs[4 * i + 2] = c4.z; cs[4 * i + 3] = c4.w;
    sn[4 * i] = s4.x; sn[4 * i + 1] = s4.y; sn[4 * i + 2] = s4.z; sn[4 * i + 3] = s4.w;
  }
  // dims < 32: x' = x cos - y sin; dims >= 32: y' = y cos + x sin
  const float sgn = qq < 2 ? -1.f : 1.f;
  #pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t pw = __shfl_xor_sync(0xffffffffu, w[i], 2);
    const float2 own = bf16x2_to_float2(w[i]);
    const float2 par = bf16x2_to_float2(pw);
    const float r0 = fmaf(own.x, cs[2 * i], sgn * par.x * sn[2 * i]);
    const float r1 = fmaf(own.y, cs[2 * i + 1], sgn * par.y * sn[2 * i + 1]);
    const uint32_t hi = float2_to_bf16x2(r0, r1);
    const float2 hf = bf16x2_to_float2(hi);
    const uint32_t lo = float2_to_bf16x2(r0 - hf.x, r1 - hf.y);
    // the low parts ride in the padding rows 4..7 (lanes 16..31) of the same
    // products; the scores of the two halves are added after them
    const uint32_t lo_of_head = __shfl_xor_sync(0xffffffffu, lo, 16);
    qh[i] = lane < 16 ? hi : lo_of_head;
    ql[i] = 0u;
  }
  }
}

// One page on tensor cores: K tile kt and V tile vt (swizzled, in shared
// memory), `live` valid tokens (the scores of the rest are masked by select;
// V rows at or past `live` must hold finite values, the caller zeroes them).
template <bool kRope>
__device__ __forceinline__ void attend_page_mma(const uint8_t* kt, const uint8_t* vt, int live,
                                                int lane, const uint32_t (&qh)[8],
                                                const uint32_t (&ql)[8], MmaState& st) {
  const int g = lane >> 2;
  const int qq = lane & 3;
  // ---- S = Q K^T: lane q of row group g loads token 8 nt + g, dims 16 q .. + 15
  float s[4];
  #pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint8_t* row = kt + (8 * nt + g) * kRowBytes;
    const uint4 k0 = *reinterpret_cast<const uint4*>(row + (((2 * qq) ^ g) << 4));
    const uint4 k1 = *reinterpret_cast<const uint4*>(row + (((2 * qq + 1) ^ g) << 4));
    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    #pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      mma_bf16_16816(d, qh[2 * sl], qh[2 * sl + 1], kw[2 * sl], kw[2 * sl + 1]);
    }
    if (kRope) {   // rows g and g + 4: the high and low parts of head g's q
      d[0] += __shfl_xor_sync(0xffffffffu, d[0], 16);
      d[1] += __shfl_xor_sync(0xffffffffu, d[1], 16);
    }
    s[2 * nt] = d[0];
    s[2 * nt + 1] = d[1];
  }
  // ---- online softmax of head g over its tokens 2 q, 2 q + 1, 8 + 2 q, 9 + 2 q
  const float c = 1.4426950408889634f * 0.125f;   // log2(e) / sqrt(64)
  float x[4];
  #pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 8 * (i >> 1) + 2 * qq + (i & 1);
    x[i] = t < live ? s[i] * c : -INFINITY;
  }
  float pm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
  // the max used moves only when the head's max grows by more than 2^8
  const bool grow = pm > st.m_run + kRescaleLog2;
  if (__any_sync(0xffffffffu, grow)) {
    const float alpha = grow ? fast_exp2(st.m_run - pm) : 1.f;   // 0 on the first valid page
    if (grow) st.m_run = pm;
    st.l_run *= alpha;
    #pragma unroll
    for (int j = 0; j < 8; ++j) {
      st.o[j][0] *= alpha;
      st.o[j][1] *= alpha;
    }
  }
  const float mu = st.m_run == -INFINITY ? 0.f : st.m_run;
  float p[4];
  #pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - mu);
  st.l_run += (p[0] + p[1]) + (p[2] + p[3]);
  // P as the A fragments of the value products: tokens 2 q, 2 q + 1 (pair 0)
  // and 8 + 2 q, 9 + 2 q (pair 2), high parts truncated, low parts rounded
  uint32_t ah[2], al[2];
  #pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t b0 = __float_as_uint(p[2 * h]), b1 = __float_as_uint(p[2 * h + 1]);
    ah[h] = __byte_perm(b0, b1, 0x7632);
    al[h] = float2_to_bf16x2(p[2 * h] - __uint_as_float(b0 & 0xffff0000u),
                             p[2 * h + 1] - __uint_as_float(b1 & 0xffff0000u));
  }
  // ---- O += P V: lane L addresses row L % 8 of matrix L / 8 (tokens 0..7 or
  // 8..15, dim chunk 2 jj or 2 jj + 1), the transposed loads giving the
  // B fragments of dim tiles 2 jj and 2 jj + 1
  const int mrow = lane & 7;
  const int mat = lane >> 3;
  const uint32_t vrow = smem_u32(vt) + (mrow + 8 * (mat & 1)) * kRowBytes;
  #pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    uint32_t bv[4];
    ldsm_x4_trans(bv, vrow + (((2 * jj + (mat >> 1)) ^ mrow) << 4));
    mma_bf16_16816(st.o[2 * jj], ah[0], ah[1], bv[0], bv[1]);
    mma_bf16_16816(st.o[2 * jj], al[0], al[1], bv[0], bv[1]);
    mma_bf16_16816(st.o[2 * jj + 1], ah[0], ah[1], bv[2], bv[3]);
    mma_bf16_16816(st.o[2 * jj + 1], al[0], al[1], bv[2], bv[3]);
  }
}

// ---------------------------------------------------------------- merges
// The block's warps merged in shared memory: lanes 0..15 of each warp store
// head lane / 4's max, sum (summed over the lane quad) and output tiles;
// then thread t < 128 gets the log-sum-exp state of head g = (t / 32) % 4
// for dims d0 = 2 (t % 32), d0 + 1 (M: max, L: sum, O: unnormalised output).
template <int kWarps, class Smem>
__device__ __forceinline__ void block_merge_mma(Smem& sm, MmaState& st, int warp, int lane,
                                                float& M, float& L, float2& O) {
  st.l_run += __shfl_xor_sync(0xffffffffu, st.l_run, 1);
  st.l_run += __shfl_xor_sync(0xffffffffu, st.l_run, 2);
  if (lane < 16) {
    const int g = lane >> 2;
    const int qq = lane & 3;
    if (qq == 0) {
      sm.m[warp][g] = st.m_run;
      sm.l[warp][g] = st.l_run;
    }
    #pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float2*>(&sm.acc[warp][g][8 * j + 2 * qq]) =
          make_float2(st.o[j][0], st.o[j][1]);
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
// size), after each block merged its warps (M, L, O of thread t < 128: head
// t / 32, dims 2 (t % 32), + 1): threads 0..127 send one (m, l, o) part per
// head straight into the inbox of the head's leader, block g mod S of the
// cluster; every thread arrives on the cluster barrier, and in each leader
// warp w combines the S parts of head rank + w S into out_kv ([4][64], the
// kv head's query heads). A block that leads no head returns after its
// arrival, or, with `wait_always` (blocks that go on to use the cluster
// barrier again), after the wait as well.
__device__ __forceinline__ void cluster_merge(ClusterInbox& inbox, float M, float L, float2 O,
                                              int warp, int lane, float* out_kv,
                                              bool wait_always) {
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

// Cluster merge without a closing cluster barrier: after the block merge
// (M, L, O of thread t < 128: head t / 32, dims 2 (t % 32), + 1), threads
// 0..127 send the block's (o, m, l) part of head t / 32 to the head's leader
// (block g mod S) with st.async stores; a block that leads no head is then
// done. In a leader, warp w waits until the parts of head rank + w S have
// landed and combines them into out_kv.
__device__ __forceinline__ void cluster_merge_async(AsyncInbox& inbox, float M, float L, float2 O,
                                                    int warp, int lane, float* out_kv, int* err) {
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
// Blocks start in linear block order (x fastest). With mixed lengths,
// handing out the longest sequences first shortens the launch's tail (the
// longest-processing-time-first rule), and ranges sized to the batch keep
// the blocks' work even. So a longest-first ticket launch has the grid
// (1, kv heads, units): unit u is the u-th (sequence, range) pair with the
// sequences ordered by page count, most pages first, ties by index, and each
// sequence's ranges in order. The range size comes from the batch itself:
// at least `least_pages`, else ceil(T / range_div) for T the batch's pages
// (per kv head), at most kMaxPages. Since ceil(p / r) < p / r + 1 and
// r >= T / range_div (or r = kMaxPages, one range per sequence), the units
// number fewer than batch + range_div, the units in the grid. Each block finds
// its own unit with a counting sort of the page counts in shared memory:
// O(batch / threads + 128) work and four block barriers, reading only
// seq_lens (which may be read before the wait for the previous launch).
// Pages of a sequence, clamped to [0, max_pages] (an over-long sequence
// counts as max_pages: its blocks only report the length).
__device__ __forceinline__ int page_count(int len, int max_pages) {
  return min(max((len + kPage - 1) / kPage, 0), max_pages);
}

// Returns the sequence of unit u (and its range index and the range size),
// or -1 past the last unit. A sequence of length < 1 has one unit (its block
// reports the length). max_pages <= kMaxPages: the handle's pages per
// sequence. kWhole: ranges of all of max_pages (least_pages >= max_pages),
// every sequence one unit and the grid one unit per sequence, so the pass
// skips the page total and the range arithmetic: every block's first
// copies wait on it.
template <int kWarps, bool kWhole, class Smem>
__device__ int longest_first_unit(int u, int batch, const int32_t* seq_lens, int max_pages,
                                  int least_pages, int range_div, Smem& sm, int& split,
                                  int& range_pages) {
  constexpr int kThreads = kWarps * 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kHeld = 4;                 // page counts kept in registers per thread
  int held[kHeld];
  #pragma unroll
  for (int e = 0; e < kHeld; ++e) {
    const int s = static_cast<int>(threadIdx.x) + e * kThreads;
    held[e] = s < batch ? page_count(seq_lens[s], max_pages) : -1;
  }
  for (int i = threadIdx.x; i <= kMaxPages; i += kThreads) sm.order.hist[i] = 0;
  __syncthreads();
  #pragma unroll
  for (int e = 0; e < kHeld; ++e)
    if (held[e] >= 0) atomicAdd(&sm.order.hist[held[e]], 1);
  for (int s = static_cast<int>(threadIdx.x) + kHeld * kThreads; s < batch; s += kThreads)
    atomicAdd(&sm.order.hist[page_count(seq_lens[s], max_pages)], 1);
  __syncthreads();
  // lane l owns the buckets kMaxPages - 4l - e (e < 4), most pages first;
  // bucket 0 comes last
  if (warp == 0) {
    int cnt[4];
    #pragma unroll
    for (int e = 0; e < 4; ++e) cnt[e] = sm.order.hist[kMaxPages - 4 * lane - e];
    // Split launches: the ranges of a p-page sequence, ceil(p / range), and
    // the unit's rank and range come by float reciprocals (exact here: p +
    // range - 1 < 256, so a true quotient is an integer or at least 1/128
    // above one, and the rank is corrected by one step), not divisions.
    int range = least_pages;
    float inv_range = 0.f;
    if constexpr (!kWhole) {
      int pages = 0;
      #pragma unroll
      for (int e = 0; e < 4; ++e) pages += cnt[e] * (kMaxPages - 4 * lane - e);
      #pragma unroll
      for (int o = 16; o > 0; o >>= 1) pages += __shfl_xor_sync(0xffffffffu, pages, o);
      if (range_div > 0)
        range = max(least_pages, min(kMaxPages, (pages + range_div - 1) / range_div));
      inv_range = __frcp_rn(static_cast<float>(range));
    }
    auto ranges_of = [&](int p) {
      if constexpr (kWhole) return 1;
      return static_cast<int>(static_cast<float>(p + range - 1) * inv_range + (1.f / 256.f));
    };
    int units[4], sum = 0;
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
      units[e] = kWhole ? cnt[e] : cnt[e] * ranges_of(kMaxPages - 4 * lane - e);
      sum += units[e];
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
      if (u >= excl && u < excl + units[e]) {
        const int p = kMaxPages - 4 * lane - e;
        sm.order.pick[0] = p;
        if constexpr (kWhole) {
          sm.order.pick[1] = u - excl;
        } else {
          const int per_seq = ranges_of(p);
          const int off = u - excl;
          int k = off;
          if (per_seq > 1) {
            k = static_cast<int>(__fdividef(static_cast<float>(off), static_cast<float>(per_seq)));
            if (k * per_seq > off) --k;
            if ((k + 1) * per_seq <= off) ++k;
          }
          sm.order.pick[1] = k;
          sm.order.pick[3] = off - k * per_seq;
        }
      }
      excl += units[e];
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      if (u >= total) {   // the sequences without pages, then nothing
        sm.order.pick[0] = 0;
        sm.order.pick[1] = u - total;
        if constexpr (!kWhole) sm.order.pick[3] = 0;
      }
      if constexpr (!kWhole) sm.order.pick[4] = range;
    }
  }
  __syncthreads();
  const int p = sm.order.pick[0];
  const int k = sm.order.pick[1];
  if constexpr (kWhole) {
    split = 0;
    range_pages = least_pages;
  } else {
    split = sm.order.pick[3];
    range_pages = sm.order.pick[4];
    if (p == 0 && k >= sm.order.hist[0]) return -1;   // the same decision in every thread
  }
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
    scan(s, s < batch ? page_count(seq_lens[s], max_pages) : -1);
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
