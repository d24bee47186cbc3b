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
//    ring of page stages in shared memory, filled by the tensor copy engine
//    (cp.async.bulk.tensor with the 128-byte swizzle, the K and V tiles of a
//    page in one instruction, completion counted on an mbarrier), so bytes in
//    flight do not depend on registers and warps never wait on each other
//    inside the page loop;
//  * the page math runs on the tensor cores, warp-wide (mma.sync m16n8k16,
//    BF16 in, FP32 accumulate): S = Q K^T with the group's 4 heads as the
//    rows (padded to 16), then a base-2 online softmax in registers whose
//    max moves only when a head's max grows by more than 2^8, then O += P V
//    with P as a BF16 high plus low part; per page and lane about a quarter
//    of the instructions the same work takes in FP32 FMAs, which leaves the
//    step bound by HBM rather than by issue;
//  * warps merge in shared memory; splits merge in the same launch, in a
//    cluster through st.async stores into the head leaders' shared memory,
//    or through global partials and a ticket: every split block writes its
//    (o, m, l) partial and takes a ticket, and the last to arrive merges (no
//    spinning).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "decode_device.cuh"
#include "device_common.cuh"
#include "pool_internal.h"

using namespace pkv_dev;
using namespace pkv_decode;

namespace {

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

// ---------------------------------------------------------------- decode
// kCluster: the splits of one (sequence, kv head) form one thread-block
// cluster (gridDim.x == cluster size) and merge through distributed shared
// memory; otherwise splits merge through global partials and a ticket.
// tmap_k, tmap_v: the K and V pools as 3-D tensors (dims, kv head x token,
// page), boxes of one (page, kv head) tile.
template <bool kFused, bool kCluster, int kWarps, int kStages, bool kRope>
__global__ void __launch_bounds__(kWarps * 32, kCluster && kStages == kNarrowStages ? 3 : 16 / kWarps)
decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const DecodeParams prm) {
  constexpr int kThreads = kWarps * 32;
  using Smem = DecodeSmem<kWarps, kStages>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled tiles need a 1024-byte aligned base (the launch adds 1 KiB)
  uint8_t* smem_base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem& sm = *reinterpret_cast<Smem*>(smem_base);

  int split = blockIdx.x;
  const int kvh = blockIdx.y;
  int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A block past the first wave of resident blocks starts only once a slot
  // has been left, so there is nothing to prefetch ahead of the wait: it
  // waits and lets the next launch start right away, before its own
  // prologue, so the launch's trigger does not wait on the prologues of its
  // last blocks (the wait still comes first in every block).
  // (Cluster launches fit one wave.)
  const bool late =
      !kCluster && prm.resident_blocks > 0 &&
      static_cast<long long>(blockIdx.x) +
              gridDim.x * (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z) >=
          prm.resident_blocks;
  if (late) {
    pdl_wait();
    pdl_launch_dependents();
  }
  // Ticket plans: ranges of chunk_pages pages; a longest-first launch has
  // the grid (1, kv heads, units) and sizes its ranges to the batch.
  int range_pages = prm.chunk_pages;
  if (!kCluster && prm.longest_first) {
    const int u = static_cast<int>(blockIdx.z);
    b = prm.range_div == 0
            ? longest_first_unit<kWarps, true>(u, prm.batch, prm.seq_lens, prm.table_stride,
                                               prm.chunk_pages, 0, sm, split, range_pages)
            : longest_first_unit<kWarps, false>(u, prm.batch, prm.seq_lens, prm.table_stride,
                                                prm.chunk_pages, prm.range_div, sm, split,
                                                range_pages);
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
                                       : range_pages;
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

  PageRing<kStages>& ws = sm.warp[warp];
  unsigned long long* bars = sm.bar[warp];
  AsyncInbox& inbox = *reinterpret_cast<AsyncInbox*>(smem_base + sizeof(Smem));
  // pages of this warp: page_begin + warp + 4 i
  const int mine = page_begin + warp < page_end
                       ? (page_end - (page_begin + warp) + kWarps - 1) / kWarps
                       : 0;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (warp == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
  }
  // the leaders' inbox barriers are armed before any part is sent (every
  // block of the cluster takes this branch: it depends on the length only)
  if (kCluster && n_splits > 1) async_inbox_setup(inbox);
  __syncthreads();   // the block-table row is in shared memory

  // Physical page of this warp's i-th page (i < mine <= 32) sits in lane i:
  // one parallel read of the block table instead of one per page.
  int my_phys = -1;
  if (lane < mine) my_phys = sm.pages[page_begin + warp + kWarps * lane];

  // Copy engine: the (page, kv head) tiles of this warp's i-th page into
  // stage i % kStages, whole 16-row tiles (rows past the sequence are masked
  // or zeroed after they land). A copy instruction costs its warp a few
  // hundred cycles whatever its size, so the K and V copies go out together
  // from lanes 0 and 1. A page whose only row is the appended one (fused
  // step) is not copied: that row comes from k/v.
  auto issue_copy = [&](int i, int stage, int phys) {
    if (lane > 1) return;
    const int lp = page_begin + warp + kWarps * i;
    const bool ok = phys >= 0 && phys < prm.num_pages;
    const bool rows = !(kFused && lp == last_page && new_slot == 0);
    if (!ok && lane == 0) set_error(prm.err, kErrPage);
    if (ok && rows) {
      if (lane == 0) mbar_arrive_expect_tx(&bars[stage], 2 * kTileBytes);
      __syncwarp(0x3u);   // the expected bytes are set before either copy can land
      tma_load_tile(lane == 0 ? ws.k[stage] : ws.v[stage], lane == 0 ? &tmap_k : &tmap_v,
                    kvh * kPage, phys, &bars[stage]);
    } else if (lane == 0) {
      mbar_arrive(&bars[stage]);
    }
  };
  // Rotary angles of the position len - 1 for pairs 8 (lane & 3) .. + 7: the
  // key rotation of the appended row uses them in lanes 0..7 (chunk c = lane,
  // c & 3 == lane & 3). The tables are constant inputs, read ahead of the
  // wait for the previous launch.
  float rcs[8], rsn[8];
  if (kRope) {
    load_angles(prm.rope_cos + static_cast<size_t>(len - 1) * (kDim / 2), lane & 3, rcs);
    load_angles(prm.rope_sin + static_cast<size_t>(len - 1) * (kDim / 2), lane & 3, rsn);
  }

  // Fused step: the warp whose i_new-th page is the sequence's last page
  // writes the appended token's K/V row to the pool, and into the stage tile
  // once that tile has landed. Lanes 0..15 load one 16-byte chunk each (K for
  // lanes 0..7, V for 8..15), only after the wait: k/v may come from the
  // previous kernel.
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
  // The loaded chunk `val` of the appended row into the pool (page phys);
  // with rotary tables lanes 0..7 rotate the key first, the partner chunk
  // coming from lane ^ 4. Returns the chunk as stored. Called by the whole warp.
  auto store_new_row = [&](int phys, uint4 val, bool preloaded) {
    const bool is_v = lane >= 8;
    const int c = lane & 7;
    if (kRope) {
      const uint4 partner = shfl_xor_uint4(val, 4);
      if (lane < 8) {
        if (preloaded) {
          val = rope_key_chunk(val, partner, c >= 4, rcs, rsn);
        } else {   // in the page loop the angles are read again (from cache)
          float cs[8], sn[8];
          load_angles(prm.rope_cos + static_cast<size_t>(len - 1) * (kDim / 2), c & 3, cs);
          load_angles(prm.rope_sin + static_cast<size_t>(len - 1) * (kDim / 2), c & 3, sn);
          val = rope_key_chunk(val, partner, c >= 4, cs, sn);
        }
      }
    }
    if (lane < 16 && phys >= 0 && phys < prm.num_pages) {
      uint16_t* pool = is_v ? prm.v_pool : prm.k_pool;
      *reinterpret_cast<uint4*>(pool + ((static_cast<size_t>(phys) * kHkv + kvh) * kPage +
                                        new_slot) * kDim + c * 8) = val;
    }
    return val;
  };

  // Prefetch: the first n_prefetch pages' tiles in one copy instruction,
  // lane 2i (K) and 2i + 1 (V) serving page i, so the warp pays one copy
  // round instead of n_prefetch before its first page can land; the rules
  // are issue_copy's. The unfused kernel defers the page holding the
  // appended slot, which the preceding append kernel may still be writing.
  const int n_prefetch = min(mine, kStages);
  int deferred = -1;
  {
    const int i = lane >> 1;
    const int phys = __shfl_sync(0xffffffffu, my_phys, i);
    const int lp = page_begin + warp + kWarps * i;
    const bool serves = i < n_prefetch && (kFused || lp != last_page);
    const bool ok = phys >= 0 && phys < prm.num_pages;
    const bool rows = !(kFused && lp == last_page && new_slot == 0);
    if (serves && (lane & 1) == 0) {
      if (!ok) set_error(prm.err, kErrPage);
      if (ok && rows) {
        mbar_arrive_expect_tx(&bars[i], 2 * kTileBytes);
      } else {
        mbar_arrive(&bars[i]);
      }
    }
    __syncwarp();   // every stage's expected bytes are set before any copy can land
    if (serves && ok && rows)
      tma_load_tile((lane & 1) == 0 ? ws.k[i] : ws.v[i], (lane & 1) == 0 ? &tmap_k : &tmap_v,
                    kvh * kPage, phys, &bars[i]);
    if (!kFused)
      for (int j = 0; j < n_prefetch; ++j)
        if (page_begin + warp + kWarps * j == last_page) deferred = j;
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
  if (!late) {
    pdl_wait();
    // The next launch may start once every block of this one has passed
    // this point, so its blocks take the slots this launch frees and
    // prefetch their pages while this launch's last blocks run (no block of
    // this launch is still waiting for a slot then: each has started). The
    // trigger comes after the wait: the next launch's pre-wait reads then
    // start only once every launch before this one has completed, so only
    // the launch immediately before it can still be writing. (Measured on
    // GB300 against a trigger after the page loop for launches of several
    // waves: batch-256 ragged step 6508 vs 6404 GB/s, batch-64 mix 4175 vs
    // 3878.)
    pdl_launch_dependents();
  }
  // the new row's load goes out before q's, so the two latencies overlap
  const bool new_in_prologue = i_new >= 0 && i_new < n_prefetch;
  uint4 new_val = make_uint4(0u, 0u, 0u, 0u);
  if (new_in_prologue) new_val = load_new_row();
  if (deferred >= 0) issue_copy(deferred, deferred, __shfl_sync(0xffffffffu, my_phys, deferred));
  int issued = n_prefetch;

  uint32_t qh[8], ql[8];
  load_q_mma<kRope>(prm.q + (static_cast<size_t>(b) * kHq + kvh * kGroup) * kDim, lane,
                    kRope ? prm.rope_cos + static_cast<size_t>(len - 1) * (kDim / 2) : nullptr,
                    kRope ? prm.rope_sin + static_cast<size_t>(len - 1) * (kDim / 2) : nullptr,
                    qh, ql);
  if (new_in_prologue)
    new_val = store_new_row(__shfl_sync(0xffffffffu, my_phys, i_new), new_val, true);

  MmaState st;
  st.reset();

  bool timed_out = false;
  int consumed = 0;
  // tokens of the warp's i-th page that count (0 for a page id out of range)
  auto live_of = [&](int i, int phys) {
    const int lp = page_begin + warp + kWarps * i;
    const int valid = lp == last_page ? len - lp * kPage : kPage;
    return phys >= 0 && phys < prm.num_pages ? valid : 0;
  };
  // A landed stage holding fewer than 16 live tokens or the appended row: V
  // rows at or past `live` are zeroed (p = 0 times them must stay 0 whatever
  // the pool held there), and the appended row goes into its slot (over
  // what the copy brought, which may predate this step's write). The stores
  // reach the copy engine's view (async proxy) before the stage is refilled.
  auto patch_stage = [&](int stage, int live, bool with_new) {
    uint8_t* vt = ws.v[stage];
    for (int idx = live * 8 + lane; idx < kPage * 8; idx += 32)
      *reinterpret_cast<uint4*>(vt + (idx >> 3) * kRowBytes + (idx & 7) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    if (with_new && lane < 16) {
      uint8_t* t = lane >= 8 ? ws.v[stage] : ws.k[stage];
      const int c = lane & 7;
      *reinterpret_cast<uint4*>(t + new_slot * kRowBytes + ((c ^ (new_slot & 7)) << 4)) = new_val;
    }
    fence_proxy_async_smem();
    __syncwarp();
  };
  // after page i is consumed: the copy of page i + kStages into its stage
  auto refill = [&](int i, int stage) {
    if (i + kStages < mine) {
      const int next_phys = __shfl_sync(0xffffffffu, my_phys, i + kStages);
      issue_copy(i + kStages, stage, next_phys);
      if (i + kStages == i_new) new_val = store_new_row(next_phys, load_new_row(), false);
      issued = i + kStages + 1;
    }
  };
  int stage = 0;            // i % kStages
  uint32_t phase = 0;       // (i / kStages) & 1
  for (int i = 0; i < mine; ++i) {
    const int phys = __shfl_sync(0xffffffffu, my_phys, i);
    // one verdict per warp: the page work below shuffles across all lanes
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[stage], phase))) {
      timed_out = true;
      break;
    }
    consumed = i + 1;
    const int live = live_of(i, phys);
    if (live < kPage || i == i_new) patch_stage(stage, live, i == i_new && live > 0);
    attend_page_mma<kRope>(ws.k[stage], ws.v[stage], live, lane, qh, ql, st);
    __syncwarp();   // every lane's reads of the stage are done before it is refilled
    refill(i, stage);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  if (timed_out) {
    // let this warp's copies still in flight land before the block exits
    // (each wait bounded again)
    for (int j = consumed; j < issued; ++j) mbar_wait(&bars[j % kStages], (j / kStages) & 1);
  }

  // ---- block merge
  if (timed_out) {
    if (lane == 0) set_error(prm.err, kErrTimeout);
    st.m_run = -INFINITY;
    st.l_run = 0.f;
  }
  float M, L;
  float2 O;
  block_merge_mma<kWarps>(sm, st, warp, lane, M, L, O);
  if constexpr (kCluster) {
    if (n_splits > 1) {
      cluster_merge_async(inbox, M, L, O, warp, lane,
                          prm.out + (static_cast<size_t>(b) * kHq + kvh * kGroup) * kDim,
                          prm.err);
      return;
    }
  }

  // every ticket-mode block; a cluster whose sequence has a single split
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

}  // namespace

// ================================================================= host side

namespace {

// The three kernel shapes (the cluster kernels add the leaders' inbox).
enum Shape { kTicketShape = 0, kNarrowShape = 1, kWideShape = 2 };
template <bool kFused, bool kRope = false>
constexpr auto ticket_kernel = decode_kernel<kFused, false, kTicketWarps, kTicketStages, kRope>;
template <bool kFused, bool kRope = false>
constexpr auto narrow_kernel = decode_kernel<kFused, true, kClusterWarps, kNarrowStages, kRope>;
template <bool kFused, bool kRope = false>
constexpr auto wide_kernel = decode_kernel<kFused, true, kWideWarps, kWideStages, kRope>;

// + 1 KiB: the kernel rounds the dynamic shared memory base up to 1024 bytes
size_t smem_bytes(Shape shape) {
  switch (shape) {
    case kNarrowShape: return sizeof(NarrowDecodeSmem) + sizeof(AsyncInbox) + 1024;
    case kWideShape: return sizeof(WideDecodeSmem) + sizeof(AsyncInbox) + 1024;
    default: return sizeof(TicketDecodeSmem) + 1024;
  }
}

// ---------------------------------------------------------------- pool tensor maps
// The K or V pool of num_pages pages as a 3-D BF16 tensor for the copy
// engine: (dim, kv head x 16 + token, page), rows of 128 B, pages of 16 KiB;
// a box is one (page, kv head) tile of 16 x 64, written with the 128-byte
// swizzle. Encoding is host work only; the last maps are kept per base
// address (the map depends on nothing else).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

}  // namespace

bool pkv_pool_tensor_map(const void* pool, int num_pages, CUtensorMap* map) {
  constexpr int kCacheSlots = 64;
  struct Slot {
    const void* base;
    int num_pages;
    CUtensorMap map;
  };
  static std::mutex lock;
  static Slot cache[kCacheSlots] = {};
  const size_t slot = (reinterpret_cast<uintptr_t>(pool) >> 8) % kCacheSlots;
  {
    std::lock_guard<std::mutex> guard(lock);
    if (cache[slot].base == pool && cache[slot].num_pages == num_pages) {
      *map = cache[slot].map;
      return true;
    }
  }
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {kDim, static_cast<cuuint64_t>(kHkv) * kPage,
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[2] = {kRowBytes, static_cast<cuuint64_t>(kHkv) * kPage * kRowBytes};
  const cuuint32_t box[3] = {kDim, kPage, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  if (fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box,
         elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> guard(lock);
  cache[slot].base = pool;
  cache[slot].num_pages = num_pages;
  cache[slot].map = *map;
  return true;
}

namespace {

int block_threads(Shape shape) {
  return 32 * (shape == kTicketShape ? kTicketWarps
               : shape == kWideShape ? kWideWarps
                                     : kClusterWarps);
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


static_assert(kTicketShape == PKV_SHAPE_TICKET && kNarrowShape == PKV_SHAPE_NARROW &&
                  kWideShape == PKV_SHAPE_WIDE,
              "the plan's shape codes are the kernel shapes");

// Ticket plans when the caller leaves the choice to the library: ranges of
// at least kLeastRangePages pages (and few enough per sequence for the
// partial rows). When the blocks of full-length sequences would not fit one
// wave of resident ticket blocks, the launch takes (sequence, range) units
// longest sequence first. Up to kSplitWaves waves of sequences, it sizes the
// ranges to the batch it finds: ceil(T / range_div) pages, T the batch's
// pages per kv head, range_div = resident blocks x 3 / 40 (rounded), i.e.
// about 1.65 times the pages per resident block slot (8 kv heads);
// sequences longer than that split, the rest run whole. Past that many
// sequences every sequence runs whole. Measured on a 152-SM GB300 (GB/s per
// 16-layer fused step; the log-uniform and uniform batches of 64 and 256
// are the configured workloads). Ranges of one fixed size (dependents
// triggered after the page loop):
//   log-uniform b48:  32 3798, 40 3827, 48 3604, 64 3290, 128 2358
//   log-uniform b64:  32 3562, 40 3803, 48 3990, 56 3760, 64 3500, 128 2687
//   log-uniform b96:  32 3495, 48 3901, 64 4220, 96 3502, 128 3123
//   log-uniform b128: 48 4163, 64 4534, 96 4563, 128 4228
//   log-uniform b256: 64 5008, 96 5164, 128 5448
//   uniform b64:      48 4541, 64 4978, 96 5142, 128 4790
//   uniform b256:     64 6080, 96 6303, 128 6329
//   full-length b40:  48 4995, 96 4497, 128 5322; b64: 64 5705, 128 6241
// Ranges sized to the batch, range_div 38 / 42 / 46 / 50 (dependents
// triggered after the wait):
//   log-uniform b48 3939 / 4048 / 4292 / 4279; b64 3950 / 4214 / 4239 / 4039;
//   b96 4369 / 4393 / 4227 / 4084; b128 4695 / 4815 / 4708 / 4613;
//   uniform b64 5046 / 5233 / 5469 / 5443; b128 6494 / 6481 / 6465 / 6450;
//   full-length b33 4833 / 5078 / 5315 / 5466, b36 4865 / 5202 / 5347 / 5578,
//   b40 5357 / 4667 / 4693 / 4491
// (a full-length batch just short of range_div sequences splits each into
// a long and a short range). Splitting into even ranges (round(p / r) of
// them) lost 5-15 % on the mixes. A grid with a fixed count of blocks per
// (sequence, kv head), most of them empty for short sequences, cost up to
// 6 %, hence the units; spare units cost 3-5 % at 192 and 256 sequences
// (log-uniform b192 4944 vs 5087 whole, b256 5299 vs 5578), hence whole
// sequences past kSplitWaves waves.
constexpr int kLeastRangePages = 16;
constexpr int kSplitWaves = 2;

// The launch plan for a batch. Cluster plans when the library chooses: the
// split count S (16, 12, 8, 4, 2) and the block shape, from sweeps on a
// 152-SM GB300 with full-length sequences (GB/s per 16-layer step; the
// first sweep with the barrier-based cluster merge, the second with the
// asynchronous one):
//   batch 2:  narrow S = 16 (256 blocks) 1522; wide S = 16 1453; S = 8 1337;
//             async: narrow S = 12 (192) 1720, S = 16 1574, S = 14 1495,
//             S = 10 1565; wide S = 16 1677;
//   batch 4:  narrow S = 8 (256) 2304; narrow S = 16 1404; wide S = 8 2015;
//             async: narrow S = 8 2374, S = 7 2216, S = 6 2282; wide S = 16 1950;
//   batch 8:  wide S = 8 (512) 3462; narrow S = 4 (256) 2680; wide S = 16 2016;
//   batch 16: wide S = 4 (512) 4214; narrow S = 2 (256) 3187; wide S = 8 3443;
// and with the page math on the tensor cores:
//   batch 2:  narrow S = 12 1855; wide S = 16 1766;
//   batch 4:  wide S = 8 (256) 2972-2974; narrow S = 8 2627-2630;
//   batch 8:  wide S = 8 (512) 4024; wide S = 4 (256) 3886;
//   batch 16: wide S = 4 (512) 5079; wide S = 2 (256) 4379.
// So: the narrow shape with S = 16 or 12 when the blocks of two consecutive
// launches fit its resident slots at once (the next layer's blocks then
// become resident and prefetch during this one); else the wide shape with
// S = 8 when two consecutive launches fit its slots (batch 3-4); else the
// narrow S = 8 when one launch's blocks take at most 9/16 of its slots (a
// device with fewer wide slots); else the wide
// shape with the largest S <= 8 whose blocks take at most 27/32 of its slots
// (512 of 608); else (large batches) the ticket merge over page ranges.
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
    for (const int s : {16, 12}) {
      if (!p.cluster && usable(s) && 2 * static_cast<long long>(batch) * kHkv * s <= narrow) {
        p.cluster = s;
        p.shape = kNarrowShape;
      }
    }
    if (!p.cluster && usable(8) && 2 * static_cast<long long>(batch) * kHkv * 8 <= wide) {
      p.cluster = 8;
      p.shape = kWideShape;
    }
    if (!p.cluster && usable(8) && 16 * static_cast<long long>(batch) * kHkv * 8 <= 9 * narrow) {
      p.cluster = 8;
      p.shape = kNarrowShape;
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
      p.chunk_pages = std::max(std::min(kLeastRangePages, max_pages),
                               (max_pages + d.max_splits - 1) / d.max_splits);
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
  // more than one wave of ticket-mode blocks: units, longest first
  p.longest_first = (!p.cluster && num_splits == 0 && blocks > resident) ? 1 : 0;
  if (p.longest_first) {
    if (static_cast<long long>(batch) * kHkv > kSplitWaves * resident) {
      // enough sequences to fill the slots whole: no ranges (and no empty units)
      p.chunk_pages = max_pages;
      p.grid_splits = 1;
      p.grid_units = batch;
    } else {
      p.range_div = static_cast<int>(std::max<long long>((resident * 3 + 20) / 40, 1));
      p.grid_units = batch + p.range_div;
    }
  }
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
  if (!pkv_aligned16(q) || !pkv_aligned16(k_pool) || !pkv_aligned16(v_pool) ||
      !pkv_aligned16(block_tables) || !pkv_aligned16(seq_lens) || !pkv_aligned16(out))
    return PKV_ERR_INVALID_ARG;
  if (kFused && (!pkv_aligned16(k) || !pkv_aligned16(v))) return PKV_ERR_INVALID_ARG;
  if (rope && (!rope_cos || !rope_sin || !pkv_aligned16(rope_cos) || !pkv_aligned16(rope_sin)))
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
  prm.range_div = plan.range_div;
  prm.batch = batch;
  prm.resident_blocks = static_cast<long long>(
      plan.shape == kNarrowShape ? pool->cluster_blocks_per_sm
      : plan.shape == kWideShape ? pool->wide_blocks_per_sm
                                 : pool->blocks_per_sm) * pool->num_sms;
  prm.longest_first = plan.longest_first;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = plan.longest_first ? dim3(1, kHkv, plan.grid_units)
                                    : dim3(grid_splits, kHkv, batch);
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
  CUtensorMap tk, tv;
  if (!pkv_pool_tensor_map(k_pool, c.num_pages, &tk) ||
      !pkv_pool_tensor_map(v_pool, c.num_pages, &tv))
    return PKV_ERR_CUDA;
  cudaError_t e;
  if (rope) {
    e = shape == kNarrowShape ? cudaLaunchKernelEx(&cfg, narrow_kernel<kFused, true>, tk, tv, prm)
        : shape == kWideShape ? cudaLaunchKernelEx(&cfg, wide_kernel<kFused, true>, tk, tv, prm)
                              : cudaLaunchKernelEx(&cfg, ticket_kernel<kFused, true>, tk, tv, prm);
  } else {
    e = shape == kNarrowShape ? cudaLaunchKernelEx(&cfg, narrow_kernel<kFused>, tk, tv, prm)
        : shape == kWideShape ? cudaLaunchKernelEx(&cfg, wide_kernel<kFused>, tk, tv, prm)
                              : cudaLaunchKernelEx(&cfg, ticket_kernel<kFused>, tk, tv, prm);
  }
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return pkv_check_launch();
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
  if (!pkv_aligned16(q) || !pkv_aligned16(k_pool) || !pkv_aligned16(v_pool) ||
      !pkv_aligned16(block_tables) || !pkv_aligned16(seq_lens) || !pkv_aligned16(out) ||
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
  prm.range_div = 0;
  prm.batch = batch;
  prm.resident_blocks = 0;   // launched without programmatic dependent launch
  prm.longest_first = 0;
  prm.rope_cos = nullptr;
  prm.rope_sin = nullptr;
  CUtensorMap tk, tv;
  if (!pkv_pool_tensor_map(k_pool, num_pages, &tk) ||
      !pkv_pool_tensor_map(v_pool, num_pages, &tv))
    return PKV_ERR_CUDA;
  ticket_kernel<false><<<dim3(num_splits, kHkv, batch), block_threads(kTicketShape),
                         smem_bytes(kTicketShape),
                         s>>>(tk, tv, prm);
  return pkv_check_launch();
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
  ok = ok && pkv_layers_setup(pool);
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
  if (!pkv_aligned16(k) || !pkv_aligned16(v) || !pkv_aligned16(k_pool) || !pkv_aligned16(v_pool) ||
      !pkv_aligned16(block_tables) || !pkv_aligned16(positions))
    return PKV_ERR_INVALID_ARG;
  if (rope && (!rope_cos || !rope_sin || !pkv_aligned16(rope_cos) || !pkv_aligned16(rope_sin)))
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
  return pkv_check_launch();
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
