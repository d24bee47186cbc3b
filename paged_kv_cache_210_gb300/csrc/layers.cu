// Several consecutive layers of the fused append-then-attend step in one
// persistent launch (pkv_append_attend_layers, declared in include/pkv.h).
// A decode step runs the attention of all 16 layers for each new token [6
// Hours of YouTube and 85 handtyped pages of notes on LLM Inference - Start
// here, README feature list: the fixed 16-layer Llama 3.2 1B layout and the
// batched decode bullet]; this kernel keeps each sequence's layer order with
// device-side waits instead of one launch per layer.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "pkv.h"
#include "decode_device.cuh"
#include "device_common.cuh"
#include "pool_internal.h"

using namespace pkv_dev;
using namespace pkv_decode;

namespace {

// ---------------------------------------------------------------- layer stack
// Consecutive layers of the fused step in one launch: the grid of the wide
// cluster shape (S blocks of 4 warps per (sequence, kv head), 2 page stages
// per warp, merged through distributed shared memory), made persistent. Each block loops over the
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
  const int32_t* tables;      // block tables from the launch's first layer on:
                              // [layer][max_batch][table_stride]
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

struct alignas(1024) LayersSmem {
  DecodeSmem<kClusterWarps, kWideStages> blk;
  ClusterInbox inbox;
  int ptab[kLayerTab];        // physical page of (layer j, page o of the block's range): j * span + o
  int flag;                   // thread 0's wait verdict for the block
};
// + 1 KiB: the kernel rounds the dynamic shared memory base up to 1024 bytes
constexpr size_t kLayersSmemBytes = sizeof(LayersSmem) + 1024;

static_assert(4 * (kLayersSmemBytes + 1024) <= kSmemPerSm, "4 multi-layer blocks per SM");

// Bounded wait until *ctr >= target (acquire, GPU scope): false after about
// two seconds.
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

// tmap_k, tmap_v: the K and V pools as the copy engine's 3-D tensors (dim,
// kv head x 16 + token, page), boxes of one (page, kv head) tile.
__global__ void __launch_bounds__(kClusterWarps * 32, 4)
decode_layers_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const LayersParams prm) {
  constexpr int kWarps = kClusterWarps;
  constexpr int kStages = kWideStages;
  constexpr int kThreads = kWarps * 32;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled tiles need a 1024-byte aligned base (the launch adds 1 KiB)
  LayersSmem& ls = *reinterpret_cast<LayersSmem*>(
      smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  auto& sm = ls.blk;

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
  PageRing<kStages>& ws = sm.warp[warp];
  unsigned long long* bars = sm.bar[warp];
  // this warp's pages of the range: warp, warp + 4, ...; its items run over
  // the layers: item k is page i = k % mine of layer j = k / mine
  const int mine = warp < span ? (span - warp + kWarps - 1) / kWarps : 0;
  const int total = mine * J;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (warp == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
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
  // Copy engine: item k into `stage`, whole 16-row tiles (rows past the
  // sequence are masked or zeroed after they land), K by lane 0 and V by
  // lane 1 in one instruction. A last page whose only row is the appended
  // one is not copied: that row comes from k/v after the wait.
  auto issue_copy = [&](int k, int stage) {
    if (lane > 1) return;
    const int lp = page_begin + warp + kWarps * (k % mine);
    const int phys = phys_of(k);
    const bool ok = phys >= 0 && phys < prm.num_pages;
    const bool rows = !(lp == last_page && new_slot == 0);
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
  // ... written to the pool now, and into its stage tile once that tile has landed
  auto store_new_row = [&](int phys, uint4 val) {
    if (lane >= 16 || phys < 0 || phys >= prm.num_pages) return;
    const bool is_v = lane >= 8;
    const int c = lane & 7;
    uint16_t* pool = is_v ? prm.v_pool : prm.k_pool;
    *reinterpret_cast<uint4*>(pool + ((static_cast<size_t>(phys) * kHkv + kvh) * kPage +
                                      new_slot) * kDim + c * 8) = val;
  };
  uint4 new_val = make_uint4(0u, 0u, 0u, 0u);
  // A landed stage holding fewer than 16 live tokens or the appended row: V
  // rows at or past `live` zeroed, the appended row into its slot; the
  // stores reach the copy engine's view before the stage is refilled.
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

  int issued = min(total, kStages);
  for (int k = 0; k < issued; ++k) issue_copy(k, k);

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
    if (place_now) new_val = load_new_row(j);
    uint32_t qh[8], ql[8];
    load_q_mma<false>(prm.q + ((static_cast<size_t>(j) * prm.batch + b) * kHq + kvh * kGroup) *
                                  kDim,
                      lane, nullptr, nullptr, qh, ql);
    if (place_now) store_new_row(phys_of(item_new), new_val);

    MmaState st;
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
        if (kn == item_new) {
          new_val = load_new_row(j);
          store_new_row(phys_of(kn), new_val);
        }
        issued = kn + 1;
      }
    };
    for (int i = 0; i < mine && !broken; ++i, ++k) {
      // one verdict per warp: the page work below shuffles across all lanes
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[k % kStages], (k / kStages) & 1))) {
        broken = true;
        if (lane == 0) set_error(prm.err, kErrTimeout);
        break;
      }
      consumed = k + 1;
      const int live = live_of(k, i);
      if (live < kPage || k == item_new) patch_stage(k % kStages, live, k == item_new && live > 0);
      attend_page_mma<false>(ws.k[k % kStages], ws.v[k % kStages], live, lane, qh, ql, st);
      __syncwarp();   // every lane's reads of the stage are done before it is refilled
      refill(k);
    }
    lost |= broken;
    k = (j + 1) * mine;      // the next layer's first item (also after a break)
    if (lost) {
      st.m_run = -INFINITY;
      st.l_run = 0.f;
    }
    float* out_kv = prm.out + ((static_cast<size_t>(j) * prm.batch + b) * kHq + kvh * kGroup) * kDim;
    float M, L;
    float2 O;
    block_merge_mma<kWarps>(sm, st, warp, lane, M, L, O);
    if (n_splits > 1) {
      cluster_merge(ls.inbox, M, L, O, warp, lane, out_kv, true);
    } else {
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
    for (int kk = consumed; kk < issued; ++kk) mbar_wait(&bars[kk % kStages], (kk / kStages) & 1);
  }
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
  if (!pkv_aligned16(q) || !pkv_aligned16(k) || !pkv_aligned16(v) || !pkv_aligned16(k_pool) ||
      !pkv_aligned16(v_pool) || !pkv_aligned16(block_tables) || !pkv_aligned16(seq_lens) ||
      !pkv_aligned16(out))
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
      const pkv_status st = pkv_append_attend(pool, layer_begin + j, q16 + j * q_layer,
                                              k16 + j * kv_layer, v16 + j * kv_layer, k_pool,
                                              v_pool, block_tables, seq_lens, out + j * q_layer,
                                              batch, 0, stream);
      if (st != PKV_OK) return st;
    }
    return PKV_OK;
  }

  CUtensorMap tk, tv;
  if (!pkv_pool_tensor_map(k_pool, c.num_pages, &tk) ||
      !pkv_pool_tensor_map(v_pool, c.num_pages, &tv))
    return PKV_ERR_CUDA;
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
    cfg.dynamicSmemBytes = kLayersSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = S;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_layers_kernel, tk, tv, prm) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return pkv_check_launch();
}

}  // namespace

bool pkv_layers_setup(pkv_pool* pool) {
  bool ok = cudaFuncSetAttribute(decode_layers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kLayersSmemBytes)) == cudaSuccess;
  ok = ok && cudaFuncSetAttribute(decode_layers_kernel,
                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
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
    probe.dynamicSmemBytes = kLayersSmemBytes;
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
  return ok;
}

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

}  // extern "C"
