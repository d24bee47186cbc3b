// Internal to libpkv: the pool handle behind pkv_pool_t and the device error
// bits, shared by the decode (pkv.cu) and prefill (prefill.cu) sources.
#ifndef PKV_POOL_INTERNAL_H
#define PKV_POOL_INTERNAL_H

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

struct pkv_pool {
  pkv_pool_config cfg;
  int device;
  int num_sms;
  int blocks_per_sm;           // resident decode blocks per SM (occupancy API)
  int cluster_blocks_per_sm;   // the same for the narrow cluster-merge kernel
  int wide_blocks_per_sm;      // the same for the wide cluster-merge kernel
  int max_cluster;     // largest cluster size (power of two <= 16) the device schedules
  float* part_o;     // [2][max_batch][32][max_splits][64]
  float2* part_ml;   // [2][max_batch][32][max_splits]
  int* tickets;      // [2][max_batch][8]
  int* err;          // sticky error bits (PKV_DEV_ERR_*)
  int* seq_done;     // [max_batch]: layer completions per sequence (multi-layer launch)
  int layer_clusters[5];   // resident clusters of the multi-layer kernel, S = 1, 2, 4, 8, 16
};

// Sticky device error bits; pkv_get_error maps TIMEOUT to
// PKV_ERR_DEVICE_TIMEOUT and the others to PKV_ERR_OUT_OF_RANGE.
enum : int {
  PKV_DEV_ERR_PAGE = 1,       // a page id outside [0, num_pages)
  PKV_DEV_ERR_POSITION = 2,   // a position outside [0, max_seq_len)
  PKV_DEV_ERR_SEQ_LEN = 4,    // a length outside [1, max_seq_len]
  PKV_DEV_ERR_TIMEOUT = 8,    // a bounded wait gave up
};

// Host helpers of the entry points.
inline bool pkv_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pkv_status pkv_check_launch() {
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// pkv.cu: a K or V pool of num_pages pages as the copy engine's 3-D tensor
// map (dim, kv head x 16 + token, page), boxes of one (page, kv head) tile
// with the 128-byte swizzle; false if the driver refuses it.
bool pkv_pool_tensor_map(const void* pool, int num_pages, CUtensorMap* map);

// layers.cu: the multi-layer kernel's attributes and, per cluster size, how
// many of its clusters the device holds at once (pool->layer_clusters).
bool pkv_layers_setup(pkv_pool* pool);

#endif  // PKV_POOL_INTERNAL_H
