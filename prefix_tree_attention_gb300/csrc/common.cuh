// Definitions shared by the kernels and the C-ABI layer.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tree_attn.h"

namespace tree {

constexpr int kBlock = 128;   // query/key tile edge; the pages' 128-token block

// Tile classes (also the values stored by the dense expansion in tests).
constexpr int kEmpty = 0, kFull = 1, kPartial = 2;

// Word offsets inside the blockmap buffer (see tree_blockmap_build).
struct BlockmapView {
  int32_t nb;
  int32_t* base;
  __host__ __device__ int32_t* col_full_hi() const { return base + 4; }
  __host__ __device__ int32_t* col_hi() const { return base + 4 + nb; }
  __host__ __device__ int32_t* row_cnt() const { return base + 4 + 2 * nb; }
  __host__ __device__ int32_t* row_nfull() const { return base + 4 + 3 * nb; }
  __host__ __device__ int32_t* row_ptr() const { return base + 4 + 4 * nb; }
  __host__ __device__ int32_t* row_order() const { return base + 5 + 5 * nb; }
  __host__ __device__ int32_t* col_order() const { return base + 5 + 6 * nb; }
  __host__ __device__ int32_t* row_idx() const { return base + 5 + 7 * nb; }
};

__host__ __device__ inline size_t blockmap_words(int64_t nb) {
  return static_cast<size_t>(5 + 7 * nb + nb * (nb + 1) / 2);
}

__device__ __forceinline__ int ld_status(const int32_t* s) {
  return *reinterpret_cast<const volatile int32_t*>(s);
}
__device__ __forceinline__ void set_status(int32_t* s, int code) { atomicCAS(s, 0, code); }

// TREE_DEBUG builds check every index read from device memory before it is
// used (see tree_debug_build).  dcheck(ok, status) is true in a release
// build; in a debug build it records TREE_ERR_BOUNDS when ok is false.
#ifdef TREE_DEBUG
constexpr bool kDebugBuild = true;
#else
constexpr bool kDebugBuild = false;
#endif
__device__ __forceinline__ bool dcheck(bool ok, int32_t* status) {
  if constexpr (kDebugBuild) {
    if (!ok) set_status(status, TREE_ERR_BOUNDS);
    return ok;
  } else {
    return true;
  }
}

// Number of kernels this library has launched in the process (all entry
// points); every launcher adds the launches it queues.
void count_launches(int n);
uint64_t launches_total();

// Launchers (one translation unit each); all return cudaGetLastError().
cudaError_t launch_pack_positions(const int32_t* token_node, int32_t T_pad,
                                  const int32_t* node_entry, const int32_t* node_exit,
                                  int32_t n_nodes, int32_t* position_ids, int32_t* key_reach,
                                  void* workspace, int32_t* dev_status, cudaStream_t s);
size_t pack_positions_workspace_bytes(int32_t T_pad, int32_t n_nodes);

cudaError_t launch_blockmap_build(const int32_t* key_reach, int32_t T_pad, void* blockmap,
                                  int32_t* dev_status, cudaStream_t s);

}  // namespace tree
