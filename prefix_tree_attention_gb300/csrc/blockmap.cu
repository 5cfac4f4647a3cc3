// tree_blockmap_build: 128x128 tile classes and non-empty tile lists.
//
// AReaL Tree Training guide, sections "树构建流程" step 4 and "FlexAttention
// + BlockMask": the mask is consumed in 128-token blocks built from the trie.
// With the interval form of the mask (visible(i, j) <=> j <= i <= reach[j])
// a key block kb needs only mn = min reach and mx = max reach over its keys:
//   qa == kb : PARTIAL iff some key is real (reach[j] >= j), else EMPTY;
//   qa >  kb : EMPTY iff mx < 128 qa; FULL iff mn >= 128 qa + 127.
// Both conditions are monotone in qa, so every column is one run
//   kb (PARTIAL) | kb+1 .. col_full_hi (FULL) | .. col_hi (PARTIAL).
// (Pad keys carry reach = j - 1 < 128 qa, so they never widen a column and a
// block holding one is never FULL, as a pad is never visible.)
//
// Kernels (skip once *dev_status is non-zero):
//  1 cols   one warp per key block: min/max reach -> col_full_hi, col_hi
//  2 rows   one warp per query block: non-empty and FULL counts
//  3 ptrs   one CTA: CSR offsets (exclusive scan), nb and nnz words
//  4 fill   one warp per query block: FULL key blocks ascending, then PARTIAL
//  5 order  rank of every row (by count) and column (by length), descending,
//           ties by index — the heaviest-first schedules of the attention
//           kernels
#include "common.cuh"

namespace tree {
namespace {

constexpr int kWarpsPerCta = 8;

__global__ void k_cols(const int32_t* reach, BlockmapView bm, int32_t* status) {
  if (ld_status(status)) return;
  const int32_t kb = blockIdx.x * kWarpsPerCta + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (kb >= bm.nb) return;
  int32_t mn = INT32_MAX, mx = INT32_MIN, real = 0;
#pragma unroll
  for (int t = 0; t < kBlock / 32; ++t) {
    int32_t j = kb * kBlock + t * 32 + lane;
    int32_t r = reach[j];
    // a key's reach lies in [j - 1, T_pad - 1] (j - 1 for a pad)
    if constexpr (kDebugBuild) dcheck(r >= j - 1 && r < bm.nb * kBlock, status);
    mn = min(mn, r);
    mx = max(mx, r);
    real |= (r >= j);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    real |= __shfl_xor_sync(0xffffffffu, real, o);
  }
  if (lane == 0) {
    int32_t hi = kb - 1, full_hi = kb - 1;
    if (real) {
      hi = mx >> 7;
      int32_t f = mn >= kBlock - 1 ? (mn - (kBlock - 1)) >> 7 : -1;
      full_hi = f > kb ? f : kb;
    }
    bm.col_hi()[kb] = hi;
    bm.col_full_hi()[kb] = full_hi;
  }
}

// Class of tile (qa, kb) from the column runs.
__device__ __forceinline__ int tile_class(const BlockmapView& bm, int32_t qa, int32_t kb) {
  if (kb > qa) return kEmpty;
  const int32_t hi = bm.col_hi()[kb];
  if (hi < qa) return kEmpty;
  if (kb == qa) return kPartial;
  return bm.col_full_hi()[kb] >= qa ? kFull : kPartial;
}

__global__ void k_rows(BlockmapView bm, const int32_t* status) {
  if (ld_status(status)) return;
  const int32_t qa = blockIdx.x * kWarpsPerCta + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (qa >= bm.nb) return;
  int32_t cnt = 0, nfull = 0;
  for (int32_t k0 = 0; k0 <= qa; k0 += 32) {
    int32_t kb = k0 + lane;
    int c = kb <= qa ? tile_class(bm, qa, kb) : kEmpty;
    cnt += __popc(__ballot_sync(0xffffffffu, c != kEmpty));
    nfull += __popc(__ballot_sync(0xffffffffu, c == kFull));
  }
  if (lane == 0) {
    bm.row_cnt()[qa] = cnt;
    bm.row_nfull()[qa] = nfull;
  }
}

__global__ void __launch_bounds__(1024) k_ptrs(BlockmapView bm, const int32_t* status) {
  if (ld_status(status)) return;
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t carry = 0;
  for (int32_t b0 = 0; b0 < bm.nb; b0 += 1024) {
    int32_t b = b0 + threadIdx.x;
    int32_t v = b < bm.nb ? bm.row_cnt()[b] : 0;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int32_t t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;
    }
    __syncthreads();
    int32_t incl = x + (wid > 0 ? warp_tot[wid - 1] : 0);
    if (b < bm.nb) bm.row_ptr()[b] = carry + incl - v;
    carry += warp_tot[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    bm.row_ptr()[bm.nb] = carry;
    bm.base[0] = bm.nb;
    bm.base[1] = carry;
    bm.base[2] = 0;
    bm.base[3] = 0;
  }
}

__global__ void k_fill(BlockmapView bm, const int32_t* status) {
  if (ld_status(status)) return;
  const int32_t qa = blockIdx.x * kWarpsPerCta + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (qa >= bm.nb) return;
  int32_t* out = bm.row_idx() + bm.row_ptr()[qa];
  int32_t nf = 0, np = bm.row_nfull()[qa];
  const unsigned lower = (1u << lane) - 1u;
  for (int32_t k0 = 0; k0 <= qa; k0 += 32) {
    int32_t kb = k0 + lane;
    int c = kb <= qa ? tile_class(bm, qa, kb) : kEmpty;
    unsigned f = __ballot_sync(0xffffffffu, c == kFull);
    unsigned p = __ballot_sync(0xffffffffu, c == kPartial);
    if (c == kFull) out[nf + __popc(f & lower)] = kb;
    if (c == kPartial) out[np + __popc(p & lower)] = kb;
    nf += __popc(f);
    np += __popc(p);
  }
}

__global__ void k_order(BlockmapView bm, const int32_t* status) {
  if (ld_status(status)) return;
  const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  const int32_t nb = bm.nb;
  if (t < nb) {
    const int32_t* cnt = bm.row_cnt();
    const int32_t mine = cnt[t];
    int32_t rank = 0;
    for (int32_t q = 0; q < nb; ++q) {
      int32_t c = cnt[q];
      rank += (c > mine) | ((c == mine) & (q < t));
    }
    bm.row_order()[rank] = t;
  } else if (t < 2 * nb) {
    const int32_t kb = t - nb;
    const int32_t* hi = bm.col_hi();
    const int32_t mine = hi[kb] - kb;
    int32_t rank = 0;
    for (int32_t k = 0; k < nb; ++k) {
      int32_t c = hi[k] - k;
      rank += (c > mine) | ((c == mine) & (k < kb));
    }
    bm.col_order()[rank] = kb;
  }
}

}  // namespace

cudaError_t launch_blockmap_build(const int32_t* key_reach, int32_t T_pad, void* blockmap,
                                  int32_t* status, cudaStream_t s) {
  BlockmapView bm{T_pad / kBlock, static_cast<int32_t*>(blockmap)};
  const int warp_grid = (bm.nb + kWarpsPerCta - 1) / kWarpsPerCta;
  k_cols<<<warp_grid, 32 * kWarpsPerCta, 0, s>>>(key_reach, bm, status);
  k_rows<<<warp_grid, 32 * kWarpsPerCta, 0, s>>>(bm, status);
  k_ptrs<<<1, 1024, 0, s>>>(bm, status);
  k_fill<<<warp_grid, 32 * kWarpsPerCta, 0, s>>>(bm, status);
  k_order<<<(2 * bm.nb + 255) / 256, 256, 0, s>>>(bm, status);
  count_launches(5);
  return cudaGetLastError();
}

}  // namespace tree
