// tree_lm_head_logprobs_entropy: the LM head (logits = hidden W^T) fused
// with the row statistics and label log-probabilities of the tree log-prob
// gather, so the [T_pad, V] logits never reach global memory.
//
// AReaL Tree Training guide, section "Log Probability 计算：树结构的特殊处理":
// per packed row the log-sum-exp and entropy of its next-token distribution,
// per token the log-probability of its id under its predicting row pred(j)
// (the last key before j that row j may attend to), computed chunk by chunk
// so that the whole [tokens, vocabulary] logits are never held at once.
// Here the chunk is a 128 x 256 logits tile, which lives only in tensor
// memory.
//
// Kernels (each skips its work once *dev_status is non-zero):
//  1 k_lmh_gemm<false> persistent, one CTA per SM.  A work item is a block
//     of 128 rows and a chunk of kChunkTiles vocabulary tiles of 256
//     columns.  Per vocabulary tile the logits accumulate in TMEM over the
//     hidden size, 64 at a time (tcgen05.mma M = 128, N = 256, K = 16, bf16
//     operands staged by TMA in 128-byte-swizzled shared memory, fp32
//     accumulator).  Two 256-column accumulators alternate, so the epilogue
//     of one tile runs under the MMAs of the next.  The epilogue warps fold
//     each tile into per-row running statistics (max m, s = sum 2^u,
//     t = sum 2^u u, min) and store them at the end of the item as the
//     item's partial for the row (one per 128-column half).  Warp 0 is the
//     TMA producer (a 4-stage ring of 16 KB hidden and 32 KB weight tiles),
//     warp 1 the MMA issuer, warps 2-9 the epilogue.  Items are ordered so
//     that the CTAs running at any moment share 16 row blocks and a few
//     vocabulary chunks: the weight tiles they stream are served from L2.
//  2 k_lmh_combine     one thread per row: the row's partials -> lse,
//     entropy, vocab min / max (pads 0).
//  3 k_lmh_labels      one warp per token: pred(j) by the search of the
//     gather, then the label logit as a fp32 dot product of hidden[pred(j)]
//     and W[token_ids[j]]; logprob = dot - lse[pred(j)].
//
// The gradient with respect to the logits (tree_lm_head_logits_grad), for
// a chunk of rows [row_lo, row_hi) written to a caller's [rows, V] buffer:
//  4 k_lmh_grad_coef   one thread per row: with G the sum of the log-prob
//     gradients of the row's children (the tokens it predicts), E its
//     entropy gradient, every logit's gradient is -p_v (A + E x_v),
//     A = G + E (H - lse); the row's (-lse log2 e, -E, -A).
//  5 k_lmh_gemm<true>  the same GEMM; its epilogue turns each logits tile
//     into its gradient p_v (-A - E x_v), p_v = 2^(x_v log2 e - lse log2 e),
//     as bf16, each warp's 32 x 32 blocks staged in shared memory and
//     written by bulk tensor stores (no statistics).
//  6 k_lmh_grad_labels one warp per row: for each child j, the one-hot term
//     g_lp[j] at the label column, on the label logit recomputed as a fp32
//     dot product, rewritten with one rounding (a row's children carry
//     distinct labels in a trie).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace tree {
namespace {

constexpr int kBM = 128;                 // rows per tile (TMEM lanes)
constexpr int kBN = 256;                 // vocabulary columns per tile
constexpr int kBK = 64;                  // hidden elements per stage (128-byte rows)
constexpr int kStages = 4;
constexpr int kChunkTiles = 8;           // vocabulary tiles per work item
constexpr int kGroupM = 16;              // row blocks sharing weight tiles in L2
constexpr int kGemmThreads = 320;        // producer, MMA, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr uint32_t kATileBytes = kBM * kBK * 2;
constexpr uint32_t kBTileBytes = kBN * kBK * 2;
constexpr int kCombineThreads = 256;
constexpr int kLabelWarps = 8;

constexpr int kOutBox = 32;              // gradient store box: 32 rows x 32 columns (bf16)

struct LmhSmem {
  uint8_t a[kStages][kATileBytes];       // 1024-byte aligned (the struct is)
  uint8_t b[kStages][kBTileBytes];
  uint8_t out[kEpiThreads / 32][kOutBox * kOutBox * 2];   // per epilogue warp, 64-byte swizzled
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

struct LmhParams {
  int32_t T_pad, H, V;
  int32_t mb0;                           // first row block of the work
  int32_t n_mblk, n_ntiles, n_chunks, n_items;
  float4* partial;                       // statistics: [2 * n_chunks][T_pad] (m, s, t, min)
  const float4* coef;                    // gradient: per row of the chunk (nL, nE, nA, pad)
  __nv_bfloat16* grad;                   // gradient: [n_mblk * 128 rows, ldg] bf16
  int64_t ldg;
  int32_t* status;
};

// Work item w -> (row block, vocabulary chunk).  Items run in groups of
// kGroupM row blocks; inside a group, chunk-major: the items resident at
// once cover ~kGroupM row blocks x (#CTAs / kGroupM) chunks.
__device__ __forceinline__ void item_coords(int32_t w, const LmhParams& p, int32_t& mb,
                                            int32_t& chunk) {
  const int32_t per_group = kGroupM * p.n_chunks;
  const int32_t g = w / per_group;
  const int32_t r = w - g * per_group;
  const int32_t gm = min(kGroupM, p.n_mblk - g * kGroupM);   // only the last group is short
  chunk = r / gm;
  mb = g * kGroupM + r % gm;
}

// Fold 64 accumulator columns (x[e] = logit of column col0 + e) into a.
__device__ __forceinline__ void fold64(Acc& a, const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                       int32_t nvalid) {
  if (nvalid >= 64) {
    float mx = -INFINITY, mn = INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      mx = fmaxf(mx, fmaxf(__uint_as_float(r0[e]), __uint_as_float(r1[e])));
      mn = fminf(mn, fminf(__uint_as_float(r0[e]), __uint_as_float(r1[e])));
    }
    a.mn = fminf(a.mn, mn);
    if (mx > a.m) acc_rebase(a, mx);
    const float nmL = -a.m * kLog2e;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      acc_pair(a, nmL, __uint_as_float(r0[e]), __uint_as_float(r0[e + 1]));
      acc_pair(a, nmL, __uint_as_float(r1[e]), __uint_as_float(r1[e + 1]));
    }
  } else if (nvalid > 0) {              // the vocabulary ends inside these columns
#pragma unroll
    for (int e = 0; e < 32; ++e) {       // static indices keep r0 / r1 in registers
      if (e < nvalid) acc_one(a, __uint_as_float(r0[e]));
      if (e + 32 < nvalid) acc_one(a, __uint_as_float(r1[e]));
    }
  }
}

// Gradient of 64 accumulator columns, d = 2^(x log2 e + nL) (nA + nE x),
// packed as 32 bf16 pairs; zeros for a pad row.
__device__ __forceinline__ void grad64(const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                       const float4& cf, uint32_t (&o)[32]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float u0, u1, w0, w1, d0, d1;
    const float x0 = __uint_as_float(r0[e]), x1 = __uint_as_float(r0[e + 1]);
    fma2(u0, u1, x0, x1, kLog2e, kLog2e, cf.x, cf.x);
    fma2(w0, w1, x0, x1, cf.y, cf.y, cf.z, cf.z);
    mul2(d0, d1, ex2f(u0), ex2f(u1), w0, w1);
    o[e >> 1] = pack_bf16x2(d0, d1);
    const float y0 = __uint_as_float(r1[e]), y1 = __uint_as_float(r1[e + 1]);
    fma2(u0, u1, y0, y1, kLog2e, kLog2e, cf.x, cf.x);
    fma2(w0, w1, y0, y1, cf.y, cf.y, cf.z, cf.z);
    mul2(d0, d1, ex2f(u0), ex2f(u1), w0, w1);
    o[16 + (e >> 1)] = pack_bf16x2(d0, d1);
  }
  if (cf.w != 0.f) {
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = 0u;
  }
}

// One 32 x 32 block of the gradient (this warp's 32 rows, 32 columns from
// col) through the warp's staging buffer: each lane writes its row's 64
// bytes in the 64-byte-swizzled layout of the store's tensor map (16-byte
// chunk c of row r at chunk c ^ ((r >> 1) & 3)), then one lane issues the
// bulk tensor store.  The buffer is reused once the previous store has read
// it.  Blocks that start at or past V are skipped.  The block that holds
// column V - 1 with columns past it is written element by element instead:
// the bulk store bounds the row in whole 16-byte units, which would write
// into a row stride's padding past V.
__device__ __forceinline__ void store_block(const CUtensorMap* tm_g, uint8_t* buf,
                                            const uint32_t* w16, int32_t col, int32_t row0,
                                            int32_t V, int lane, __nv_bfloat16* grad,
                                            int64_t ldg) {
  if (col >= V) return;                  // warp-uniform
  if (col + 32 > V) {                    // warp-uniform: the last, partial block
    uint16_t* d2 = reinterpret_cast<uint16_t*>(grad + static_cast<size_t>(row0 + lane) * ldg +
                                               col);
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (col + e < V) d2[e] = static_cast<uint16_t>(w16[e >> 1] >> ((e & 1) * 16));
    return;
  }
  if (lane == 0) bulk_wait_read();
  __syncwarp();
  uint8_t* row = buf + lane * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(w16[4 * c], w16[4 * c + 1], w16[4 * c + 2], w16[4 * c + 3]);
  fence_proxy_async_smem();              // generic-proxy writes -> visible to the bulk copy
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm_g, buf, col, row0);
    bulk_commit();
  }
}

template <bool kGrad>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_lmh_gemm(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
           const __grid_constant__ CUtensorMap tm_g, const LmhParams p) {
  if (ld_status(p.status)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* aligned = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  LmhSmem& sm = *reinterpret_cast<LmhSmem*>(aligned);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  AbortState ab{&sm.abort_flag, p.status};
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], kEpiThreads);
    }
    mbar_init(&sm.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_slot;
  const int32_t ksteps = p.H / kBK;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_h);
      prefetch_tmap(&tm_w);
      uint32_t kc = 0;                   // stages issued so far
      bool ok = true;
      for (int32_t w = blockIdx.x; ok && w < p.n_items; w += gridDim.x) {
        int32_t mb, chunk;
        item_coords(w, p, mb, chunk);
        const int32_t t0 = chunk * kChunkTiles, t1 = min(t0 + kChunkTiles, p.n_ntiles);
        for (int32_t nt = t0; ok && nt < t1; ++nt) {
          for (int32_t ks = 0; ks < ksteps; ++ks) {
            const int s = kc % kStages;
            if (kc >= kStages && !(ok = mbar_wait(&sm.empty[s], (kc / kStages - 1) & 1, ab)))
              break;
            mbar_arrive_expect_tx(&sm.full[s], kATileBytes + kBTileBytes);
            tma_load_2d(sm.a[s], &tm_h, &sm.full[s], ks * kBK, (p.mb0 + mb) * kBM);
            tma_load_2d(sm.b[s], &tm_w, &sm.full[s], ks * kBK, nt * kBN);
            ++kc;
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        for (uint32_t i = kc > kStages ? kc - kStages : 0; i < kc; ++i)
          mbar_drain(&sm.full[i % kStages], (i / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, 0, 0);   // both K-major
      uint32_t kc = 0, tc = 0;
      bool ok = true;
      for (int32_t w = blockIdx.x; ok && w < p.n_items; w += gridDim.x) {
        int32_t mb, chunk;
        item_coords(w, p, mb, chunk);
        const int32_t t0 = chunk * kChunkTiles, t1 = min(t0 + kChunkTiles, p.n_ntiles);
        for (int32_t nt = t0; ok && nt < t1; ++nt, ++tc) {
          const uint32_t buf = tc & 1;
          if (tc >= 2 && !(ok = mbar_wait(&sm.acc_empty[buf], ((tc >> 1) - 1) & 1, ab))) break;
          tc_fence_after();
          const uint32_t acc = tbase + buf * kBN;
          for (int32_t ks = 0; ks < ksteps; ++ks, ++kc) {
            const int s = kc % kStages;
            if (!(ok = mbar_wait(&sm.full[s], (kc / kStages) & 1, ab))) break;
            tc_fence_after();
            const uint32_t abase = smem_u32(sm.a[s]), bbase = smem_u32(sm.b[s]);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_ss(acc, sdesc_sw128(abase + kk * 32, 16, 1024),
                      sdesc_sw128(bbase + kk * 32, 16, 1024), kIdesc, (ks | kk) != 0);
            umma_commit(&sm.empty[s]);   // the stage is free once these MMAs are done
          }
          if (ok) umma_commit(&sm.acc_full[buf]);
        }
      }
      if (!ok) {
        umma_commit(&sm.drain);          // wait for every MMA already issued
        mbar_drain(&sm.drain, 0);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;              // the TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;    // which 128 columns of the 256-column tile
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tc = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; ok && w < p.n_items; w += gridDim.x) {
      int32_t mb, chunk;
      item_coords(w, p, mb, chunk);
      const int32_t t0 = chunk * kChunkTiles, t1 = min(t0 + kChunkTiles, p.n_ntiles);
      const int32_t lrow = mb * kBM + q * 32 + lane;   // row within the work's rows
      Acc a;
      acc_init(a);
      float4 cf = make_float4(0.f, 0.f, 0.f, 1.f);
      if constexpr (kGrad) cf = p.coef[lrow];
      const int32_t brow0 = mb * kBM + q * 32;         // this warp's rows in the gradient
      uint8_t* obuf = sm.out[warp - 2];
      for (int32_t nt = t0; nt < t1; ++nt, ++tc) {
        const uint32_t buf = tc & 1;
        if (!(ok = mbar_wait_warp(&sm.acc_full[buf], (tc >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t taddr = tbase + lane_off + buf * kBN + half * 128;
        const int32_t col0 = nt * kBN + half * 128;
        const int32_t nvalid = p.V - col0;             // columns < V from here
        uint32_t r0[32], r1[32];
        tmem_ld32x2(taddr, taddr + 32, r0, r1);
        if constexpr (kGrad) {
          uint32_t o[32];
          grad64(r0, r1, cf, o);
          store_block(&tm_g, obuf, o, col0, brow0, p.V, lane, p.grad, p.ldg);
          store_block(&tm_g, obuf, o + 16, col0 + 32, brow0, p.V, lane, p.grad, p.ldg);
        } else {
          fold64(a, r0, r1, nvalid);
        }
        tmem_ld32x2(taddr + 64, taddr + 96, r0, r1);
        tc_fence_before();
        mbar_arrive(&sm.acc_empty[buf]); // the accumulator may be overwritten now
        if constexpr (kGrad) {
          uint32_t o[32];
          grad64(r0, r1, cf, o);
          store_block(&tm_g, obuf, o, col0 + 64, brow0, p.V, lane, p.grad, p.ldg);
          store_block(&tm_g, obuf, o + 16, col0 + 96, brow0, p.V, lane, p.grad, p.ldg);
        } else {
          fold64(a, r0, r1, nvalid - 64);
        }
      }
      if (!ok) break;
      if constexpr (!kGrad)
        p.partial[static_cast<size_t>(chunk * 2 + half) * p.T_pad + lrow] =
            make_float4(a.m, a.s0 + a.s1, a.t0 + a.t1, a.mn);
    }
    if constexpr (kGrad) {
      // the gradient stores must have landed before the CTA exits
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

__global__ void __launch_bounds__(kCombineThreads) k_lmh_combine(
    const float4* __restrict__ partial, int32_t n_part, int32_t T_pad,
    const int32_t* __restrict__ reach, float* __restrict__ lse, float* __restrict__ entropy,
    float* __restrict__ vmin, float* __restrict__ vmax, const int32_t* status) {
  if (ld_status(status)) return;
  const int32_t row = blockIdx.x * kCombineThreads + threadIdx.x;
  if (row >= T_pad) return;
  if (reach[row] < row) {               // pad token: no distribution
    lse[row] = 0.f;
    if (entropy) entropy[row] = 0.f;
    if (vmin) vmin[row] = 0.f;
    if (vmax) vmax[row] = 0.f;
    return;
  }
  Acc a;
  acc_init(a);
  for (int32_t i = 0; i < n_part; ++i) {
    const float4 v = partial[static_cast<size_t>(i) * T_pad + row];
    Acc b;
    b.m = v.x;
    b.s0 = v.y;
    b.s1 = 0.f;
    b.t0 = v.z;
    b.t1 = 0.f;
    b.mn = v.w;
    acc_merge(a, b);
  }
  const float s = a.s0 + a.s1, t = a.t0 + a.t1;
  float l = -INFINITY, h = 0.f;
  if (s > 0.f) {
    const float l2s = log2f(s);
    l = fmaf(kLn2, l2s, a.m);
    h = kLn2 * (l2s - t / s);
  }
  lse[row] = l;
  if (entropy) entropy[row] = h;
  if (vmin) vmin[row] = a.mn;
  if (vmax) vmax[row] = a.m;
}

__global__ void __launch_bounds__(kLabelWarps * 32) k_lmh_labels(
    const __nv_bfloat16* __restrict__ hidden, const __nv_bfloat16* __restrict__ weight,
    int32_t H, int32_t V, const int32_t* __restrict__ token_ids,
    const int32_t* __restrict__ reach, BlockmapView bm, const float* __restrict__ lse,
    float* __restrict__ logprob, int32_t* __restrict__ pred_out, int32_t* status) {
  if (ld_status(status)) return;
  const int lane = threadIdx.x & 31;
  const int32_t j = blockIdx.x * kLabelWarps + (threadIdx.x >> 5);   // T_pad % 8 == 0
  int32_t pred = -1;
  if (reach[j] >= j && j > 0)           // warp-uniform: the whole warp serves token j
    pred = reach[j - 1] >= j ? j - 1 : find_pred(j, reach, bm.col_hi(), lane);
  if (pred_out && lane == 0) pred_out[j] = pred;
  if (!logprob) return;
  float out = 0.f;
  if (pred >= 0) {
    const int32_t y = token_ids[j];
    if (y < 0 || y >= V) {
      if (lane == 0) set_status(status, TREE_ERR_MALFORMED_TREE);
      out = __int_as_float(0x7fc00000);
    } else {
      const uint4* hr = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(pred) * H);
      const uint4* wr = reinterpret_cast<const uint4*>(weight + static_cast<size_t>(y) * H);
      float acc0 = 0.f, acc1 = 0.f;
      for (int32_t i = lane; i < H / 8; i += 32) {
        const uint4 x = hr[i], w = wr[i];
        fma2(acc0, acc1, bf_lo(x.x), bf_hi(x.x), bf_lo(w.x), bf_hi(w.x), acc0, acc1);
        fma2(acc0, acc1, bf_lo(x.y), bf_hi(x.y), bf_lo(w.y), bf_hi(w.y), acc0, acc1);
        fma2(acc0, acc1, bf_lo(x.z), bf_hi(x.z), bf_lo(w.z), bf_hi(w.z), acc0, acc1);
        fma2(acc0, acc1, bf_lo(x.w), bf_hi(x.w), bf_lo(w.w), bf_hi(w.w), acc0, acc1);
      }
      float dot = acc0 + acc1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      out = dot - lse[pred];
    }
  }
  if (lane == 0) logprob[j] = out;
}

// The next child of a row after child j (the token after j's subtree), or
// INT32_MAX (and a MALFORMED_TREE status) if key_reach does not advance.
__device__ __forceinline__ int32_t lmh_next_child(int32_t j, const int32_t* __restrict__ reach,
                                                  int32_t* status) {
  const int32_t n = reach[j] + 1;
  if (n <= j) {
    set_status(status, TREE_ERR_MALFORMED_TREE);
    return INT32_MAX;
  }
  return n;
}

__global__ void __launch_bounds__(kCombineThreads) k_lmh_grad_coef(
    int32_t row_lo, int32_t rows, int32_t T_pad, const int32_t* __restrict__ reach,
    const float* __restrict__ lse, const float* __restrict__ entropy,
    const float* __restrict__ g_lp, const float* __restrict__ g_ent, float4* __restrict__ coef,
    int32_t* status) {
  if (ld_status(status)) return;
  const int32_t t = blockIdx.x * kCombineThreads + threadIdx.x;
  if (t >= rows) return;
  const int32_t r = row_lo + t;
  int32_t rr = reach[r];
  if (rr < r) {                          // pad: gradient 0
    coef[t] = make_float4(0.f, 0.f, 0.f, 1.f);
    return;
  }
  if (rr >= T_pad) {
    set_status(status, TREE_ERR_MALFORMED_TREE);
    rr = T_pad - 1;
  }
  float G = 0.f;
  if (g_lp)
    for (int32_t j = r + 1; j <= rr; j = lmh_next_child(j, reach, status)) G += g_lp[j];
  const float L = lse[r];
  const float E = g_ent ? g_ent[r] : 0.f;
  const float H = E != 0.f ? entropy[r] : 0.f;
  coef[t] = make_float4(-L * kLog2e, -E, -(G + E * (H - L)), 0.f);
}

__global__ void __launch_bounds__(kLabelWarps * 32) k_lmh_grad_labels(
    const __nv_bfloat16* __restrict__ hidden, const __nv_bfloat16* __restrict__ weight,
    int32_t H, int32_t V, int32_t T_pad, int32_t row_lo, int32_t rows,
    const int32_t* __restrict__ token_ids, const int32_t* __restrict__ reach,
    const float* __restrict__ g_lp, const float4* __restrict__ coef,
    __nv_bfloat16* __restrict__ grad, int64_t ldg, int32_t* status) {
  if (ld_status(status)) return;
  const int lane = threadIdx.x & 31;
  const int32_t t = blockIdx.x * kLabelWarps + (threadIdx.x >> 5);   // warp-uniform
  if (t >= rows) return;
  const int32_t r = row_lo + t;
  const float4 cf = coef[t];
  if (cf.w != 0.f) return;
  const int32_t rr = min(reach[r], T_pad - 1);
  const uint4* hr = reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(r) * H);
  for (int32_t j = r + 1; j <= rr; j = lmh_next_child(j, reach, status)) {
    const int32_t y = token_ids[j];
    if (y < 0 || y >= V) {
      if (lane == 0) set_status(status, TREE_ERR_MALFORMED_TREE);
      continue;
    }
    const uint4* wr = reinterpret_cast<const uint4*>(weight + static_cast<size_t>(y) * H);
    float acc0 = 0.f, acc1 = 0.f;
    for (int32_t i = lane; i < H / 8; i += 32) {
      const uint4 x = hr[i], w = wr[i];
      fma2(acc0, acc1, bf_lo(x.x), bf_hi(x.x), bf_lo(w.x), bf_hi(w.x), acc0, acc1);
      fma2(acc0, acc1, bf_lo(x.y), bf_hi(x.y), bf_lo(w.y), bf_hi(w.y), acc0, acc1);
      fma2(acc0, acc1, bf_lo(x.z), bf_hi(x.z), bf_lo(w.z), bf_hi(w.z), acc0, acc1);
      fma2(acc0, acc1, bf_lo(x.w), bf_hi(x.w), bf_lo(w.w), bf_hi(w.w), acc0, acc1);
    }
    float x = acc0 + acc1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) {
      const float d = fmaf(ex2f(fmaf(x, kLog2e, cf.x)), fmaf(x, cf.y, cf.z), g_lp[j]);
      grad[static_cast<size_t>(t) * ldg + y] = __float2bfloat16_rn(d);
    }
  }
}

}  // namespace

size_t lm_head_workspace_bytes(int32_t T_pad, int32_t V) {
  const int64_t n_ntiles = (static_cast<int64_t>(V) + kBN - 1) / kBN;
  const int64_t n_chunks = (n_ntiles + kChunkTiles - 1) / kChunkTiles;
  return static_cast<size_t>(2 * n_chunks * T_pad) * sizeof(float4);
}

cudaError_t launch_lm_head(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const void* hidden,
                           const void* weight, int32_t T_pad, int32_t H, int32_t V,
                           const int32_t* token_ids, const int32_t* key_reach,
                           const void* blockmap, float* lse, float* entropy, float* vmin,
                           float* vmax, float* logprob, int32_t* token_pred, void* workspace,
                           int32_t* status, cudaStream_t s, int num_sms) {
  LmhParams p;
  p.T_pad = T_pad;
  p.H = H;
  p.V = V;
  p.n_mblk = T_pad / kBM;
  p.n_ntiles = (V + kBN - 1) / kBN;
  p.n_chunks = (p.n_ntiles + kChunkTiles - 1) / kChunkTiles;
  p.n_items = p.n_mblk * p.n_chunks;
  p.mb0 = 0;
  p.partial = static_cast<float4*>(workspace);
  p.coef = nullptr;
  p.grad = nullptr;
  p.ldg = 0;
  p.status = status;
  const size_t smem = sizeof(LmhSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_lmh_gemm<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < num_sms ? p.n_items : num_sms;
  k_lmh_gemm<false><<<grid, kGemmThreads, smem, s>>>(tm_h, tm_w, tm_w, p);   // no gradient map
  k_lmh_combine<<<(T_pad + kCombineThreads - 1) / kCombineThreads, kCombineThreads, 0, s>>>(
      p.partial, 2 * p.n_chunks, T_pad, key_reach, lse, entropy, vmin, vmax, status);
  int launches = 2;
  if (logprob || token_pred) {
    const BlockmapView bm{T_pad / kBlock, static_cast<int32_t*>(const_cast<void*>(blockmap))};
    k_lmh_labels<<<T_pad / kLabelWarps, kLabelWarps * 32, 0, s>>>(
        static_cast<const __nv_bfloat16*>(hidden), static_cast<const __nv_bfloat16*>(weight), H,
        V, token_ids, key_reach, bm, lse, logprob, token_pred, status);
    ++launches;
  }
  count_launches(launches);
  return cudaGetLastError();
}

cudaError_t launch_lm_head_grad(const CUtensorMap& tm_h, const CUtensorMap& tm_w,
                                const CUtensorMap& tm_g, const void* hidden, const void* weight,
                                int32_t T_pad, int32_t H,
                                int32_t V, int32_t row_lo, int32_t row_hi,
                                const int32_t* token_ids, const int32_t* key_reach,
                                const float* lse, const float* entropy, const float* g_lp,
                                const float* g_ent, void* grad, int64_t ldg, void* workspace,
                                int32_t* status, cudaStream_t s, int num_sms) {
  const int32_t rows = row_hi - row_lo;
  LmhParams p;
  p.T_pad = T_pad;
  p.H = H;
  p.V = V;
  p.mb0 = row_lo / kBM;
  p.n_mblk = rows / kBM;
  p.n_ntiles = (V + kBN - 1) / kBN;
  p.n_chunks = (p.n_ntiles + kChunkTiles - 1) / kChunkTiles;
  p.n_items = p.n_mblk * p.n_chunks;
  p.partial = nullptr;
  p.coef = static_cast<const float4*>(workspace);
  p.grad = static_cast<__nv_bfloat16*>(grad);
  p.ldg = ldg;
  p.status = status;
  k_lmh_grad_coef<<<(rows + kCombineThreads - 1) / kCombineThreads, kCombineThreads, 0, s>>>(
      row_lo, rows, T_pad, key_reach, lse, entropy, g_lp, g_ent,
      static_cast<float4*>(workspace), status);
  const size_t smem = sizeof(LmhSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_lmh_gemm<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < num_sms ? p.n_items : num_sms;
  k_lmh_gemm<true><<<grid, kGemmThreads, smem, s>>>(tm_h, tm_w, tm_g, p);
  int launches = 2;
  if (g_lp) {
    k_lmh_grad_labels<<<(rows + kLabelWarps - 1) / kLabelWarps, kLabelWarps * 32, 0, s>>>(
        static_cast<const __nv_bfloat16*>(hidden), static_cast<const __nv_bfloat16*>(weight), H,
        V, T_pad, row_lo, rows, token_ids, key_reach, g_lp, p.coef, p.grad, ldg, status);
    ++launches;
  }
  count_launches(launches);
  return cudaGetLastError();
}

}  // namespace tree
