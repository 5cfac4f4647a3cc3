// tree_logprobs_entropy and tree_merge_per_sequence: log-probabilities and
// entropies of packed next-token logits, and their per-sequence merge.
//
// AReaL Tree Training guide, section "Log Probability 计算：树结构的特殊处理".
// A packed row's logits predict the next token of every sequence through it:
// inside a node the next packed row, across a node boundary (the page's
// transition from the parent's last row to a child's first token) every
// child's first token.  So each real token j has one predicting row pred(j),
// and the page's per-node caches become plain structure: every row's
// distribution is reduced once, every (pred, label) pair is gathered once.
//
// pred(j) from the interval form of the mask, visible(i, j) <=> j <= i <=
// reach[j]: pred(j) is the last key before j that row j sees, i.e. the
// largest i < j with reach[i] >= j (-1 for the first token of a top-level
// node).  It is j - 1 except at node starts, where the search skips the
// subtrees of earlier siblings.  A key block b can hold pred(j) only if the
// tile (block(j), b) is non-empty, i.e. col_hi[b] >= block(j) in the blockmap,
// so whole blocks are skipped with one word.
//
// Kernels (each skips its work once *dev_status is non-zero):
//  1 k_row_stats     one CTA per packed row: one streaming pass over the V
//                    logits keeps a running max m, s = sum 2^u and
//                    t = sum 2^u * u with u = (x - m) log2(e); then
//                    lse = m + ln s and entropy = ln 2 * (log2 s - t / s)
//                    (entropy = lse - sum p x, written relative to m).
//                    HBM-bound: reads V logits per row once.
//  2 k_label_lp      one thread per token: pred(j), then
//                    logprob[j] = logits[pred(j), token_ids[j]] - lse[pred(j)].
//  3 k_merge         one thread per output element of [n_seqs, max_len].
//
// The gradient (tree_logprobs_entropy_bwd, tree_merge_per_sequence_bwd):
//  4 k_merge_bwd     the merge's adjoint: one thread per [n_seqs, max_len]
//                    entry adds its gradient to the packed token (or row) it
//                    was read from; shared-prefix tokens sum over sequences.
//  5 k_row_bwd       one CTA per packed row r.  Row r predicts exactly the
//                    tokens j with pred(j) = r: its children in the token
//                    tree, which in packed order are r + 1 and then each
//                    next sibling at reach[j] + 1, while j <= reach[r].  With
//                    G = sum of their logprob gradients, E the row's entropy
//                    gradient, p = softmax(x), H the entropy:
//                      d x_v = -p_v (G + E (x_v - lse + H)) + g_lp[j] [v = y_j]
//                    = -p_v (A + E x_v) with A = G + E (H - lse), one
//                    streaming pass that reads and writes V values; then the
//                    CTA's first thread adds each child's g_lp at its label
//                    (labels of one row's children are distinct in a trie)
//                    and rewrites those few entries.  HBM-bound: V reads and
//                    V writes per row.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace tree {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kUnroll = 4;            // 16-byte loads in flight per thread
constexpr int kLabelThreads = 128;
constexpr int kMergeThreads = 256;
template <bool kBf16>
__device__ __forceinline__ float load_logit(const void* row, int64_t e) {
  if constexpr (kBf16) {
    const uint16_t bits = reinterpret_cast<const uint16_t*>(row)[e];
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  } else {
    return reinterpret_cast<const float*>(row)[e];
  }
}

// A 16-byte group of logits at the current reference: 8 bf16 or 4 fp32.
template <bool kBf16, bool kMin>
__device__ __forceinline__ void acc_group_max(const uint4& v, uint32_t& mx_bf, float& mx_f,
                                              uint32_t& mn_bf, float& mn_f) {
  if constexpr (kBf16) {
    mx_bf = max_bf16x2(max_bf16x2(mx_bf, max_bf16x2(v.x, v.y)), max_bf16x2(v.z, v.w));
    if constexpr (kMin)
      mn_bf = min_bf16x2(min_bf16x2(mn_bf, min_bf16x2(v.x, v.y)), min_bf16x2(v.z, v.w));
  } else {
    mx_f = fmaxf(fmaxf(mx_f, fmaxf(__uint_as_float(v.x), __uint_as_float(v.y))),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    if constexpr (kMin)
      mn_f = fminf(fminf(mn_f, fminf(__uint_as_float(v.x), __uint_as_float(v.y))),
                   fminf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

template <bool kBf16>
__device__ __forceinline__ void acc_group(Acc& a, float nmL, const uint4& v) {
  if constexpr (kBf16) {
    acc_pair(a, nmL, bf_lo(v.x), bf_hi(v.x));
    acc_pair(a, nmL, bf_lo(v.y), bf_hi(v.y));
    acc_pair(a, nmL, bf_lo(v.z), bf_hi(v.z));
    acc_pair(a, nmL, bf_lo(v.w), bf_hi(v.w));
  } else {
    acc_pair(a, nmL, __uint_as_float(v.x), __uint_as_float(v.y));
    acc_pair(a, nmL, __uint_as_float(v.z), __uint_as_float(v.w));
  }
}

// kVec: every row starts on a 16-byte boundary (checked on the host), so the
// first V - V % W logits are read as 16-byte groups of W.
template <bool kBf16, bool kVec, bool kMin>
__global__ void __launch_bounds__(kRowThreads) k_row_stats(
    const void* __restrict__ logits, int64_t row_stride, int32_t V,
    const int32_t* __restrict__ reach, float* __restrict__ lse, float* __restrict__ entropy,
    float* __restrict__ vmin, float* __restrict__ vmax, const int32_t* status) {
  if (ld_status(status)) return;
  const int32_t row = blockIdx.x;
  const int tid = threadIdx.x;
  if (reach[row] < row) {            // pad token: no distribution
    if (tid == 0) {
      lse[row] = 0.f;
      if (entropy) entropy[row] = 0.f;
      if (vmin) vmin[row] = 0.f;
      if (vmax) vmax[row] = 0.f;
    }
    return;
  }
  constexpr int kEsz = kBf16 ? 2 : 4;
  constexpr int kW = 16 / kEsz;      // logits per 16-byte group
  const char* base = reinterpret_cast<const char*>(logits) + row * row_stride * kEsz;
  Acc a;
  acc_init(a);
  int64_t done = 0;
  if constexpr (kVec) {
    const uint4* g = reinterpret_cast<const uint4*>(base);
    const int32_t ng = V / kW;
    int32_t i = tid;
    for (; i + (kUnroll - 1) * kRowThreads < ng; i += kUnroll * kRowThreads) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(g + i + u * kRowThreads);
      uint32_t mx_bf = 0xff80ff80u, mn_bf = 0x7f807f80u;   // (-inf, -inf), (+inf, +inf)
      float mx_f = -INFINITY, mn_f = INFINITY;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) acc_group_max<kBf16, kMin>(v[u], mx_bf, mx_f, mn_bf, mn_f);
      if constexpr (kBf16) {
        mx_f = fmaxf(bf_lo(mx_bf), bf_hi(mx_bf));
        if constexpr (kMin) mn_f = fminf(bf_lo(mn_bf), bf_hi(mn_bf));
      }
      if constexpr (kMin) a.mn = fminf(a.mn, mn_f);
      if (mx_f > a.m) acc_rebase(a, mx_f);
      const float nmL = -a.m * kLog2e;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) acc_group<kBf16>(a, nmL, v[u]);
    }
    for (; i < ng; i += kRowThreads) {
      const uint4 v = __ldcs(g + i);
      uint32_t mx_bf = 0xff80ff80u, mn_bf = 0x7f807f80u;
      float mx_f = -INFINITY, mn_f = INFINITY;
      acc_group_max<kBf16, kMin>(v, mx_bf, mx_f, mn_bf, mn_f);
      if constexpr (kBf16) {
        mx_f = fmaxf(bf_lo(mx_bf), bf_hi(mx_bf));
        if constexpr (kMin) mn_f = fminf(bf_lo(mn_bf), bf_hi(mn_bf));
      }
      if constexpr (kMin) a.mn = fminf(a.mn, mn_f);
      if (mx_f > a.m) acc_rebase(a, mx_f);
      acc_group<kBf16>(a, -a.m * kLog2e, v);
    }
    done = static_cast<int64_t>(ng) * kW;
  }
  for (int64_t e = done + tid; e < V; e += kRowThreads) acc_one(a, load_logit<kBf16>(base, e));

  // CTA reduction: warps by shuffles, then the warp leaders in warp 0.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Acc b = acc_shfl_xor(a, o);
    acc_merge(a, b);
  }
  __shared__ Acc part[kRowWarps];
  if ((tid & 31) == 0) part[tid >> 5] = a;
  __syncthreads();
  if (tid < 32) {
    if (tid < kRowWarps) a = part[tid];
    else acc_init(a);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const Acc b = acc_shfl_xor(a, o);
      acc_merge(a, b);
    }
    if (tid == 0) {
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
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kLabelThreads) k_label_lp(
    const void* __restrict__ logits, int64_t row_stride, int32_t V,
    const int32_t* __restrict__ token_ids, const int32_t* __restrict__ reach,
    BlockmapView bm, const float* __restrict__ lse, float* __restrict__ logprob,
    int32_t* __restrict__ pred_out, int32_t* status) {
  if (ld_status(status)) return;
  const int32_t j = blockIdx.x * kLabelThreads + threadIdx.x;   // T_pad % 128 == 0
  const int lane = threadIdx.x & 31;
  const bool real = reach[j] >= j;
  int32_t pred = -1;
  bool slow = false;
  if (real && j > 0) {
    if (reach[j - 1] >= j) pred = j - 1;
    else slow = true;
  }
  uint32_t pend = __ballot_sync(0xffffffffu, slow);
  while (pend) {
    const int src = __ffs(pend) - 1;
    pend &= pend - 1;
    const int32_t q = __shfl_sync(0xffffffffu, j, src);
    const int32_t found = find_pred(q, reach, bm.col_hi(), lane);
    if (lane == src) pred = found;
  }
  if (pred_out) pred_out[j] = pred;
  if (logprob) {
    float out = 0.f;
    if (pred >= 0) {
      const int32_t tok = token_ids[j];
      if (tok < 0 || tok >= V) {
        set_status(status, TREE_ERR_MALFORMED_TREE);
        out = __int_as_float(0x7fc00000);
      } else {
        constexpr int kEsz = kBf16 ? 2 : 4;
        const char* row = reinterpret_cast<const char*>(logits) + pred * row_stride * kEsz;
        out = load_logit<kBf16>(row, tok) - lse[pred];
      }
    }
    logprob[j] = out;
  }
}

__global__ void __launch_bounds__(kMergeThreads) k_merge(
    const float* __restrict__ src, int64_t n_src, const int32_t* __restrict__ seq_pos,
    int64_t n_pos, const int64_t* __restrict__ seq_off, int32_t n_seqs, int32_t max_len,
    int32_t shift, int32_t trim, float pad, float* __restrict__ out, int32_t* status) {
  if (ld_status(status)) return;
  const int32_t t = blockIdx.x * kMergeThreads + threadIdx.x;
  if (t >= max_len) return;
  for (int32_t s = blockIdx.y; s < n_seqs; s += gridDim.y) {
    const int64_t off = seq_off[s], end = seq_off[s + 1];
    const int64_t n = end - off - trim;              // entries of sequence s
    float v = pad;
    if (off < 0 || end < off || end > n_pos) {
      set_status(status, TREE_ERR_INVALID_ARG);
      v = __int_as_float(0x7fc00000);
    } else if (t < n) {
      const int32_t p = seq_pos[off + t + shift];
      if (p < 0 || p >= n_src) {
        set_status(status, TREE_ERR_MALFORMED_TREE);
        v = __int_as_float(0x7fc00000);
      } else {
        v = src[p];
      }
    }
    if (t == 0 && n > max_len) set_status(status, TREE_ERR_CAPACITY);
    out[static_cast<int64_t>(s) * max_len + t] = v;
  }
}

__global__ void __launch_bounds__(kMergeThreads) k_merge_bwd(
    const float* __restrict__ out_grad, const int32_t* __restrict__ seq_pos, int64_t n_pos,
    const int64_t* __restrict__ seq_off, int32_t n_seqs, int32_t max_len, int32_t shift,
    int32_t trim, float* __restrict__ src_grad, int64_t n_src, int32_t* status) {
  if (ld_status(status)) return;
  const int32_t t = blockIdx.x * kMergeThreads + threadIdx.x;
  if (t >= max_len) return;
  for (int32_t s = blockIdx.y; s < n_seqs; s += gridDim.y) {
    const int64_t off = seq_off[s], end = seq_off[s + 1];
    if (off < 0 || end < off || end > n_pos) {
      set_status(status, TREE_ERR_INVALID_ARG);
      continue;
    }
    const int64_t n = end - off - trim;
    if (t == 0 && n > max_len) set_status(status, TREE_ERR_CAPACITY);
    if (t >= n) continue;
    const int32_t p = seq_pos[off + t + shift];
    if (p < 0 || p >= n_src) {
      set_status(status, TREE_ERR_MALFORMED_TREE);
      continue;
    }
    const float g = out_grad[static_cast<int64_t>(s) * max_len + t];
    if (g != 0.f) atomicAdd(src_grad + p, g);
  }
}

template <bool kBf16>
__device__ __forceinline__ void store_grad(void* row, int64_t e, float d) {
  if constexpr (kBf16)
    reinterpret_cast<__nv_bfloat16*>(row)[e] = __float2bfloat16_rn(d);
  else
    reinterpret_cast<float*>(row)[e] = d;
}

// d = p (nA + nE x) for the 16-byte group v, p = 2^(x log2 e + nL).
template <bool kBf16>
__device__ __forceinline__ uint4 grad_group(const uint4& v, float nL, float nE, float nA) {
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
  const uint32_t* iw = reinterpret_cast<const uint32_t*>(&v);
  if constexpr (kBf16) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float u0, u1, w0, w1, d0, d1;
      const float x0 = bf_lo(iw[k]), x1 = bf_hi(iw[k]);
      fma2(u0, u1, x0, x1, kLog2e, kLog2e, nL, nL);
      fma2(w0, w1, x0, x1, nE, nE, nA, nA);
      mul2(d0, d1, ex2f(u0), ex2f(u1), w0, w1);
      ow[k] = pack_bf16x2(d0, d1);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; k += 2) {
      float u0, u1, w0, w1, d0, d1;
      const float x0 = __uint_as_float(iw[k]), x1 = __uint_as_float(iw[k + 1]);
      fma2(u0, u1, x0, x1, kLog2e, kLog2e, nL, nL);
      fma2(w0, w1, x0, x1, nE, nE, nA, nA);
      mul2(d0, d1, ex2f(u0), ex2f(u1), w0, w1);
      ow[k] = __float_as_uint(d0);
      ow[k + 1] = __float_as_uint(d1);
    }
  }
  return o;
}

// The next child of a row after child j: the token after j's subtree.
// key_reach from tree_pack_positions makes this strictly increasing; a
// malformed one that does not ends the walk (and is reported) instead of
// looping.
__device__ __forceinline__ int32_t next_child(int32_t j, const int32_t* __restrict__ reach,
                                              int32_t* status) {
  const int32_t n = reach[j] + 1;
  if (n <= j) {
    set_status(status, TREE_ERR_MALFORMED_TREE);
    return INT32_MAX;
  }
  return n;
}

// kVec: logits and gradient rows both start on 16-byte boundaries.
template <bool kBf16, bool kVec>
__global__ void __launch_bounds__(kRowThreads) k_row_bwd(
    const void* __restrict__ logits, int64_t row_stride, int32_t V,
    const int32_t* __restrict__ token_ids, const int32_t* __restrict__ reach,
    const float* __restrict__ lse, const float* __restrict__ entropy,
    const float* __restrict__ g_lp, const float* __restrict__ g_ent, void* __restrict__ dlogits,
    int64_t drow_stride, int32_t* status) {
  if (ld_status(status)) return;
  const int32_t row = blockIdx.x;
  const int tid = threadIdx.x;
  constexpr int kEsz = kBf16 ? 2 : 4;
  constexpr int kW = 16 / kEsz;
  const char* src = reinterpret_cast<const char*>(logits) + row * row_stride * kEsz;
  char* dst = reinterpret_cast<char*>(dlogits) + row * drow_stride * kEsz;
  int32_t rr = reach[row];
  if (rr >= static_cast<int32_t>(gridDim.x)) {       // past the last row: malformed
    if (tid == 0) set_status(status, TREE_ERR_MALFORMED_TREE);
    rr = gridDim.x - 1;
  }
  __shared__ float sh_G;
  float nL = 0.f, nE = 0.f, nA = 0.f;
  if (rr >= row) {                       // a real row: gather its children's gradients
    if (tid == 0) {
      float G = 0.f;
      if (g_lp)
        for (int32_t j = row + 1; j <= rr; j = next_child(j, reach, status)) G += g_lp[j];
      sh_G = G;
    }
    const float L = lse[row];
    const float E = g_ent ? g_ent[row] : 0.f;
    const float H = E != 0.f ? entropy[row] : 0.f;
    __syncthreads();
    nL = -L * kLog2e;
    nE = -E;
    nA = -(sh_G + E * (H - L));
  }
  // A pad row (rr < row) has nE = nA = 0: every gradient is +0 * p = 0, but
  // p may be anything there, so write zeros directly.
  const bool pad = rr < row;
  int64_t done = 0;
  if constexpr (kVec) {
    const uint4* g = reinterpret_cast<const uint4*>(src);
    uint4* o = reinterpret_cast<uint4*>(dst);
    const int32_t ng = V / kW;
    int32_t i = tid;
    if (pad) {
      for (; i < ng; i += kRowThreads) __stcs(o + i, make_uint4(0, 0, 0, 0));
    } else {
      for (; i + (kUnroll - 1) * kRowThreads < ng; i += kUnroll * kRowThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(g + i + u * kRowThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          __stcs(o + i + u * kRowThreads, grad_group<kBf16>(v[u], nL, nE, nA));
      }
      for (; i < ng; i += kRowThreads) __stcs(o + i, grad_group<kBf16>(__ldcs(g + i), nL, nE, nA));
    }
    done = static_cast<int64_t>(ng) * kW;
  }
  for (int64_t e = done + tid; e < V; e += kRowThreads) {
    float d = 0.f;
    if (!pad) {
      const float x = load_logit<kBf16>(src, e);
      d = ex2f(fmaf(x, kLog2e, nL)) * fmaf(x, nE, nA);
    }
    store_grad<kBf16>(dst, e, d);
  }
  if (pad || !g_lp) return;
  __syncthreads();                       // the dense values are written
  if (tid == 0) {
    for (int32_t j = row + 1; j <= rr; j = next_child(j, reach, status)) {
      const int32_t y = token_ids[j];
      if (y < 0 || y >= V) {
        set_status(status, TREE_ERR_MALFORMED_TREE);
        continue;
      }
      const float x = load_logit<kBf16>(src, y);
      const float d = fmaf(ex2f(fmaf(x, kLog2e, nL)), fmaf(x, nE, nA), g_lp[j]);
      store_grad<kBf16>(dst, y, d);
    }
  }
}

template <bool kBf16>
cudaError_t launch_stats(const void* logits, int64_t stride, int32_t T_pad, int32_t V, bool vec,
                         const int32_t* reach, float* lse, float* ent, float* vmin, float* vmax,
                         int32_t* status, cudaStream_t s) {
  const dim3 grid(T_pad), block(kRowThreads);
  const bool want_min = vmin != nullptr;
  if (vec && want_min)
    k_row_stats<kBf16, true, true><<<grid, block, 0, s>>>(logits, stride, V, reach, lse, ent,
                                                          vmin, vmax, status);
  else if (vec)
    k_row_stats<kBf16, true, false><<<grid, block, 0, s>>>(logits, stride, V, reach, lse, ent,
                                                           vmin, vmax, status);
  else if (want_min)
    k_row_stats<kBf16, false, true><<<grid, block, 0, s>>>(logits, stride, V, reach, lse, ent,
                                                           vmin, vmax, status);
  else
    k_row_stats<kBf16, false, false><<<grid, block, 0, s>>>(logits, stride, V, reach, lse, ent,
                                                            vmin, vmax, status);
  return cudaGetLastError();
}

}  // namespace
}  // namespace tree

extern "C" {

tree_status_t tree_logprobs_entropy(const void* logits, int32_t dtype, int64_t row_stride,
                                    int32_t T_pad, int32_t V, const int32_t* token_ids,
                                    const int32_t* key_reach, const void* blockmap,
                                    size_t blockmap_bytes, float* lse, float* entropy,
                                    float* vocab_min, float* vocab_max, float* logprob,
                                    int32_t* token_pred, int32_t* dev_status,
                                    tree_stream_t stream) {
  using namespace tree;
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32) return TREE_ERR_UNSUPPORTED;
  if (T_pad < 0 || V < 1 || row_stride < V) return TREE_ERR_INVALID_ARG;
  if (T_pad % kBlock) return TREE_ERR_ALIGNMENT;
  if (T_pad == 0) return TREE_OK;
  if (!logits || !key_reach || !lse || !dev_status) return TREE_ERR_INVALID_ARG;
  const bool labels = logprob != nullptr || token_pred != nullptr;
  if (labels && !blockmap) return TREE_ERR_INVALID_ARG;
  if (logprob && !token_ids) return TREE_ERR_INVALID_ARG;
  if (labels && blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == TREE_DTYPE_BF16;
  const int64_t esz = bf16 ? 2 : 4;
  const bool vec = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (row_stride * esz) % 16 == 0;
  cudaError_t e = bf16 ? launch_stats<true>(logits, row_stride, T_pad, V, vec, key_reach, lse,
                                            entropy, vocab_min, vocab_max, dev_status, s)
                       : launch_stats<false>(logits, row_stride, T_pad, V, vec, key_reach, lse,
                                             entropy, vocab_min, vocab_max, dev_status, s);
  count_launches(1);
  if (e != cudaSuccess) return TREE_ERR_CUDA;
  if (labels) {
    BlockmapView bm{T_pad / kBlock,
                    static_cast<int32_t*>(const_cast<void*>(blockmap))};
    const dim3 grid(T_pad / kLabelThreads), block(kLabelThreads);
    if (bf16)
      k_label_lp<true><<<grid, block, 0, s>>>(logits, row_stride, V, token_ids, key_reach, bm,
                                              lse, logprob, token_pred, dev_status);
    else
      k_label_lp<false><<<grid, block, 0, s>>>(logits, row_stride, V, token_ids, key_reach, bm,
                                               lse, logprob, token_pred, dev_status);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess) return TREE_ERR_CUDA;
  }
  return TREE_OK;
}

tree_status_t tree_merge_per_sequence(const float* src, int64_t n_src, const int32_t* seq_pos,
                                      int64_t n_pos, const int64_t* seq_offsets, int32_t n_seqs,
                                      int32_t max_len, int32_t shift, int32_t trim,
                                      float padding_value, float* out, int32_t* dev_status,
                                      tree_stream_t stream) {
  using namespace tree;
  if (n_seqs < 0 || max_len < 0 || n_src < 0 || n_pos < 0 || shift < 0 || trim < shift)
    return TREE_ERR_INVALID_ARG;
  if (n_seqs == 0 || max_len == 0) return TREE_OK;
  if (!src || !seq_pos || !seq_offsets || !out || !dev_status) return TREE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((max_len + kMergeThreads - 1) / kMergeThreads, n_seqs < 65535 ? n_seqs : 65535);
  k_merge<<<grid, kMergeThreads, 0, s>>>(src, n_src, seq_pos, n_pos, seq_offsets, n_seqs, max_len,
                                         shift, trim, padding_value, out, dev_status);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TREE_OK : TREE_ERR_CUDA;
}

tree_status_t tree_merge_per_sequence_bwd(const float* out_grad, const int32_t* seq_pos,
                                          int64_t n_pos, const int64_t* seq_offsets,
                                          int32_t n_seqs, int32_t max_len, int32_t shift,
                                          int32_t trim, float* src_grad, int64_t n_src,
                                          int32_t* dev_status, tree_stream_t stream) {
  using namespace tree;
  if (n_seqs < 0 || max_len < 0 || n_src < 0 || n_pos < 0 || shift < 0 || trim < shift)
    return TREE_ERR_INVALID_ARG;
  if (n_seqs == 0 || max_len == 0) return TREE_OK;
  if (!out_grad || !seq_pos || !seq_offsets || !src_grad || !dev_status)
    return TREE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((max_len + kMergeThreads - 1) / kMergeThreads, n_seqs < 65535 ? n_seqs : 65535);
  k_merge_bwd<<<grid, kMergeThreads, 0, s>>>(out_grad, seq_pos, n_pos, seq_offsets, n_seqs,
                                             max_len, shift, trim, src_grad, n_src, dev_status);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TREE_OK : TREE_ERR_CUDA;
}

tree_status_t tree_logprobs_entropy_bwd(const void* logits, int32_t dtype, int64_t row_stride,
                                        int32_t T_pad, int32_t V, const int32_t* token_ids,
                                        const int32_t* key_reach, const float* lse,
                                        const float* entropy, const float* grad_logprob,
                                        const float* grad_entropy, void* grad_logits,
                                        int64_t grad_row_stride, int32_t* dev_status,
                                        tree_stream_t stream) {
  using namespace tree;
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32) return TREE_ERR_UNSUPPORTED;
  if (T_pad < 0 || V < 1 || row_stride < V || grad_row_stride < V) return TREE_ERR_INVALID_ARG;
  if (T_pad % kBlock) return TREE_ERR_ALIGNMENT;
  if (T_pad == 0) return TREE_OK;
  if (!logits || !key_reach || !lse || !grad_logits || !dev_status) return TREE_ERR_INVALID_ARG;
  if (grad_logprob && !token_ids) return TREE_ERR_INVALID_ARG;
  if (grad_entropy && !entropy) return TREE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == TREE_DTYPE_BF16;
  const int64_t esz = bf16 ? 2 : 4;
  const bool vec = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(grad_logits) & 15u) == 0 &&
                   (row_stride * esz) % 16 == 0 && (grad_row_stride * esz) % 16 == 0;
  const dim3 grid(T_pad), block(kRowThreads);
#define TREE_ROW_BWD(B, VEC)                                                                  \
  k_row_bwd<B, VEC><<<grid, block, 0, s>>>(logits, row_stride, V, token_ids, key_reach, lse,  \
                                           entropy, grad_logprob, grad_entropy, grad_logits,  \
                                           grad_row_stride, dev_status)
  if (bf16 && vec) TREE_ROW_BWD(true, true);
  else if (bf16) TREE_ROW_BWD(true, false);
  else if (vec) TREE_ROW_BWD(false, true);
  else TREE_ROW_BWD(false, false);
#undef TREE_ROW_BWD
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TREE_OK : TREE_ERR_CUDA;
}

}  // extern "C"
