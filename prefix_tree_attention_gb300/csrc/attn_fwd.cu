// tree_attn_fwd: tree-masked flash attention forward on tcgen05/TMEM.
//
// AReaL Tree Training guide, packing figure and section "两种注意力实现":
// softmax attention under the ancestor mask, consumed in 128-token blocks,
// batch 1.  Visibility is the interval test j <= i <= key_reach[j]; EMPTY
// tiles never reach the kernel (the blockmap lists only non-empty ones) and
// the per-element test runs only on PARTIAL tiles.
//
// One CTA = one 128-row query block x up to two query heads that read the
// same key/value head (GQA), so each K/V tile is loaded once for both.
//   warp 0     TMA producer: Q tiles once, then K, V (and the 128 reach
//              values) per listed key block through a 2-stage ring.
//   warp 1     TMEM allocator and MMA issuer (one thread):
//                S_t = Q_t K^T   (SS, both K-major)          -> TMEM S_t
//                O_t += P_t V    (TS: P_t read from TMEM, V MN-major)
//   warps 2-5  softmax for head slot 0, warps 6-9 for head slot 1.  One
//              thread owns one query row (TMEM lane), so row max and row sum
//              need no shuffles.  P is written back as bf16 over the first
//              64 columns of S_t and consumed there by the PV MMA.
// TMEM: S_0 [0,128) S_1 [128,256) O_0 [256,256+d) O_1 [384,384+d).
// tcgen05.mma operations issued by one thread execute in issue order, so the
// issuer queues QK of tile k+1 for a head slot right behind PV of tile k
// (PV reads P from the S columns before the later QK writes them) instead of
// draining the pipe to wait for PV to finish; the softmax of tile k+1 starts
// only once QK(k+1) has completed, so PV(k) is done by then and its O
// rescale never races an MMA.  The two slots interleave on the tensor pipe.  The running max is refreshed only when it grows by more than
// 8 (log2 units): P stays <= 256, and O is rescaled in TMEM only then.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace tree {
namespace {

constexpr int kFwdThreads = 320;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kGrowthLimit = 256.0f;     // 2^kRescaleThreshold

template <int D>
struct __align__(1024) FwdSmem {
  __nv_bfloat16 q[2][kBlock * D];      // per head slot, D/64 swizzled [128][64] sub-tiles
  __nv_bfloat16 k[2][kBlock * D];      // ring stages
  __nv_bfloat16 v[2][kBlock * D];
  int32_t reach[2][kBlock];
  uint64_t bar_q;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;
  uint32_t tmem_slot;
  int abort_flag;
};

struct FwdParams {
  const int32_t* key_reach;
  const int32_t* blockmap;
  int32_t T_pad, Hq, Hkv, nb, heads_per_cta, n_hgroups;
  // Query-row window [row_lo, row_hi): only these rows' O and LSE are
  // written.  The grid covers query blocks qa_lo .. qa_lo + n_qa - 1; with
  // the whole trie as the window they are visited heaviest row first.
  int32_t row_lo, row_hi, qa_lo, n_qa, windowed;
  float scale_log2;                    // softmax scale * log2(e)
  __nv_bfloat16* o;
  float* lse;
  int32_t* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Visibility bits of the 64 scores c2*64 .. c2*64+63 of a tile for query
// row i, key j = j0 + column: bit e of vis[w] stands for column
// c2*64 + 32*w + e and is set when j <= i <= reach[j].  The j <= i part is a
// prefix of each 32-column group.  For the reach part the warp lists the
// group's distinct reach values, largest first, with the mask of the keys
// that reach at least that far (one warp max and one ballot per value; the
// keys of one node share one value, so a group rarely holds more than a
// few); a row's mask is the one of the smallest listed value >= i.  A group
// with more than kRuns values falls back to testing its keys one by one
// (reach values read four at a time, a broadcast).  Warp-collective: every
// lane holds a row of the same tile.
constexpr int kRuns = 4;

__device__ __forceinline__ void visible_bits(const int32_t* rch, int c2, int32_t j0, int32_t i,
                                             uint32_t (&vis)[2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const int g = c2 * 2 + w;
    const int32_t n = i - (j0 + g * 32) + 1;   // columns with j <= i
    const uint32_t pre = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
    const int32_t r = rch[g * 32 + lane];
    uint32_t rb = 0u, left = 0xffffffffu;      // keys not yet listed (warp-uniform)
#pragma unroll
    for (int t = 0; t < kRuns; ++t) {
      if (!left) break;
      const int32_t v = __reduce_max_sync(0xffffffffu, ((left >> lane) & 1u) ? r : INT32_MIN);
      const uint32_t m = __ballot_sync(0xffffffffu, r >= v);
      if (i <= v) rb = m;
      left = ~m;
    }
    if (left) {
      rb = 0u;
      const int4* r4 = reinterpret_cast<const int4*>(rch) + g * 8;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int4 x = r4[q];
        rb |= (i <= x.x ? 1u : 0u) << (4 * q);
        rb |= (i <= x.y ? 1u : 0u) << (4 * q + 1);
        rb |= (i <= x.z ? 1u : 0u) << (4 * q + 2);
        rb |= (i <= x.w ? 1u : 0u) << (4 * q + 3);
      }
    }
    vis[w] = pre & rb;
  }
}

// Largest raw score among the visible columns c2*64 .. c2*64+63 (four
// independent max chains); -inf when none is visible.
template <bool kMasked>
__device__ __forceinline__ float half_max(uint32_t s_addr, int c2, int32_t j0, int32_t i,
                                          const int32_t* rch) {
  uint32_t vis[2] = {0xffffffffu, 0xffffffffu};
  if constexpr (kMasked) visible_bits(rch, c2, j0, i, vis);
  uint32_t ra[32], rb[32];
  tmem_ld32x2(s_addr + c2 * 64, s_addr + c2 * 64 + 32, ra, rb);
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    float xv = __uint_as_float(e < 32 ? ra[e] : rb[e - 32]);
    if constexpr (kMasked) {
      if (!(vis[e >> 5] & (1u << (e & 31)))) xv = -INFINITY;
    }
    mx[e & 3] = fmaxf(mx[e & 3], xv);
  }
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// Scores c2*64 .. c2*64+63 of a tile against the reference max m (log2
// units): P = 2^(s*scale*log2e - m) as 32 bf16 pairs in pk, their fp32 sum
// added to ls.  Paired fp32 math and two independent sum chains.  Returns,
// warp-uniformly, whether some row of the warp may have a score more than
// the threshold above m: the half's sum of P exceeds 2^threshold (or is not
// a number).  Every P is >= 0, so a P above 2^threshold always trips it; a
// sum that exceeds it without such a P only sends the tile down the exact
// path, which recomputes the same values when the max has not grown.
template <bool kMasked>
__device__ __forceinline__ bool score_half(uint32_t s_addr, int c2, int32_t j0, int32_t i,
                                           const int32_t* rch, float sl2, float m,
                                           uint32_t (&pk)[32], float& ls) {
  uint32_t vis[2] = {0xffffffffu, 0xffffffffu};
  if constexpr (kMasked) visible_bits(rch, c2, j0, i, vis);
  uint32_t ra[32], rb[32];
  tmem_ld32x2(s_addr + c2 * 64, s_addr + c2 * 64 + 32, ra, rb);
  float lt[4] = {0.f, 0.f, 0.f, 0.f};
  const float nm = -m;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    float x0, x1;
    fma2(x0, x1, __uint_as_float(e < 16 ? ra[2 * e] : rb[2 * e - 32]),
         __uint_as_float(e < 16 ? ra[2 * e + 1] : rb[2 * e - 31]), sl2, sl2, nm, nm);
    if constexpr (kMasked) {
      const uint32_t wv = vis[e >> 4];
      if (!(wv & (1u << ((2 * e) & 31)))) x0 = -INFINITY;
      if (!(wv & (2u << ((2 * e) & 31)))) x1 = -INFINITY;
    }
    const float p0 = ex2(x0);
    const float p1 = ex2(x1);
    const int a = e & 1;
    add2(lt[2 * a], lt[2 * a + 1], lt[2 * a], lt[2 * a + 1], p0, p1);
    pk[e] = pack_bf16x2(p0, p1);
  }
  const float hs = (lt[0] + lt[1]) + (lt[2] + lt[3]);
  ls += hs;
  return __any_sync(0xffffffffu, !(hs <= kGrowthLimit));
}

// O *= alpha (per row) in TMEM; warp-collective.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t o_addr, float alpha) {
#pragma unroll
  for (int c4 = 0; c4 < D / 32; ++c4) {
    uint32_t reg[32];
    tmem_ld32(o_addr + c4 * 32, reg);
#pragma unroll
    for (int e = 0; e < 32; ++e) reg[e] = __float_as_uint(__uint_as_float(reg[e]) * alpha);
    tmem_st32(o_addr + c4 * 32, reg);
  }
}

// Rare case: some row's max grew past the threshold within the second half
// of a tile after the first half's P had already been written over S.  The
// new reference max is the old one plus a whole number n of log2 units, so
// the stored first-half P (bf16) and O scale by the exact power of two 2^-n;
// the second half is recomputed from its scores, still intact in TMEM.
// Warp-collective: every TMEM access runs for the whole warp, with scale 1
// on the rows that did not grow.
template <int D, bool kMasked>
__device__ __forceinline__ void late_growth(uint32_t s_addr, uint32_t o_addr, int32_t j0, int32_t i,
                                            const int32_t* rch, float sl2, bool has_o, float& m,
                                            float& l, float ls0) {
  tmem_st_wait();   // the first-half P store must land before it is read back
  const float mt = half_max<kMasked>(s_addr, 1, j0, i, rch) * sl2;
  const bool grow = mt > m + kRescaleThreshold;
  const int n = grow ? static_cast<int>(ceilf(mt - m)) : 0;
  const float alpha = n > 125 ? 0.f : __int_as_float((127 - n) << 23);   // 2^-n
  m += static_cast<float>(n);
  l = (l + ls0) * alpha;
  if (__any_sync(0xffffffffu, grow)) {
    if (has_o) rescale_o<D>(o_addr, alpha);
    uint32_t pk[32];
    tmem_ld32(s_addr, pk);
#pragma unroll
    for (int e = 0; e < 32; ++e)
      pk[e] = pack_bf16x2(__uint_as_float(pk[e] << 16) * alpha,
                          __uint_as_float(pk[e] & 0xffff0000u) * alpha);
    tmem_st32(s_addr, pk);
  }
  uint32_t pk[32];
  float ls1 = 0.f;
  score_half<kMasked>(s_addr, 1, j0, i, rch, sl2, m, pk, ls1);   // now within the threshold
  tmem_st32(s_addr + 32, pk);
  l += ls1;
}

// One key tile of the online softmax for the query row held in this thread's
// TMEM lane: reads S (128 fp32 columns at s_addr), writes P as bf16 pairs over
// its first 64 columns, updates the running max m (log2 units) and sum l, and
// rescales O (at o_addr) in the rare case the max grew past the threshold.
// kMasked is a template argument so that FULL tiles run without the
// visibility test.
template <int D, bool kMasked>
__device__ __forceinline__ void softmax_tile(uint32_t s_addr, uint32_t o_addr, int32_t j0,
                                             int32_t i, const int32_t* rch, float sl2,
                                             bool has_o, float& m, float& l) {
  uint32_t pk[32];
  // Common path: one pass per 64-column half against the running max of the
  // earlier tiles (one FMA + ex2 per score).  Half 0's P goes over columns
  // 0..31 once its 64 scores are in registers and no row grew past the
  // threshold; half 1's P over columns 32..63.  Growth in half 0 leaves S
  // intact for the exact path below; growth in half 1 goes to late_growth.
  // Rows with no running max yet (a row's first visible tile) always take
  // the exact path.
  if (!__any_sync(0xffffffffu, m == -INFINITY)) {
    float ls0 = 0.f;
    if (!score_half<kMasked>(s_addr, 0, j0, i, rch, sl2, m, pk, ls0)) {
      tmem_st32(s_addr, pk);
      float ls1 = 0.f;
      if (!score_half<kMasked>(s_addr, 1, j0, i, rch, sl2, m, pk, ls1)) {
        tmem_st32(s_addr + 32, pk);
        l += ls0 + ls1;
      } else {
        late_growth<D, kMasked>(s_addr, o_addr, j0, i, rch, sl2, has_o, m, l, ls0);
      }
      return;
    }
  }
  // Exact path: the tile's row max first, then the same two half passes
  // against the updated reference.  The decision is per row, but tcgen05
  // loads and stores are warp-collective: O is rescaled for the whole warp
  // when any of its rows needs it, with alpha = 1 on the rows that do not.
  // (A row whose earlier tiles were all masked, e.g. one past a top-level
  // subtree boundary inside the block, first sees a key at a later tile.)
  const float mt = fmaxf(half_max<kMasked>(s_addr, 0, j0, i, rch),
                         half_max<kMasked>(s_addr, 1, j0, i, rch)) * sl2;
  const float mnew = fmaxf(m, mt);
  const bool grow = mnew > m + kRescaleThreshold;
  const float alpha = grow ? ex2(m - mnew) : 1.f;   // 0 when m = -inf
  if (grow) {
    l *= alpha;
    m = mnew;
  }
  if (has_o && __any_sync(0xffffffffu, grow)) rescale_o<D>(o_addr, alpha);
  // A row with nothing visible so far keeps m = -inf; its scores are all
  // masked here, so any finite reference gives P = 0.
  const float mref = (m == -INFINITY) ? 0.f : m;
  float ls = 0.f;
  score_half<kMasked>(s_addr, 0, j0, i, rch, sl2, mref, pk, ls);
  tmem_st32(s_addr, pk);
  score_half<kMasked>(s_addr, 1, j0, i, rch, sl2, mref, pk, ls);
  tmem_st32(s_addr + 32, pk);
  l += ls;
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
tree_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  if (ld_status(p.status)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* aligned = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(aligned);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BlockmapView bm{p.nb, const_cast<int32_t*>(p.blockmap)};
  // KV-head-major order: the CTAs resident at any moment serve one kv head,
  // so its K/V tiles stay hot in L2.  Within a kv head, the rows of all its
  // head groups (which read the same K/V tiles) run together, heaviest row
  // first, so the last kv head's long rows start with twice the span of a
  // single head group ahead of them.
  const int32_t gpk = p.n_hgroups / p.Hkv;          // head groups per kv head
  const int32_t unit = blockIdx.x / (gpk * p.n_qa);
  const int32_t j = blockIdx.x % (gpk * p.n_qa);
  const int32_t qa = p.windowed ? p.qa_lo + j / gpk : bm.row_order()[j / gpk];
  if (!dcheck(qa >= 0 && qa < p.nb, p.status)) return;
  const int32_t h0 = (unit * gpk + j % gpk) * p.heads_per_cta;
  const int nh = p.heads_per_cta;
  const int32_t kvh = h0 / (p.Hq / p.Hkv);
  const int32_t ntiles = bm.row_cnt()[qa];
  const int32_t nfull = bm.row_nfull()[qa];
  const int32_t row_off = bm.row_ptr()[qa];
  const int32_t* tiles = bm.row_idx() + row_off;
  if constexpr (kDebugBuild) {
    // The row's list must lie inside the CSR array (nb (nb + 1) / 2 words),
    // hold at most qa + 1 key blocks, FULL ones first, each in [0, qa].
    const int64_t cap = static_cast<int64_t>(p.nb) * (p.nb + 1) / 2;
    if (!dcheck(row_off >= 0 && ntiles >= 0 && ntiles <= qa + 1 &&
                    row_off + static_cast<int64_t>(ntiles) <= cap && nfull >= 0 &&
                    nfull <= ntiles,
                p.status))
      return;
    bool bad = false;
    for (int32_t k = threadIdx.x; k < ntiles; k += blockDim.x) bad |= tiles[k] < 0 || tiles[k] > qa;
    if (__syncthreads_or(bad)) {
      dcheck(false, p.status);
      return;
    }
  }
  AbortState ab{&sm.abort_flag, p.status};

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.bar_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], kBlock);
      mbar_init(&sm.o_full[s], 1);
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
  constexpr uint32_t kTileBytes = kBlock * D * 2;
  constexpr int kHalves = D / 64;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && ntiles > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&sm.bar_q, nh * kTileBytes);
      for (int t = 0; t < nh; ++t)
        for (int hf = 0; hf < kHalves; ++hf)
          tma_load_3d(sm.q[t] + hf * kBlock * 64, &tm_q, &sm.bar_q, hf * 64, h0 + t, qa * kBlock);
      int issued = 0;
      for (int k = 0; k < ntiles; ++k) {
        const int s = k & 1;
        if (k >= 2 && !mbar_wait(&sm.kv_empty[s], ((k >> 1) - 1) & 1, ab)) break;
        const int32_t kb = tiles[k];
        mbar_arrive_expect_tx(&sm.kv_full[s], 2 * kTileBytes + kBlock * 4);
        for (int hf = 0; hf < kHalves; ++hf) {
          tma_load_3d(sm.k[s] + hf * kBlock * 64, &tm_k, &sm.kv_full[s], hf * 64, kvh, kb * kBlock);
          tma_load_3d(sm.v[s] + hf * kBlock * 64, &tm_v, &sm.kv_full[s], hf * 64, kvh, kb * kBlock);
        }
        bulk_load(sm.reach[s], p.key_reach + kb * kBlock, kBlock * 4, &sm.kv_full[s]);
        issued = k + 1;
      }
      if (sm.abort_flag) {
        // Let every copy already issued land before the CTA can exit.
        mbar_drain(&sm.bar_q, 0);
        for (int k = (issued > 2 ? issued - 2 : 0); k < issued; ++k)
          mbar_drain(&sm.kv_full[k & 1], (k >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(kBlock, kBlock, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlock, D, 0, 1);
      auto issue_qk = [&](int t, uint32_t kbase) {
        const uint32_t qbase = smem_u32(sm.q[t]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBlock * 128) + (kk & 3) * 32;
          umma_ss(tbase + t * 128, sdesc_sw128(qbase + off, 16, 1024),
                  sdesc_sw128(kbase + off, 16, 1024), kIdescQK, kk > 0);
        }
        umma_commit(&sm.s_full[t]);
      };
      auto issue_pv = [&](int t, uint32_t vbase, bool accumulate) {
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk)
          umma_ts(tbase + 256 + t * 128, tbase + t * 128 + kk * 8,
                  sdesc_sw128(vbase + kk * 2048, kBlock * 128, 1024), kIdescPV,
                  (accumulate || kk > 0));
        umma_commit(&sm.o_full[t]);
      };
      // Slot by slot: QK_t(k+1) follows PV_t(k) as soon as that completes,
      // so each head slot runs its own QK -> softmax -> PV cycle and the two
      // slots settle into an offset schedule that keeps the tensor pipe fed
      // while the other slot's softmax runs.
      bool ok = mbar_wait(&sm.bar_q, 0, ab) && mbar_wait(&sm.kv_full[0], 0, ab);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < nh; ++t) issue_qk(t, smem_u32(sm.k[0]));
      }
      for (int k = 0; ok && k < ntiles; ++k) {
        const int s = k & 1, s1 = (k + 1) & 1;
        const bool more = k + 1 < ntiles;
        bool next_loaded = false;
        for (int t = 0; t < nh && ok; ++t) {
          if (!(ok = mbar_wait(&sm.p_full[t], k & 1, ab))) break;
          tc_fence_after();
          issue_pv(t, smem_u32(sm.v[s]), k > 0);
          if (t == nh - 1) umma_commit(&sm.kv_empty[s]);   // all PVs of tile k issued
          if (!more) continue;
          if (!next_loaded) {
            if (!(ok = mbar_wait(&sm.kv_full[s1], ((k + 1) >> 1) & 1, ab))) break;
            next_loaded = true;
          }
          issue_qk(t, smem_u32(sm.k[s1]));       // in order behind PV_t(k)
        }
      }
      if (!ok) {
        umma_commit(&sm.drain);   // wait for every MMA already issued
        mbar_drain(&sm.drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    if (t < nh) {
      const int32_t h = h0 + t;
      const int32_t i = qa * kBlock + r;
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t s_addr = tbase + lane_off + t * 128;
      const uint32_t o_addr = tbase + lane_off + 256 + t * 128;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      int32_t kb_next = ntiles > 0 ? tiles[0] : 0;
      for (int k = 0; k < ntiles; ++k) {
        // the tile index is read before the wait so its latency overlaps it
        const int32_t j0 = kb_next * kBlock;
        if (k + 1 < ntiles) kb_next = tiles[k + 1];
        if (!(ok = mbar_wait_warp(&sm.s_full[t], k & 1, ab))) break;
        tc_fence_after();
        const int32_t* rch = sm.reach[k & 1];
        if (k >= nfull)
          softmax_tile<D, true>(s_addr, o_addr, j0, i, rch, p.scale_log2, k > 0, m, l);
        else
          softmax_tile<D, false>(s_addr, o_addr, j0, i, rch, p.scale_log2, k > 0, m, l);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[t]);
      }
      // ---------------------------------------------------------- epilogue
      // (every lane takes part in the warp-collective TMEM loads; only rows
      // inside the window store)
      const bool in_window = i >= p.row_lo && i < p.row_hi;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(i) * p.Hq + h) * D;
      const bool have_o = ok && ntiles > 0 && mbar_wait_warp(&sm.o_full[t], (ntiles - 1) & 1, ab);
      if (have_o && !p.windowed) {
        // O through shared memory: this slot's Q tile, which its last QK has
        // finished reading, takes the normalised rows in the Q tile's own
        // 128-byte-swizzled layout; one lane then writes the warp's 32 rows
        // with a bulk tensor store per 64-column half (a thread's direct
        // stores would touch 32 rows of O per instruction).
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        uint8_t* stage = reinterpret_cast<uint8_t*>(sm.q[t]);
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t reg[32];
          tmem_ld32(o_addr + c4 * 32, reg);
          uint8_t* row = stage + (c4 >> 1) * (kBlock * 128) + r * 128;
#pragma unroll
          for (int e8 = 0; e8 < 4; ++e8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 0]) * inv_l, __uint_as_float(reg[e8 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 2]) * inv_l, __uint_as_float(reg[e8 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 4]) * inv_l, __uint_as_float(reg[e8 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 6]) * inv_l, __uint_as_float(reg[e8 * 8 + 7]) * inv_l);
            const int chunk = (c4 & 1) * 4 + e8;
            *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) = w;
          }
        }
        fence_proxy_async_smem();        // generic-proxy writes -> visible to the bulk copy
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf)
            tma_store_3d(&tm_o, stage + hf * (kBlock * 128) + quarter * 32 * 128, hf * 64, h,
                         qa * kBlock + quarter * 32);
          bulk_commit();
          bulk_wait_read();              // the tile must outlive the copy's reads
        }
        __syncwarp();
        p.lse[static_cast<size_t>(h) * p.T_pad + i] =
            l > 0.f ? m * 0.69314718055994531f + logf(l) : -INFINITY;
      } else if (have_o) {
        // a window may start or end inside the warp's rows: direct stores
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t reg[32];
          tmem_ld32(o_addr + c4 * 32, reg);
#pragma unroll
          for (int e8 = 0; e8 < 4; ++e8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 0]) * inv_l, __uint_as_float(reg[e8 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 2]) * inv_l, __uint_as_float(reg[e8 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 4]) * inv_l, __uint_as_float(reg[e8 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(reg[e8 * 8 + 6]) * inv_l, __uint_as_float(reg[e8 * 8 + 7]) * inv_l);
            if (in_window) *reinterpret_cast<uint4*>(orow + c4 * 32 + e8 * 8) = w;
          }
        }
        if (in_window)
          p.lse[static_cast<size_t>(h) * p.T_pad + i] =
              l > 0.f ? m * 0.69314718055994531f + logf(l) : -INFINITY;
      } else if (ntiles == 0 && in_window) {
#pragma unroll
        for (int c = 0; c < D; c += 8)
          *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
        p.lse[static_cast<size_t>(h) * p.T_pad + i] = -INFINITY;
      }
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

template <int D>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdParams& p, int grid, cudaStream_t s) {
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(tree_attn_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  tree_attn_fwd_kernel<D><<<grid, kFwdThreads, smem, s>>>(tq, tk, tv, to, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const int32_t* key_reach, const void* blockmap, int32_t T_pad,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale, void* o, float* lse,
                            int32_t* status, cudaStream_t s, int32_t row_lo, int32_t row_hi) {
  const int g = Hq / Hkv;
  FwdParams p;
  p.key_reach = key_reach;
  p.blockmap = static_cast<const int32_t*>(blockmap);
  p.T_pad = T_pad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.nb = T_pad / kBlock;
  p.heads_per_cta = (g % 2 == 0) ? 2 : 1;
  p.n_hgroups = Hq / p.heads_per_cta;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = status;
  p.row_lo = row_lo;
  p.row_hi = row_hi;
  p.windowed = (row_lo > 0 || row_hi < T_pad) ? 1 : 0;
  p.qa_lo = row_lo / kBlock;
  p.n_qa = row_hi > row_lo ? (row_hi - 1) / kBlock - p.qa_lo + 1 : 0;
  if (p.n_qa == 0) return cudaSuccess;
  const int grid = p.n_qa * p.n_hgroups;
  return d == 64 ? launch_fwd_d<64>(tq, tk, tv, to, p, grid, s)
                 : launch_fwd_d<128>(tq, tk, tv, to, p, grid, s);
}

}  // namespace tree
