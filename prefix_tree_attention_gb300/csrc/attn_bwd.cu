// tree_attn_bwd: backward of the tree-masked attention on tcgen05/TMEM.
//
// AREAL-DTA, section 3 "Problem formalisation": the training loss is a sum of
// per-sequence losses, a shared prefix is processed once, and its gradient
// accumulates the contributions of all descendant sequences.  Here that is
// automatic: a shared-prefix key is visible to the queries of every
// continuation, so its dK/dV sum over all of them.
//
// Kernels:
//  a4 prep     D[h,i] = sum_d dO[i,h,d] O[i,h,d];  lse2 = LSE * log2(e); both
//              are stored negated (the main kernel adds them);
//              the fp32 dQ accumulator is zeroed.
//  a5 main     one CTA per (key block kb, kv head).  The key block's
//              non-empty query tiles form the column run kb..col_hi of the
//              blockmap; the CTA visits every (query head of this kv head,
//              query block) pair of that run.  Per pair, with keys on TMEM
//              lanes (M = 128 keys):
//                S^T  = K Q^T            SS  -> TMEM [256,384)
//                dP^T = V dO^T           SS  -> TMEM [384,512)
//                P^T  = exp2(S^T*scale*log2e - lse2)  (mask on PARTIAL tiles)
//                dS^T = P^T * (dP^T - D)
//                dV  += P^T dO           TS (P^T bf16 in TMEM) -> [0, d)
//                dK  += dS^T Q           TS (dS^T bf16 in TMEM) -> [128, 128+d)
//                dQ   = dS K             SS (dS staged in smem, MN-major)
//                                        -> TMEM [384, 384+d), then fp32
//                                        vector atomics into the accumulator.
//              Sixteen warps in four warpgroups:
//                warps 0-3   dQ warpgroup: per pair, dQ out of TMEM, staged in
//                            the smem dS tile (free once the dQ MMA has read
//                            it) and added into the fp32 accumulator by bulk
//                            tensor reduce-adds at L2;
//                warps 4-11  element-wise warps (P, dS) on query columns 0-63
//                            and 64-127;
//                warp 12     TMA producer (K, V once; Q, dO, lse2, D per pair in
//                            a 2-stage ring);
//                warp 13     TMEM allocator + MMA issuer; warps 14-15 idle.
//              The element-wise warps never wait for a bulk copy: only their
//              next dS store waits until the dQ warps' reduces have read the
//              tile, so every element-wise warp reaches the next pair at the
//              same time.  setmaxnreg moves registers from the control and dQ
//              warpgroups to the element-wise ones.
//  a6 convert  dQ = bf16(scale * accumulator).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace tree {
namespace {

constexpr int kBwdThreads = 512;
// Per-thread registers after the split (launch: 512 x 128).
constexpr uint32_t kRegsDq = 96, kRegsEw = 168, kRegsCtl = 72;
static_assert(128 * kRegsDq + 256 * kRegsEw + 128 * kRegsCtl <= kBwdThreads * 128,
              "register split exceeds the launch allocation");
constexpr int kWarpProducer = 12, kWarpMma = 13, kWarpEw0 = 4;
// Query blocks of a key block's column one CTA walks in the fp32-accumulate
// (windowed stack-gradient) mode.
constexpr int kSplitQ = 4;

template <int D>
struct __align__(1024) BwdSmem {
  __nv_bfloat16 k[kBlock * D];          // resident key tile (D/64 swizzled sub-tiles)
  __nv_bfloat16 v[kBlock * D];
  __nv_bfloat16 q[2][kBlock * D];       // ring stages
  __nv_bfloat16 dout[2][kBlock * D];
  __nv_bfloat16 ds[kBlock * kBlock];    // dS^T as [key][query], two 64-query halves;
                                        // then eight 4 KB dQ staging boxes
  float lse2[2][kBlock];
  float dd[2][kBlock];
  uint64_t bar_kv;
  uint64_t full[2], empty[2];
  uint64_t s_full, dp_full, ew_done, dvdk_done, dq_full, dq_free, dsbuf_free, drain;
  uint32_t tmem_slot;
  int abort_flag;
};

struct BwdParams {
  const int32_t* key_reach;
  const int32_t* blockmap;
  const float* lse2;          // [Hq, T_pad], -LSE * log2(e)
  const float* dd;            // [Hq, T_pad], -D
  float* dq_acc;              // [T_pad, Hq, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  // Accumulate mode (both non-null): dK (scaled) and dV are added in fp32
  // into these [T_pad, Hkv, D] rows instead of being stored as bf16, and a
  // key block whose clipped column run is empty leaves its rows untouched.
  float* dk_acc;
  float* dv_acc;
  int32_t T_pad, Hq, Hkv, nb, num_sms;
  // Query-row window [row_lo, row_hi): only these rows' gradients flow; each
  // key block's column run is clipped to the query blocks the window meets,
  // and rows outside it count as masked.
  int32_t row_lo, row_hi, windowed;
  float scale, scale_log2;
  int32_t* status;
};

// Fire-and-forget fp32 vector atomic add of four consecutive floats
// (16-byte aligned): the accumulate-mode dK/dV epilogue.
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Stages a warp's 32 rows x 32 fp32 columns (lane = row, v = that row's 32
// values) as one 4 KB box in the layout of a 128-byte-swizzled TMA box (row
// r's 16-byte chunk c at (c ^ (r & 7)) * 16, conflict-free).
__device__ __forceinline__ void stage_rows32(uint8_t* box, const uint32_t (&v)[32], int lane) {
  uint8_t* mine = box + lane * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(mine + ((c ^ (lane & 7)) << 4)) =
        make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
tree_attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq,
                     const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  if (ld_status(p.status)) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {          // the layout needs 1024-byte alignment
    if (threadIdx.x == 0) set_status(p.status, TREE_ERR_UNSUPPORTED);
    return;
  }
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BlockmapView bm{p.nb, const_cast<int32_t*>(p.blockmap)};
  const int32_t g = p.Hq / p.Hkv;
  // Launch order.  A column longer than nnz / #SMs tiles would outlast its
  // kv head's share of the run, so such "heavy" columns are launched first
  // (for every kv head); they would otherwise start late and form a tail.
  // Both the heavy and the light CTAs run kv-head-major and heaviest column
  // first (the blockmap's column order): the CTAs resident at any moment
  // mostly serve one kv head, so they stream the same Q/dO tiles and add
  // into the same dQ rows close together in time (L2 reuse).  The light
  // CTAs take the kv heads in reverse, starting with the one whose heavy
  // columns ran last.  Each thread tests one or more columns; the counts
  // are summed by the prologue barrier(s) below.
  const bool accumulate = p.dk_acc != nullptr;
  const int32_t heavy_len = bm.base[1] / (p.num_sms > 0 ? p.num_sms : 1);
  int heavy_local = 0;
  if (!accumulate)
    for (int32_t k = threadIdx.x; k < p.nb; k += kBwdThreads)
      heavy_local += (bm.col_hi()[k] - k + 1) > heavy_len;
  AbortState ab{&sm.abort_flag, p.status};

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.ew_done, 256);        // eight element-wise warps
    mbar_init(&sm.dvdk_done, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, 128);        // the dQ warpgroup
    mbar_init(&sm.dsbuf_free, 128);
    mbar_init(&sm.drain, 1);
    fence_mbar_init();
  }
  int32_t kvh, kb, qlo_c, qhi_c;         // the query blocks this CTA may walk
  if (accumulate) {
    const int32_t qlo = p.row_lo / kBlock, qhi = (p.row_hi - 1) / kBlock;
    const int32_t nsplit = (qhi - qlo + kSplitQ) / kSplitQ;
    const int32_t per_kv = (qhi + 1) * nsplit;
    kvh = blockIdx.x / per_kv;
    const int32_t rem = blockIdx.x % per_kv, c = rem % nsplit;
    kb = rem / nsplit;
    qlo_c = qlo + c * kSplitQ;
    qhi_c = min(qhi, qlo_c + kSplitQ - 1);
  } else {
    int32_t heavy_n = __syncthreads_count(heavy_local > 0);
    for (int i = 1; i * kBwdThreads < p.nb; ++i) heavy_n += __syncthreads_count(heavy_local > i);
    int32_t rank;
    if (static_cast<int32_t>(blockIdx.x) < heavy_n * p.Hkv) {
      kvh = blockIdx.x / heavy_n;
      rank = blockIdx.x % heavy_n;
    } else {
      const int32_t j = blockIdx.x - heavy_n * p.Hkv, nl = p.nb - heavy_n;
      kvh = p.Hkv - 1 - j / nl;
      rank = heavy_n + j % nl;
    }
    kb = bm.col_order()[rank];
    if (!dcheck(kb >= 0 && kb < p.nb, p.status)) return;    // CTA-uniform, before TMEM
    qlo_c = p.row_lo / kBlock;
    qhi_c = (p.row_hi - 1) / kBlock;
  }
  // the key block's column run kb..col_hi, clipped to those query blocks
  const int32_t qa_first = max(kb, qlo_c);
  const int32_t qa_last = min(bm.col_hi()[kb], qhi_c);
  const int32_t col_full_hi = bm.col_full_hi()[kb];
  const int32_t col_len = qa_last >= qa_first ? qa_last - qa_first + 1 : 0;
  const int32_t nsteps = col_len * g;
  if (accumulate && nsteps == 0) return;     // CTA-uniform: nothing to add
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_slot;
  constexpr uint32_t kTileBytes = kBlock * D * 2;
  constexpr int kHalves = D / 64;
  constexpr uint32_t kDV = 0, kDK = 128, kS = 256, kDP = 384, kDQ = 384;

  if (warp >= kWarpProducer) {
    warpgroup_regs_dec<kRegsCtl>();
    if (warp == kWarpProducer && lane == 0 && nsteps > 0) {
      // ---------------------------------------------------------- producer
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(&sm.bar_kv, 2 * kTileBytes);
      for (int hf = 0; hf < kHalves; ++hf) {
        tma_load_3d(sm.k + hf * kBlock * 64, &tm_k, &sm.bar_kv, hf * 64, kvh, kb * kBlock);
        tma_load_3d(sm.v + hf * kBlock * 64, &tm_v, &sm.bar_kv, hf * 64, kvh, kb * kBlock);
      }
      int issued = 0;
      for (int n = 0; n < nsteps; ++n) {
        const int s = n & 1;
        if (n >= 2 && !mbar_wait(&sm.empty[s], ((n >> 1) - 1) & 1, ab)) break;
        const int32_t h = kvh * g + n % g;      // query block outer, heads inner
        const int32_t qa = qa_first + n / g;
        mbar_arrive_expect_tx(&sm.full[s], 2 * kTileBytes + 2 * kBlock * 4);
        for (int hf = 0; hf < kHalves; ++hf) {
          tma_load_3d(sm.q[s] + hf * kBlock * 64, &tm_q, &sm.full[s], hf * 64, h, qa * kBlock);
          tma_load_3d(sm.dout[s] + hf * kBlock * 64, &tm_do, &sm.full[s], hf * 64, h, qa * kBlock);
        }
        const size_t row0 = static_cast<size_t>(h) * p.T_pad + qa * kBlock;
        bulk_load(sm.lse2[s], p.lse2 + row0, kBlock * 4, &sm.full[s]);
        bulk_load(sm.dd[s], p.dd + row0, kBlock * 4, &sm.full[s]);
        issued = n + 1;
      }
      if (sm.abort_flag) {
        mbar_drain(&sm.bar_kv, 0);
        for (int n = (issued > 2 ? issued - 2 : 0); n < issued; ++n)
          mbar_drain(&sm.full[n & 1], (n >> 1) & 1);
      }
    } else if (warp == kWarpMma && lane == 0 && nsteps > 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescSS = idesc_bf16_f32(kBlock, kBlock, 0, 0);   // K-major both
      constexpr uint32_t kIdescTS = idesc_bf16_f32(kBlock, D, 0, 1);        // B MN-major
      constexpr uint32_t kIdescDQ = idesc_bf16_f32(kBlock, D, 1, 1);        // A, B MN-major
      const uint32_t kbase = smem_u32(sm.k), vbase = smem_u32(sm.v), dsbase = smem_u32(sm.ds);
      bool ok = mbar_wait(&sm.bar_kv, 0, ab);
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n & 1;
        if (!(ok = mbar_wait(&sm.full[s], (n >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t qbase = smem_u32(sm.q[s]), obase = smem_u32(sm.dout[s]);
        // S^T(n) overwrites the columns that held P^T(n-1) and dS^T(n-1).  It
        // is queued behind dV(n-1) and dK(n-1), and tcgen05.mma operations of
        // one thread execute in issue order, so those reads come first and the
        // pipe is not drained here.
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBlock * 128) + (kk & 3) * 32;
          umma_ss(tbase + kS, sdesc_sw128(kbase + off, 16, 1024),
                  sdesc_sw128(qbase + off, 16, 1024), kIdescSS, kk > 0);
        }
        umma_commit(&sm.s_full);
        if (n > 0) {
          if (!(ok = mbar_wait(&sm.dq_free, (n - 1) & 1, ab))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBlock * 128) + (kk & 3) * 32;
          umma_ss(tbase + kDP, sdesc_sw128(vbase + off, 16, 1024),
                  sdesc_sw128(obase + off, 16, 1024), kIdescSS, kk > 0);
        }
        umma_commit(&sm.dp_full);
        if (!(ok = mbar_wait(&sm.ew_done, n & 1, ab))) break;
        tc_fence_after();
        // dQ first: its read-out and adds then overlap the dV/dK MMAs, and
        // the next dP^T (same TMEM columns) is not held up by them.
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk)
          umma_ss(tbase + kDQ, sdesc_sw128(dsbase + kk * 2048, kBlock * 128, 1024),
                  sdesc_sw128(kbase + kk * 2048, kBlock * 128, 1024), kIdescDQ, kk > 0);
        umma_commit(&sm.dq_full);
        // P^T for queries 0-63 sits at [256,288), 64-127 at [320,352);
        // dS^T at [288,320) and [352,384).
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint32_t pcol = kS + (kk >> 2) * 64 + (kk & 3) * 8;
          umma_ts(tbase + kDV, tbase + pcol, sdesc_sw128(obase + kk * 2048, kBlock * 128, 1024),
                  kIdescTS, (n > 0 || kk > 0));
        }
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk) {
          const uint32_t dcol = kS + 32 + (kk >> 2) * 64 + (kk & 3) * 8;
          umma_ts(tbase + kDK, tbase + dcol, sdesc_sw128(qbase + kk * 2048, kBlock * 128, 1024),
                  kIdescTS, (n > 0 || kk > 0));
        }
        umma_commit(&sm.dvdk_done);
        umma_commit(&sm.empty[s]);
      }
      if (!ok) {
        umma_commit(&sm.drain);
        mbar_drain(&sm.drain, 0);
      }
    }
  } else if (warp < kWarpEw0) {
    // --------------------------------------------------------- dQ warpgroup
    // Warp q reads dQ rows 32q .. 32q+31 (its TMEM lane quarter) in rounds
    // of 64 columns, stages each round as two 4 KB boxes in slots 2q, 2q+1
    // of the dS tile and issues their reduce-adds.  TMEM is released as soon
    // as the last round is in registers; the dS tile once the reduces have
    // read it.
    warpgroup_regs_dec<kRegsDq>();
    const int quarter = warp;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint8_t* box0 = reinterpret_cast<uint8_t*>(sm.ds) + (2 * quarter) * 4096;
    uint8_t* box1 = box0 + 4096;
    bool ok = true;
    for (int n = 0; ok && n < nsteps; ++n) {
      const int32_t h = kvh * g + n % g;
      const int32_t qa = qa_first + n / g;
      const int row0 = qa * kBlock + quarter * 32;
      if (!(ok = mbar_wait_warp(&sm.dq_full, n & 1, ab))) break;
      tc_fence_after();
#pragma unroll
      for (int rd = 0; rd < D / 64; ++rd) {
        uint32_t ra[32], rb[32];
        tmem_ld32x2(tbase + lane_off + kDQ + rd * 64, tbase + lane_off + kDQ + rd * 64 + 32, ra,
                    rb);
        if (rd == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(&sm.dq_free);       // the dQ columns are in registers
        }
        if (rd > 0) {                     // the previous round's reduces must have read the slots
          if (lane == 0) bulk_wait_read();
          __syncwarp();
        }
        stage_rows32(box0, ra, lane);
        stage_rows32(box1, rb, lane);
        fence_proxy_async_smem();         // generic-proxy writes -> visible to the bulk copy
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, box0, rd * 64, h, row0);
          tma_reduce_add_3d(&tm_dq, box1, rd * 64 + 32, h, row0);
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait_read();
      __syncwarp();
      mbar_arrive(&sm.dsbuf_free);        // the element-wise warps may rewrite the tile
    }
    // The last reduces must have landed before a later kernel reads the
    // accumulator (and have read the tile before the CTA exits).
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    // ------------------------------------------------ element-wise warps
    warpgroup_regs_inc<kRegsEw>();
    const int w = (warp - kWarpEw0) >> 2;   // query half
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;      // key row (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int32_t jkey = kb * kBlock + r;
    const int32_t reach = p.key_reach[jkey];
    bool ok = true;
    for (int n = 0; ok && n < nsteps; ++n) {
      const int s = n & 1;
      const int32_t qa = qa_first + n / g;
      // window edges count as PARTIAL: rows outside the window are masked
      const bool partial = (qa == kb) || (qa > col_full_hi) ||
                           (p.windowed && (qa * kBlock < p.row_lo || qa * kBlock + kBlock > p.row_hi));
      if (!(ok = mbar_wait_warp(&sm.s_full, n & 1, ab))) break;
      tc_fence_after();
      float pv[64];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32x2(tbase + lane_off + kS + w * 64, tbase + lane_off + kS + w * 64 + 32, ra, rb);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          pv[e] = __uint_as_float(ra[e]);
          pv[32 + e] = __uint_as_float(rb[e]);
        }
      }
      // P^T = 2^(S^T*scale*log2e - LSE*log2e) with paired FMAs; the negated
      // LSE row is read 4 at a time (broadcast).
      const float4* lse4 = reinterpret_cast<const float4*>(sm.lse2[s] + w * 64);
      const float sl2 = p.scale_log2;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = lse4[c4];
        float* x = pv + 4 * c4;
        fma2(x[0], x[1], x[0], x[1], sl2, sl2, l4.x, l4.y);
        fma2(x[2], x[3], x[2], x[3], sl2, sl2, l4.z, l4.w);
        x[0] = ex2(x[0]);
        x[1] = ex2(x[1]);
        x[2] = ex2(x[2]);
        x[3] = ex2(x[3]);
      }
      if (partial) {   // warp-uniform: only PARTIAL tiles evaluate the mask
        const int32_t q0 = qa * kBlock + w * 64;
        const int32_t lo = max(jkey, p.row_lo), hi = min(reach, p.row_hi - 1);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (!(lo <= q0 + c && q0 + c <= hi)) pv[c] = 0.f;
      }
      {
        // P^T (bf16) over the S^T columns just read, while dP^T is still
        // being computed: off the path that waits for dP^T.
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
        tmem_st32(tbase + lane_off + kS + w * 64, pk);
      }
      if (!(ok = mbar_wait_warp(&sm.dp_full, n & 1, ab))) break;
      tc_fence_after();
      uint32_t dsw[32];
      {
        const float4* dd4 = reinterpret_cast<const float4*>(sm.dd[s] + w * 64);
        uint32_t ra[32], rb[32];
        tmem_ld32x2(tbase + lane_off + kDP + w * 64, tbase + lane_off + kDP + w * 64 + 32, ra, rb);
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const uint32_t* reg = c2 == 0 ? ra : rb;
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 d4 = dd4[c2 * 8 + e4];    // -D
            const int c = c2 * 32 + 4 * e4;
            float t0, t1, t2, t3, ds0, ds1, ds2, ds3;
            add2(t0, t1, __uint_as_float(reg[4 * e4 + 0]), __uint_as_float(reg[4 * e4 + 1]),
                 d4.x, d4.y);
            add2(t2, t3, __uint_as_float(reg[4 * e4 + 2]), __uint_as_float(reg[4 * e4 + 3]),
                 d4.z, d4.w);
            mul2(ds0, ds1, pv[c + 0], pv[c + 1], t0, t1);
            mul2(ds2, ds3, pv[c + 2], pv[c + 3], t2, t3);
            dsw[c2 * 16 + 2 * e4] = pack_bf16x2(ds0, ds1);
            dsw[c2 * 16 + 2 * e4 + 1] = pack_bf16x2(ds2, ds3);
          }
        }
      }
      tmem_st32(tbase + lane_off + kS + w * 64 + 32, dsw);
      // dS^T row r, queries w*64 .. w*64+63 -> swizzled [key][query] half w.
      // The tile staged the previous pair's dQ: the dQ warps release it once
      // their reduces have read it.
      if (n > 0 && !(ok = mbar_wait_warp(&sm.dsbuf_free, (n - 1) & 1, ab))) break;
      {
        uint8_t* row = reinterpret_cast<uint8_t*>(sm.ds) + w * (kBlock * 128) + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
              make_uint4(dsw[4 * c], dsw[4 * c + 1], dsw[4 * c + 2], dsw[4 * c + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.ew_done);
    }
    // ---------------------------------------------------------- epilogue
    const size_t row_off = (static_cast<size_t>(jkey) * p.Hkv + kvh) * D + w * (D / 2);
    __nv_bfloat16* dvrow = p.dv + row_off;
    __nv_bfloat16* dkrow = p.dk + row_off;
    if (accumulate) {
      // fp32 vector atomic adds of this key row's half: the CTAs of one key
      // block's column chunks add into the same rows
      if (ok && mbar_wait_warp(&sm.dvdk_done, (nsteps - 1) & 1, ab)) {
        tc_fence_after();
        float* av = p.dv_acc + row_off;
        float* ak = p.dk_acc + row_off;
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2) {
          uint32_t rv[32], rk[32];
          tmem_ld32x2(tbase + lane_off + kDV + w * (D / 2) + c2 * 32,
                      tbase + lane_off + kDK + w * (D / 2) + c2 * 32, rv, rk);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            red_add_v4(av + c2 * 32 + e4 * 4, __uint_as_float(rv[4 * e4]),
                       __uint_as_float(rv[4 * e4 + 1]), __uint_as_float(rv[4 * e4 + 2]),
                       __uint_as_float(rv[4 * e4 + 3]));
            red_add_v4(ak + c2 * 32 + e4 * 4, __uint_as_float(rk[4 * e4]) * p.scale,
                       __uint_as_float(rk[4 * e4 + 1]) * p.scale,
                       __uint_as_float(rk[4 * e4 + 2]) * p.scale,
                       __uint_as_float(rk[4 * e4 + 3]) * p.scale);
          }
        }
      }
    } else if (D == 128 && ok && nsteps > 0 &&
               mbar_wait_warp(&sm.dvdk_done, (nsteps - 1) & 1, ab)) {
      // dV and dK through shared memory: the resident V and K tiles, whose
      // last readers (MMAs) have completed, take this warp's 32 rows of its
      // 64-column half in their own 128-byte-swizzled layout; one lane then
      // writes each with a bulk tensor store.
      tc_fence_after();
      uint8_t* sv = reinterpret_cast<uint8_t*>(sm.v) + w * (kBlock * 128);
      uint8_t* sk = reinterpret_cast<uint8_t*>(sm.k) + w * (kBlock * 128);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t rv[32], rk[32];
        tmem_ld32x2(tbase + lane_off + kDV + w * 64 + c2 * 32,
                    tbase + lane_off + kDK + w * 64 + c2 * 32, rv, rk);
#pragma unroll
        for (int e8 = 0; e8 < 4; ++e8) {
          const float* fv = reinterpret_cast<const float*>(rv + e8 * 8);
          const float* fk = reinterpret_cast<const float*>(rk + e8 * 8);
          const uint32_t off = r * 128 + (((c2 * 4 + e8) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(sv + off) =
              make_uint4(pack_bf16x2(fv[0], fv[1]), pack_bf16x2(fv[2], fv[3]),
                         pack_bf16x2(fv[4], fv[5]), pack_bf16x2(fv[6], fv[7]));
          *reinterpret_cast<uint4*>(sk + off) =
              make_uint4(pack_bf16x2(fk[0] * p.scale, fk[1] * p.scale),
                         pack_bf16x2(fk[2] * p.scale, fk[3] * p.scale),
                         pack_bf16x2(fk[4] * p.scale, fk[5] * p.scale),
                         pack_bf16x2(fk[6] * p.scale, fk[7] * p.scale));
        }
      }
      fence_proxy_async_smem();          // generic-proxy writes -> visible to the bulk copy
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm_dv, sv + quarter * 32 * 128, w * 64, kvh, kb * kBlock + quarter * 32);
        tma_store_3d(&tm_dk, sk + quarter * 32 * 128, w * 64, kvh, kb * kBlock + quarter * 32);
        bulk_commit();
        bulk_wait_read();                // the tiles must outlive the copies' reads
      }
      __syncwarp();
    } else if (ok && nsteps > 0 && mbar_wait_warp(&sm.dvdk_done, (nsteps - 1) & 1, ab)) {
      tc_fence_after();
#pragma unroll
      for (int c2 = 0; c2 < D / 64; ++c2) {
        uint32_t rv[32], rk[32];
        tmem_ld32x2(tbase + lane_off + kDV + w * (D / 2) + c2 * 32,
                    tbase + lane_off + kDK + w * (D / 2) + c2 * 32, rv, rk);
#pragma unroll
        for (int e8 = 0; e8 < 4; ++e8) {
          uint4 a, b;
          const float* fv = reinterpret_cast<const float*>(rv + e8 * 8);
          const float* fk = reinterpret_cast<const float*>(rk + e8 * 8);
          a = make_uint4(pack_bf16x2(fv[0], fv[1]), pack_bf16x2(fv[2], fv[3]),
                         pack_bf16x2(fv[4], fv[5]), pack_bf16x2(fv[6], fv[7]));
          b = make_uint4(pack_bf16x2(fk[0] * p.scale, fk[1] * p.scale),
                         pack_bf16x2(fk[2] * p.scale, fk[3] * p.scale),
                         pack_bf16x2(fk[4] * p.scale, fk[5] * p.scale),
                         pack_bf16x2(fk[6] * p.scale, fk[7] * p.scale));
          *reinterpret_cast<uint4*>(dvrow + c2 * 32 + e8 * 8) = a;
          *reinterpret_cast<uint4*>(dkrow + c2 * 32 + e8 * 8) = b;
        }
      }
    } else if (nsteps == 0) {
#pragma unroll
      for (int c = 0; c < D / 2; c += 8) {
        *reinterpret_cast<uint4*>(dvrow + c) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dkrow + c) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// a4: D rows, lse2 rows, zeroed dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256)
tree_attn_bwd_prep_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dout, const float* lse,
                          float* dd, float* lse2, float* dq_acc, int32_t T_pad, int32_t Hq,
                          int32_t row_lo, int32_t row_hi, const int32_t* status) {
  if (ld_status(status)) return;
  // One warp per (group of 8 consecutive tokens, head), heads inner: the
  // warps of a token group read consecutive 256-byte rows of O and dO, and
  // each warp reads and writes its head's 8 LSE / D entries as one 32-byte
  // sector (the per-head arrays are [Hq, T_pad]).
  const int lane = threadIdx.x & 31;
  const int32_t g_lo = row_lo >> 3, g_hi = (row_hi + 7) >> 3;
  const int64_t items = static_cast<int64_t>(g_hi - g_lo) * Hq;
  constexpr int kPer = D / 32;     // elements per lane (2 or 4)
  for (int64_t it = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; it < items;
       it += (int64_t(gridDim.x) * blockDim.x) >> 5) {
    const int32_t grp = g_lo + static_cast<int32_t>(it / Hq), h = static_cast<int32_t>(it % Hq);
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int32_t i = grp * 8 + r;
      acc[r] = 0.f;
      if (i < row_lo || i >= row_hi) continue;           // warp-uniform
      const int64_t row = static_cast<int64_t>(i) * Hq + h;
      const __nv_bfloat16* po = o + row * D + lane * kPer;
      const __nv_bfloat16* pd = dout + row * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(po + e));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(pd + e));
        acc[r] += a.x * b.x + a.y * b.y;
      }
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D);
      for (int c = lane; c < D / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    if (lane < 8) {
      const int32_t i = grp * 8 + lane;
      float mine = acc[0];
#pragma unroll
      for (int r = 1; r < 8; ++r) mine = lane == r ? acc[r] : mine;
      if (i >= row_lo && i < row_hi) {
        // stored negated so the main kernel's paired FMA/add consume them directly
        const int64_t hi = static_cast<int64_t>(h) * T_pad + i;
        dd[hi] = -mine;
        lse2[hi] = -lse[hi] * 1.4426950408889634f;
      }
    }
  }
}

// a6: dQ = bf16(scale * acc), 8 elements per thread.
__global__ void __launch_bounds__(256)
tree_attn_bwd_dq_kernel(const float* dq_acc, __nv_bfloat16* dq, int64_t t_lo, int64_t t_hi,
                        float scale, const int32_t* status) {
  if (ld_status(status)) return;
  for (int64_t t = t_lo + blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < t_hi;
       t += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
    reinterpret_cast<uint4*>(dq)[t] =
        make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                   pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
  }
}

struct BwdWorkspace {
  float* dq_acc;   // [T_pad, Hq, D]
  float* dd;       // [Hq, T_pad]
  float* lse2;     // [Hq, T_pad]
};

BwdWorkspace carve(void* workspace, int32_t T_pad, int32_t Hq, int32_t d) {
  const size_t rows = static_cast<size_t>(T_pad) * Hq;
  BwdWorkspace w;
  w.dq_acc = static_cast<float*>(workspace);
  w.dd = w.dq_acc + rows * d;
  w.lse2 = w.dd + rows;
  return w;
}

int grid_cap(int64_t blocks, int num_sms) {
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

size_t attn_bwd_workspace_bytes(int32_t T_pad, int32_t Hq, int32_t d) {
  const size_t rows = static_cast<size_t>(T_pad) * Hq;
  return rows * d * sizeof(float) + 2 * rows * sizeof(float);
}

cudaError_t launch_attn_bwd_prepare(const void* o, const void* d_o, const float* lse,
                                    int32_t T_pad, int32_t Hq, int32_t d, void* workspace,
                                    int32_t* status, cudaStream_t s, int num_sms,
                                    int32_t row_lo, int32_t row_hi) {
  BwdWorkspace w = carve(workspace, T_pad, Hq, d);
  if (row_hi <= row_lo) return cudaSuccess;
  const int64_t items = static_cast<int64_t>(((row_hi + 7) >> 3) - (row_lo >> 3)) * Hq;
  const int blocks = grid_cap((items * 32 + 255) / 256, num_sms);
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pd = static_cast<const __nv_bfloat16*>(d_o);
  if (d == 64)
    tree_attn_bwd_prep_kernel<64><<<blocks, 256, 0, s>>>(po, pd, lse, w.dd, w.lse2, w.dq_acc,
                                                         T_pad, Hq, row_lo, row_hi, status);
  else
    tree_attn_bwd_prep_kernel<128><<<blocks, 256, 0, s>>>(po, pd, lse, w.dd, w.lse2, w.dq_acc,
                                                          T_pad, Hq, row_lo, row_hi, status);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo,
                                 const CUtensorMap& tdq, const CUtensorMap& tdk,
                                 const CUtensorMap& tdv, const int32_t* key_reach,
                                 const void* blockmap, int32_t T_pad, int32_t Hq, int32_t Hkv,
                                 int32_t d, float scale, void* dk, void* dv, void* workspace,
                                 int32_t* status, cudaStream_t s, int num_sms, int32_t row_lo,
                                 int32_t row_hi, float* dk_acc, float* dv_acc) {
  BwdWorkspace w = carve(workspace, T_pad, Hq, d);
  if (row_hi <= row_lo) return cudaSuccess;
  BwdParams p;
  p.key_reach = key_reach;
  p.blockmap = static_cast<const int32_t*>(blockmap);
  p.lse2 = w.lse2;
  p.dd = w.dd;
  p.dq_acc = w.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dk_acc = dk_acc;
  p.dv_acc = dv_acc;
  p.row_lo = row_lo;
  p.row_hi = row_hi;
  p.windowed = (row_lo > 0 || row_hi < T_pad) ? 1 : 0;
  p.T_pad = T_pad;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.nb = T_pad / kBlock;
  p.num_sms = num_sms;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  // accumulate mode: (kv head, key block up to the window's last query
  // block, chunk of kSplitQ window query blocks); else (kv head, key block)
  const int32_t qlo = row_lo / kBlock, qhi = (row_hi - 1) / kBlock;
  const int grid = dk_acc ? Hkv * (qhi + 1) * ((qhi - qlo + kSplitQ) / kSplitQ) : p.nb * Hkv;
  cudaError_t e;
  if (d == 64) {
    e = cudaFuncSetAttribute(tree_attn_bwd_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(BwdSmem<64>)));
    if (e != cudaSuccess) return e;
    tree_attn_bwd_kernel<64><<<grid, kBwdThreads, sizeof(BwdSmem<64>), s>>>(tq, tk, tv, tdo, tdq,
                                                                          tdk, tdv, p);
  } else {
    e = cudaFuncSetAttribute(tree_attn_bwd_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(BwdSmem<128>)));
    if (e != cudaSuccess) return e;
    tree_attn_bwd_kernel<128><<<grid, kBwdThreads, sizeof(BwdSmem<128>), s>>>(tq, tk, tv, tdo,
                                                                            tdq, tdk, tdv, p);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_finish(int32_t T_pad, int32_t Hq, int32_t d, float scale,
                                   void* workspace, void* dq, int32_t* status, cudaStream_t s,
                                   int num_sms, int32_t row_lo, int32_t row_hi) {
  BwdWorkspace w = carve(workspace, T_pad, Hq, d);
  if (row_hi <= row_lo) return cudaSuccess;
  // groups of 8 elements; a token row holds Hq * d (a multiple of 64) of them
  const int64_t per_row8 = static_cast<int64_t>(Hq) * d / 8;
  const int64_t t_lo = row_lo * per_row8, t_hi = row_hi * per_row8;
  tree_attn_bwd_dq_kernel<<<grid_cap((t_hi - t_lo + 255) / 256, num_sms), 256, 0, s>>>(
      w.dq_acc, static_cast<__nv_bfloat16*>(dq), t_lo, t_hi, scale, status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace tree
