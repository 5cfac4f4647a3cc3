// Row statistics of next-token logits and the predicting-row search, shared
// by the log-prob gather over materialised logits and the fused LM head.
//
// A row's log-sum-exp and entropy are reduced in one pass as a running max m,
// s = sum 2^u and t = sum 2^u u with u = (x - m) log2(e): then
// lse = m + ln s and entropy = ln 2 (log2 s - t / s).  Partial results over
// slices of a row merge by moving both to the larger m.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace tree {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t min_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Running reduction of one row slice.  s and t are kept as two lanes each
// so the per-element updates pair up into f32x2 instructions.
struct Acc {
  float m, s0, s1, t0, t1, mn;
};

__device__ __forceinline__ void acc_init(Acc& a) {
  a.m = -INFINITY;
  a.s0 = a.s1 = a.t0 = a.t1 = 0.f;
  a.mn = INFINITY;
}

// Move the reference of (s, t) from a.m to m_new >= a.m:
// u' = u + d with d = (a.m - m_new) log2(e), so s' = 2^d s and
// t' = 2^d (t + d s).  Nothing accumulated yet (s == 0) needs no scaling.
__device__ __forceinline__ void acc_rebase(Acc& a, float m_new) {
  if (a.s0 + a.s1 > 0.f) {
    const float d = (a.m - m_new) * kLog2e;
    const float f = ex2f(d);
    a.t0 = f * fmaf(d, a.s0, a.t0);
    a.t1 = f * fmaf(d, a.s1, a.t1);
    a.s0 *= f;
    a.s1 *= f;
  }
  a.m = m_new;
}

// Two logits (x0, x1) at the current reference.
__device__ __forceinline__ void acc_pair(Acc& a, float nmL, float x0, float x1) {
  float u0, u1, e0, e1;
  fma2(u0, u1, x0, x1, kLog2e, kLog2e, nmL, nmL);
  e0 = ex2f(u0);
  e1 = ex2f(u1);
  fma2(a.t0, a.t1, e0, e1, u0, u1, a.t0, a.t1);
  add2(a.s0, a.s1, a.s0, a.s1, e0, e1);
}

// One logit of the ragged tail or of an unaligned row.
__device__ __forceinline__ void acc_one(Acc& a, float x) {
  a.mn = fminf(a.mn, x);
  if (x > a.m) acc_rebase(a, x);
  const float u = fmaf(x, kLog2e, -a.m * kLog2e);
  const float e = ex2f(u);
  a.s0 += e;
  a.t0 = fmaf(e, u, a.t0);
}

__device__ __forceinline__ void acc_merge(Acc& a, const Acc& b) {
  Acc c = b;
  const float m = fmaxf(a.m, c.m);
  acc_rebase(a, m);
  acc_rebase(c, m);
  a.s0 = (a.s0 + a.s1) + (c.s0 + c.s1);
  a.t0 = (a.t0 + a.t1) + (c.t0 + c.t1);
  a.s1 = 0.f;
  a.t1 = 0.f;
  a.mn = fminf(a.mn, c.mn);
}

__device__ __forceinline__ Acc acc_shfl_xor(const Acc& a, int o) {
  Acc b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  b.s0 = __shfl_xor_sync(0xffffffffu, a.s0, o);
  b.s1 = __shfl_xor_sync(0xffffffffu, a.s1, o);
  b.t0 = __shfl_xor_sync(0xffffffffu, a.t0, o);
  b.t1 = __shfl_xor_sync(0xffffffffu, a.t1, o);
  b.mn = __shfl_xor_sync(0xffffffffu, a.mn, o);
  return b;
}

// Largest i < q with reach[i] >= q (q - 1 is known to fail), or -1.
// Called by all 32 lanes of a warp with the same q; returns the same value
// on every lane.
__device__ inline int32_t find_pred(int32_t q, const int32_t* __restrict__ reach,
                             const int32_t* __restrict__ col_hi, int lane) {
  const int32_t qb = q >> 7;
  const int32_t lo = qb << 7;
  for (int32_t top = q - 2; top >= lo; top -= 32) {        // q's own block
    const int32_t i = top - lane;
    const bool hit = i >= lo && reach[i] >= q;
    const uint32_t b = __ballot_sync(0xffffffffu, hit);
    if (b) return top - (__ffs(b) - 1);
  }
  for (int32_t btop = qb - 1; btop >= 0; btop -= 32) {     // earlier blocks
    const int32_t bl = btop - lane;
    const bool cand = bl >= 0 && col_hi[bl] >= qb;
    uint32_t cb = __ballot_sync(0xffffffffu, cand);
    while (cb) {
      const int l = __ffs(cb) - 1;
      cb &= cb - 1;
      const int32_t blk = btop - l;                        // highest block first
      for (int w = 0; w < kBlock / 32; ++w) {
        const int32_t top = blk * kBlock + kBlock - 1 - w * 32;
        const uint32_t b = __ballot_sync(0xffffffffu, reach[top - lane] >= q);
        if (b) return top - (__ffs(b) - 1);
      }
    }
  }
  return -1;
}

}  // namespace tree
