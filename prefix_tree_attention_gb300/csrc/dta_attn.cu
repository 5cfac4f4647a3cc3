// Element-wise kernels around the depth-first execution of dynamic tree
// attention (AREAL-DTA, sections 3.1-3.2) on the packed layout.
//
// Each operation of the traversal is the packed tree attention restricted to
// a window of query rows (the stack at a chunk's forward holds exactly the
// chunk's ancestor tokens, which are the keys the packed mask lets it see),
// so the forward and backward kernels run with a row window.  Across
// operations dK and dV accumulate in fp32 (a popped node's keys have by then
// received the gradient of every descendant), and two kernels bracket the
// whole traversal:
//   k_dta_init     O = 0, LSE = -inf, dQ = 0 for every row, and the whole
//                  fp32 workspace (dQ accumulator, D and LSE rows, dK/dV
//                  accumulators) = 0.  Pads are never scheduled and keep these
//                  values.  The rows of a 128-row block outside an
//                  operation's window are masked, but the backward still
//                  reads their D and LSE entries: zeroing keeps every entry
//                  finite (0 or a value some operation wrote), so a masked
//                  P = 0 gives dS = 0 exactly.
//   k_dta_finish   dK, dV = bf16(accumulators)
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace tree {
namespace {

__global__ void __launch_bounds__(256)
k_dta_init(uint4* o16, int64_t n_o16, uint4* dq16, int64_t n_dq16, float* lse, int64_t n_lse,
           float4* ws4, int64_t n_ws4, const int32_t* status) {
  if (ld_status(status)) return;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t t0 = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  for (int64_t t = t0; t < n_o16; t += stride) o16[t] = make_uint4(0, 0, 0, 0);
  for (int64_t t = t0; t < n_dq16; t += stride) dq16[t] = make_uint4(0, 0, 0, 0);
  for (int64_t t = t0; t < n_lse; t += stride) lse[t] = -INFINITY;
  for (int64_t t = t0; t < n_ws4; t += stride) ws4[t] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// 8 elements per step: two float4 of each accumulator -> one uint4 of bf16.
__global__ void __launch_bounds__(256)
k_dta_finish(const float4* dk_acc, const float4* dv_acc, uint4* dk, uint4* dv, int64_t n8,
             const int32_t* status) {
  if (ld_status(status)) return;
  for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < n8;
       t += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = dk_acc[2 * t], b = dk_acc[2 * t + 1];
    dk[t] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                       pack_bf16x2(b.z, b.w));
    const float4 c = dv_acc[2 * t], e = dv_acc[2 * t + 1];
    dv[t] = make_uint4(pack_bf16x2(c.x, c.y), pack_bf16x2(c.z, c.w), pack_bf16x2(e.x, e.y),
                       pack_bf16x2(e.z, e.w));
  }
}

int grid_for(int64_t work, int num_sms) {
  const int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t launch_dta_init(void* o, void* dq, float* lse, void* workspace, size_t ws_bytes,
                            int32_t T_pad, int32_t Hq, int32_t d, int32_t* status,
                            cudaStream_t s, int num_sms) {
  const int64_t n_o16 = static_cast<int64_t>(T_pad) * Hq * d / 8;   // 16-byte groups of bf16
  const int64_t n_ws4 = static_cast<int64_t>(ws_bytes / 16);
  const int64_t most = n_o16 > n_ws4 ? n_o16 : n_ws4;
  k_dta_init<<<grid_for(most, num_sms), 256, 0, s>>>(
      static_cast<uint4*>(o), n_o16, static_cast<uint4*>(dq), n_o16, lse,
      static_cast<int64_t>(Hq) * T_pad, static_cast<float4*>(workspace), n_ws4, status);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dta_finish(const float* dk_acc, const float* dv_acc, void* dk, void* dv,
                              int32_t T_pad, int32_t Hkv, int32_t d, int32_t* status,
                              cudaStream_t s, int num_sms) {
  const int64_t n8 = static_cast<int64_t>(T_pad) * Hkv * d / 8;
  k_dta_finish<<<grid_for(n8, num_sms), 256, 0, s>>>(
      reinterpret_cast<const float4*>(dk_acc), reinterpret_cast<const float4*>(dv_acc),
      static_cast<uint4*>(dk), static_cast<uint4*>(dv), n8, status);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace tree
