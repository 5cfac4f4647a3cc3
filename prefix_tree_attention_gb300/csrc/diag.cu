// tree_debug_wait_timeout: exercises the bounded mbarrier wait that guards
// every pipeline wait in the attention kernels.  One thread waits on a
// shared-memory barrier that nothing ever arrives on; the wait gives up after
// `limit_ns`, records TREE_ERR_TIMEOUT in the status word and returns, so the
// CUDA context stays usable.  Used by the failure-detection tests.
#include "common.cuh"
#include "ptx.cuh"

namespace tree {
namespace {

__global__ void k_wait_probe(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  AbortState ab{&flag, status, limit_ns};
  mbar_wait_warp(&bar, 0, ab);   // never completes: runs out of time
}

}  // namespace
}  // namespace tree

extern "C" tree_status_t tree_debug_wait_timeout(int32_t* dev_status, int64_t limit_ns,
                                                 tree_stream_t stream) {
  if (!dev_status || limit_ns < 1000000 || limit_ns > 2000000000) return TREE_ERR_INVALID_ARG;
  tree::k_wait_probe<<<1, 32, 0, stream>>>(dev_status, static_cast<uint64_t>(limit_ns));
  tree::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TREE_OK : TREE_ERR_CUDA;
}
