// tree_pack_positions: per-key reach and position ids (integer, exact).
//
// AReaL Tree Training guide, section "打包数据的生成": the position id of a
// token is the number of tokens it may attend to, minus one.  The packing
// figure fixes the mask: j visible to i iff j <= i and node(j) is node(i) or
// an ancestor.  In a preorder layout (node tokens contiguous, nodes in rank
// order, a subtree's nodes a contiguous rank range [entry, exit]) the tokens
// of the subtree of node(j) are one contiguous run that ends at
//   key_reach[j] = last token of the node ranked node_exit[node(j)],
// so  visible(i, j)  <=>  j <= i <= key_reach[j]  and
//   position_ids[i] + 1 = #{ j : j <= i <= key_reach[j] }
// is an inclusive scan of D with D[j] += 1 for every real key and
// D[key_reach[j] + 1] -= 1; the -1 terms are summed per node (one atomic per
// node instead of one per token).
//
// Kernels (all skip their work once *dev_status is non-zero):
//  1 init         scratch arrays
//  2 nodes_a      range checks, rank -> node map (duplicate ranks flagged)
//  3 tokens_a     node-id range; first/last token and run count per node
//  4 nodes_b      one run per node, rank order, nested subtree ranges
//                 (children chain of every node stays inside it), node reach,
//                 the per-node -cnt term of D
//  5 scan_tiles   per-tile sums of D (+1 per real token)
//  6 scan_top     exclusive scan of tile sums (one CTA)
//  7 finalize     inclusive scan -> position ids and key_reach; a pad whose
//                 count is non-zero lies inside a subtree span -> malformed
#include <climits>
#include <mutex>

#include "common.cuh"

namespace tree {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;   // 2048 tokens per CTA
constexpr int kMalformed = TREE_ERR_MALFORMED_TREE;

struct PosWS {
  int32_t* rank_node;      // [N]   node with a given preorder rank
  int32_t* exit_by_rank;   // [N]   node_exit of the node with a given rank
  int32_t* first_tok;      // [N]
  int32_t* last_tok;       // [N]
  int32_t* runs;           // [N]   number of contiguous token runs
  int32_t* node_reach;     // [N]   last token of the subtree
  int32_t* diff;           // [T_pad + 1]
  int32_t* tile_sums;      // [n_tiles + 1]
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

PosWS carve(void* ws, int32_t T_pad, int32_t N) {
  char* p = static_cast<char*>(ws);
  PosWS w;
  int32_t** arrays[6] = {&w.rank_node, &w.exit_by_rank, &w.first_tok,
                         &w.last_tok,  &w.runs,         &w.node_reach};
  for (auto a : arrays) {
    *a = reinterpret_cast<int32_t*>(p);
    p += align256(sizeof(int32_t) * static_cast<size_t>(N > 0 ? N : 1));
  }
  w.diff = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (static_cast<size_t>(T_pad) + 1));
  w.tile_sums = reinterpret_cast<int32_t*>(p);
  return w;
}

__global__ void k_init(PosWS w, int32_t T_pad, int32_t N, const int32_t* status) {
  if (ld_status(status)) return;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i <= T_pad;
       i += int64_t(gridDim.x) * blockDim.x) {
    if (i < N) {
      w.rank_node[i] = -1;
      w.first_tok[i] = INT_MAX;
      w.last_tok[i] = -1;
      w.runs[i] = 0;
    }
    w.diff[i] = 0;
  }
}

__global__ void k_nodes_a(PosWS w, const int32_t* entry, const int32_t* exit_, int32_t N,
                          int32_t* status) {
  if (ld_status(status)) return;
  int32_t n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  int32_t e = entry[n], x = exit_[n];
  if (e < 0 || e >= N || x < e || x >= N) {
    set_status(status, kMalformed);
    return;
  }
  if (atomicExch(&w.rank_node[e], n) != -1) set_status(status, kMalformed);
  w.exit_by_rank[e] = x;
}

__global__ void k_tokens_a(PosWS w, const int32_t* token_node, int32_t T_pad, int32_t N,
                           int32_t* status) {
  if (ld_status(status)) return;
  int32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= T_pad) return;
  int32_t n = token_node[j];
  if (n < -1 || n >= N) {
    set_status(status, kMalformed);
    return;
  }
  if (n < 0) return;
  int32_t prev = j > 0 ? token_node[j - 1] : -1;
  int32_t next = j + 1 < T_pad ? token_node[j + 1] : -1;
  if (prev != n) {                 // start of a run of node n
    atomicMin(&w.first_tok[n], j);
    atomicAdd(&w.runs[n], 1);
  }
  if (next != n) atomicMax(&w.last_tok[n], j);
}

__global__ void k_nodes_b(PosWS w, const int32_t* entry, const int32_t* exit_, int32_t N,
                          int32_t T_pad, int32_t* status) {
  if (ld_status(status)) return;
  int32_t n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  if (w.runs[n] != 1) {            // empty node, or tokens split in several runs
    set_status(status, kMalformed);
    return;
  }
  const int32_t r = entry[n], x = exit_[n];
  const int32_t first = w.first_tok[n], last = w.last_tok[n];
  if (r > 0 && first <= w.last_tok[w.rank_node[r - 1]]) {   // nodes out of rank order
    set_status(status, kMalformed);
    return;
  }
  // Children of rank r are r+1, exit(r+1)+1, ...: each must stay inside [r, x].
  for (int32_t c = r + 1; c <= x;) {
    int32_t xc = w.exit_by_rank[c];
    if (xc > x) {
      set_status(status, kMalformed);
      return;
    }
    c = xc + 1;
  }
  const int32_t reach = w.last_tok[w.rank_node[x]];
  w.node_reach[n] = reach;
  if (reach + 1 < T_pad) atomicSub(&w.diff[reach + 1], last - first + 1);
}

__device__ __forceinline__ int32_t d_value(const int32_t* token_node, const PosWS& w,
                                           int32_t j) {
  return (token_node[j] >= 0 ? 1 : 0) + w.diff[j];
}

// Block-wide inclusive scan of one int per thread; returns the block total.
__device__ int32_t block_scan_incl(int32_t v, int32_t& incl) {
  __shared__ int32_t warp_tot[kScanThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int32_t t = lane < kScanThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kScanThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  incl = x + (wid > 0 ? warp_tot[wid - 1] : 0);
  int32_t total = warp_tot[kScanThreads / 32 - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kScanThreads)
k_scan_tiles(PosWS w, const int32_t* token_node, int32_t T_pad, const int32_t* status) {
  if (ld_status(status)) return;
  const int32_t base = blockIdx.x * kScanTile + threadIdx.x * kScanItems;
  int32_t sum = 0;
#pragma unroll
  for (int t = 0; t < kScanItems; ++t)
    if (base + t < T_pad) sum += d_value(token_node, w, base + t);
  int32_t incl;
  int32_t total = block_scan_incl(sum, incl);
  if (threadIdx.x == 0) w.tile_sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads)
k_scan_top(PosWS w, int32_t n_tiles, const int32_t* status) {
  if (ld_status(status)) return;
  int32_t carry = 0;
  for (int32_t b0 = 0; b0 < n_tiles; b0 += kScanThreads) {
    int32_t b = b0 + threadIdx.x;
    int32_t v = b < n_tiles ? w.tile_sums[b] : 0;
    int32_t incl;
    int32_t total = block_scan_incl(v, incl);
    if (b < n_tiles) w.tile_sums[b] = carry + incl - v;   // exclusive
    carry += total;
  }
}

__global__ void __launch_bounds__(kScanThreads)
k_finalize(PosWS w, const int32_t* token_node, int32_t T_pad, int32_t* position_ids,
           int32_t* key_reach, int32_t* status) {
  if (ld_status(status)) return;
  const int32_t base = blockIdx.x * kScanTile + threadIdx.x * kScanItems;
  int32_t v[kScanItems];
  int32_t sum = 0;
#pragma unroll
  for (int t = 0; t < kScanItems; ++t) {
    v[t] = base + t < T_pad ? d_value(token_node, w, base + t) : 0;
    sum += v[t];
  }
  int32_t incl;
  block_scan_incl(sum, incl);
  int32_t run = w.tile_sums[blockIdx.x] + incl - sum;
  bool bad = false;
#pragma unroll
  for (int t = 0; t < kScanItems; ++t) {
    int32_t j = base + t;
    if (j >= T_pad) break;
    run += v[t];
    int32_t n = token_node[j];
    if (n >= 0) {
      position_ids[j] = run - 1;
      key_reach[j] = w.node_reach[n];
    } else {
      position_ids[j] = 0;
      key_reach[j] = j - 1;
      if (run != 0) bad = true;    // pad inside some subtree's token span
    }
  }
  if (bad) set_status(status, kMalformed);
}

}  // namespace

size_t pack_positions_workspace_bytes(int32_t T_pad, int32_t n_nodes) {
  const size_t N = static_cast<size_t>(n_nodes > 0 ? n_nodes : 1);
  const size_t n_tiles = (static_cast<size_t>(T_pad) + kScanTile - 1) / kScanTile;
  return 6 * align256(sizeof(int32_t) * N) +
         align256(sizeof(int32_t) * (static_cast<size_t>(T_pad) + 1)) +
         align256(sizeof(int32_t) * (n_tiles + 1));
}

cudaError_t launch_pack_positions(const int32_t* token_node, int32_t T_pad,
                                  const int32_t* node_entry, const int32_t* node_exit,
                                  int32_t N, int32_t* position_ids, int32_t* key_reach,
                                  void* workspace, int32_t* status, cudaStream_t s) {
  PosWS w = carve(workspace, T_pad, N);
  const int threads = 256;
  const int n_tiles = (T_pad + kScanTile - 1) / kScanTile;
  const int init_blocks = (T_pad + 1 + threads - 1) / threads;
  k_init<<<init_blocks < 1024 ? init_blocks : 1024, threads, 0, s>>>(w, T_pad, N, status);
  if (N > 0) k_nodes_a<<<(N + threads - 1) / threads, threads, 0, s>>>(w, node_entry, node_exit, N, status);
  k_tokens_a<<<(T_pad + threads - 1) / threads, threads, 0, s>>>(w, token_node, T_pad, N, status);
  if (N > 0)
    k_nodes_b<<<(N + threads - 1) / threads, threads, 0, s>>>(w, node_entry, node_exit, N,
                                                              T_pad, status);
  k_scan_tiles<<<n_tiles, kScanThreads, 0, s>>>(w, token_node, T_pad, status);
  k_scan_top<<<1, kScanThreads, 0, s>>>(w, n_tiles, status);
  k_finalize<<<n_tiles, kScanThreads, 0, s>>>(w, token_node, T_pad, position_ids, key_reach,
                                              status);
  count_launches(N > 0 ? 7 : 5);
  return cudaGetLastError();
}

}  // namespace tree

// ---------------------------------------------------------------------------
// tree_pack_positions_noalloc: the same kernels with their scratch in a
// file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory: a plugin or custom operator
// running inside a host framework that owns all device memory hands its
// kernels only their input and output buffers, so there is nowhere to get a
// workspace from.  For them this entry point keeps the scratch of
// tree_pack_positions in `g_positions_scratch`, a fixed 1.75 MiB array that
// every GPU loading the library holds until the process exits.  The host
// cannot pass the array's name to a kernel (in host code it names a host-side
// stand-in, not device memory), so the first call on each device looks up the
// device address with cudaGetSymbolAddress, with that device current, and
// caches it together with the CUDA context it belongs to; make that first
// call before any stream capture.  A later call that finds a different
// context current (the primary context was reset or torn down and created
// again) looks the address up again, so no call ever launches with an
// address from a context that no longer exists.
namespace tree {
namespace {

constexpr int32_t kNoAllocMaxTokens = 65536;
constexpr int32_t kNoAllocMaxNodes = 65536;
constexpr size_t kNoAllocScratchBytes =
    6 * ((sizeof(int32_t) * kNoAllocMaxNodes + 255) / 256 * 256) +
    (sizeof(int32_t) * (kNoAllocMaxTokens + 1) + 255) / 256 * 256 +
    (sizeof(int32_t) * ((kNoAllocMaxTokens + kScanTile - 1) / kScanTile + 1) + 255) / 256 * 256;

__device__ __align__(256) uint8_t g_positions_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
  void* ctx = nullptr;    // CUDA context the address was looked up in
  void* addr = nullptr;   // device address of g_positions_scratch there
};
ScratchEntry g_scratch[kMaxDevices];

// The driver's cuCtxGetCurrent, resolved once through the runtime (the
// library does not link libcuda).
using CtxGetCurrentFn = int (*)(void**);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_positions_scratch on the current device, looked up
// once per (device, context).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (!get_ctx) return cudaErrorDeviceUninitialized;
  void* ctx = nullptr;
  if (get_ctx(&ctx) != 0) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  // No context current yet on this thread (the runtime makes the primary
  // context current lazily), or a different one: look the address up again.
  // The lookup itself makes the device's primary context current.
  if (!ent.addr || !ctx || ent.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_positions_scratch);
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
    ent.ctx = ctx;
    ent.addr = p;
  }
  *out = ent.addr;
  return cudaSuccess;
}

}  // namespace
}  // namespace tree

extern "C" tree_status_t tree_pack_positions_noalloc(const int32_t* token_node, int32_t T_pad,
                                                     const int32_t* node_entry,
                                                     const int32_t* node_exit, int32_t n_nodes,
                                                     int32_t* position_ids, int32_t* key_reach,
                                                     int32_t* dev_status, tree_stream_t stream) {
  if (T_pad < 0 || n_nodes < 0 || !dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad % tree::kBlock) return TREE_ERR_ALIGNMENT;
  if (T_pad > tree::kNoAllocMaxTokens || n_nodes > tree::kNoAllocMaxNodes)
    return TREE_ERR_WORKSPACE;   // beyond the fixed scratch array
  if (T_pad == 0) return TREE_OK;
  if (!token_node || !position_ids || !key_reach || (n_nodes > 0 && (!node_entry || !node_exit)))
    return TREE_ERR_INVALID_ARG;
  if (n_nodes > T_pad) return TREE_ERR_INVALID_ARG;
  if (tree::pack_positions_workspace_bytes(T_pad, n_nodes) > tree::kNoAllocScratchBytes)
    return TREE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (tree::scratch_address(&scratch) != cudaSuccess) return TREE_ERR_CUDA;
  // Every call re-initialises the scratch it uses (the first kernel), so the
  // previous call's contents never leak into this one.  Calls that overlap on
  // the GPU (different streams, or different host threads on one device)
  // share this one array and race: serialise them.
  cudaError_t e = tree::launch_pack_positions(token_node, T_pad, node_entry, node_exit, n_nodes,
                                              position_ids, key_reach, scratch, dev_status,
                                              stream);
  return e == cudaSuccess ? TREE_OK : TREE_ERR_CUDA;
}
