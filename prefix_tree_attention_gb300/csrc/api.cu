// C ABI of the library (declared in include/tree_attn.h): argument checks,
// TMA tensor-map encoding and kernel launches.  No allocation, no
// synchronisation: every call only queues work on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace tree {
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const int32_t* key_reach, const void* blockmap, int32_t T_pad,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale, void* o, float* lse,
                            int32_t* status, cudaStream_t s, int32_t row_lo, int32_t row_hi);
size_t attn_bwd_workspace_bytes(int32_t T_pad, int32_t Hq, int32_t d);
cudaError_t launch_attn_bwd_prepare(const void* o, const void* d_o, const float* lse,
                                    int32_t T_pad, int32_t Hq, int32_t d, void* workspace,
                                    int32_t* status, cudaStream_t s, int num_sms, int32_t row_lo,
                                    int32_t row_hi);
cudaError_t launch_attn_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo,
                                 const CUtensorMap& tdq, const CUtensorMap& tdk,
                                 const CUtensorMap& tdv, const int32_t* key_reach,
                                 const void* blockmap, int32_t T_pad, int32_t Hq, int32_t Hkv,
                                 int32_t d, float scale, void* dk, void* dv, void* workspace,
                                 int32_t* status, cudaStream_t s, int num_sms, int32_t row_lo,
                                 int32_t row_hi, float* dk_acc, float* dv_acc);
cudaError_t launch_attn_bwd_finish(int32_t T_pad, int32_t Hq, int32_t d, float scale,
                                   void* workspace, void* dq, int32_t* status, cudaStream_t s,
                                   int num_sms, int32_t row_lo, int32_t row_hi);
cudaError_t launch_dta_init(void* o, void* dq, float* lse, void* workspace, size_t ws_bytes,
                            int32_t T_pad, int32_t Hq, int32_t d, int32_t* status,
                            cudaStream_t s, int num_sms);
cudaError_t launch_dta_finish(const float* dk_acc, const float* dv_acc, void* dk, void* dv,
                              int32_t T_pad, int32_t Hkv, int32_t d, int32_t* status,
                              cudaStream_t s, int num_sms);
size_t lm_head_workspace_bytes(int32_t T_pad, int32_t V);
cudaError_t launch_lm_head(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const void* hidden,
                           const void* weight, int32_t T_pad, int32_t H, int32_t V,
                           const int32_t* token_ids, const int32_t* key_reach,
                           const void* blockmap, float* lse, float* entropy, float* vmin,
                           float* vmax, float* logprob, int32_t* token_pred, void* workspace,
                           int32_t* status, cudaStream_t s, int num_sms);
cudaError_t launch_lm_head_grad(const CUtensorMap& tm_h, const CUtensorMap& tm_w,
                                const CUtensorMap& tm_g, const void* hidden, const void* weight,
                                int32_t T_pad, int32_t H,
                                int32_t V, int32_t row_lo, int32_t row_hi,
                                const int32_t* token_ids, const int32_t* key_reach,
                                const float* lse, const float* entropy, const float* g_lp,
                                const float* g_ent, void* grad, int64_t ldg, void* workspace,
                                int32_t* status, cudaStream_t s, int num_sms);

namespace {
std::atomic<uint64_t> g_launches{0};
}
void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }
uint64_t launches_total() { return g_launches.load(); }
}  // namespace tree

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The softmax scale must be a positive finite number: the kernels take the
// row max of the raw scores before scaling, which needs scale > 0.
bool valid_scale(float scale) { return scale > 0.f && scale <= 3.0e38f; }

// The driver's tensor-map encoder, resolved once through the runtime so the
// library itself does not link libcuda (it loads on machines without a GPU).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Token-major [T, H, d] bf16 tensor viewed as a 3-D TMA map with a
// 64-element (128-byte) x 1 head x box_rows-token box (128 for the operand
// loads, 32 for the forward's per-warp O stores), 128-byte swizzle.
bool encode_map(CUtensorMap* map, const void* base, int32_t T, int32_t H, int32_t d,
                uint32_t box_rows = tree::kBlock) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t elem[3] = {1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                      const_cast<void*>(base), dims, strides, box, elem,
                                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The fp32 dQ accumulator [T, H, d] as a 3-D TMA map for reduce-add stores:
// 32-float (128-byte) x 1 head x 32-token box, 128-byte swizzle.
bool encode_map_acc(CUtensorMap* map, void* base, int32_t T, int32_t H, int32_t d) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[3] = {32, 1, 32};
  cuuint32_t elem[3] = {1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A row-major [rows, cols] bf16 matrix as a 2-D TMA map with a 64-column
// (128-byte) x box_rows box, 128-byte swizzle; rows past the end read as 0.
bool encode_map_2d(CUtensorMap* map, const void* base, int64_t rows, int32_t cols,
                   uint32_t box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t elem[2] = {1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The bf16 logits gradient [rows, V] (row stride ld elements) as a 2-D
// TMA map for stores of 32 x 32 boxes, 64-byte swizzle; columns past V and
// rows past the chunk are not written.
bool encode_map_grad(CUtensorMap* map, void* base, int32_t rows, int32_t V, int64_t ld) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t elem[2] = {1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

tree_status_t check_attn_shape(int32_t T_pad, int32_t Hq, int32_t Hkv, int32_t d) {
  if (T_pad < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return TREE_ERR_INVALID_ARG;
  if (T_pad % tree::kBlock) return TREE_ERR_ALIGNMENT;
  if (d != 64 && d != 128) return TREE_ERR_UNSUPPORTED;
  return TREE_OK;
}

tree_status_t cuda_result(cudaError_t e) { return e == cudaSuccess ? TREE_OK : TREE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* tree_status_string(int status) {
  switch (status) {
    case TREE_OK: return "TREE_OK";
    case TREE_ERR_INVALID_ARG: return "TREE_ERR_INVALID_ARG";
    case TREE_ERR_ALIGNMENT: return "TREE_ERR_ALIGNMENT";
    case TREE_ERR_CAPACITY: return "TREE_ERR_CAPACITY";
    case TREE_ERR_MALFORMED_TREE: return "TREE_ERR_MALFORMED_TREE";
    case TREE_ERR_UNSUPPORTED: return "TREE_ERR_UNSUPPORTED";
    case TREE_ERR_CUDA: return "TREE_ERR_CUDA";
    case TREE_ERR_TIMEOUT: return "TREE_ERR_TIMEOUT";
    case TREE_ERR_WORKSPACE: return "TREE_ERR_WORKSPACE";
    case TREE_ERR_BOUNDS: return "TREE_ERR_BOUNDS";
    default: return "TREE_ERR_UNKNOWN";
  }
}

const char* tree_version(void) { return "0.1.0"; }

int32_t tree_debug_build(void) { return tree::kDebugBuild ? 1 : 0; }

size_t tree_pack_positions_workspace_bytes(int32_t T_pad, int32_t n_nodes) {
  if (T_pad < 0 || n_nodes < 0) return 0;
  return tree::pack_positions_workspace_bytes(T_pad, n_nodes);
}

tree_status_t tree_pack_positions(const int32_t* token_node, int32_t T_pad,
                                  const int32_t* node_entry, const int32_t* node_exit,
                                  int32_t n_nodes, int32_t* position_ids, int32_t* key_reach,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                  tree_stream_t stream) {
  if (T_pad < 0 || n_nodes < 0 || !dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad % tree::kBlock) return TREE_ERR_ALIGNMENT;
  if (T_pad == 0) return TREE_OK;
  if (!token_node || !position_ids || !key_reach || !workspace ||
      (n_nodes > 0 && (!node_entry || !node_exit)))
    return TREE_ERR_INVALID_ARG;
  if (n_nodes > T_pad) return TREE_ERR_INVALID_ARG;   // every node owns >= 1 token
  if (!aligned16(workspace)) return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree::pack_positions_workspace_bytes(T_pad, n_nodes))
    return TREE_ERR_WORKSPACE;
  return cuda_result(tree::launch_pack_positions(token_node, T_pad, node_entry, node_exit,
                                                 n_nodes, position_ids, key_reach, workspace,
                                                 dev_status, stream));
}

size_t tree_blockmap_bytes(int32_t T_pad) {
  if (T_pad < 0) return 0;
  return sizeof(int32_t) * tree::blockmap_words(T_pad / tree::kBlock);
}

tree_status_t tree_blockmap_build(const int32_t* key_reach, int32_t T_pad, int32_t block,
                                  void* blockmap, size_t blockmap_bytes, int32_t* dev_status,
                                  tree_stream_t stream) {
  if (T_pad < 0 || !dev_status) return TREE_ERR_INVALID_ARG;
  if (block != tree::kBlock) return TREE_ERR_UNSUPPORTED;
  if (T_pad % tree::kBlock) return TREE_ERR_ALIGNMENT;
  if (T_pad == 0) return TREE_OK;
  if (!key_reach || !blockmap) return TREE_ERR_INVALID_ARG;
  if (!aligned16(blockmap)) return TREE_ERR_ALIGNMENT;
  if (blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  return cuda_result(tree::launch_blockmap_build(key_reach, T_pad, blockmap, dev_status, stream));
}

tree_status_t tree_attn_fwd(const void* q, const void* k, const void* v,
                            const int32_t* key_reach, const void* blockmap,
                            size_t blockmap_bytes, int32_t T_pad, int32_t Hq, int32_t Hkv,
                            int32_t d, float scale, void* o, float* lse, int32_t* dev_status,
                            tree_stream_t stream) {
  tree_status_t st = check_attn_shape(T_pad, Hq, Hkv, d);
  if (st != TREE_OK) return st;
  if (!valid_scale(scale)) return TREE_ERR_INVALID_ARG;
  if (!dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad == 0) return TREE_OK;
  if (!q || !k || !v || !key_reach || !blockmap || !o || !lse) return TREE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(key_reach) || !aligned16(blockmap))
    return TREE_ERR_ALIGNMENT;
  if (blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv, to;
  if (!encode_map(&tq, q, T_pad, Hq, d) || !encode_map(&tk, k, T_pad, Hkv, d) ||
      !encode_map(&tv, v, T_pad, Hkv, d) || !encode_map(&to, o, T_pad, Hq, d, 32))
    return TREE_ERR_CUDA;
  return cuda_result(tree::launch_attn_fwd(tq, tk, tv, to, key_reach, blockmap, T_pad, Hq, Hkv,
                                           d, scale, o, lse, dev_status, stream, 0, T_pad));
}

size_t tree_attn_bwd_workspace_bytes(int32_t T_pad, int32_t Hq, int32_t d) {
  if (T_pad < 0 || Hq <= 0 || d <= 0) return 0;
  return tree::attn_bwd_workspace_bytes(T_pad, Hq, d);
}

tree_status_t tree_attn_bwd_prepare(const void* o, const void* d_o, const float* lse,
                                    int32_t T_pad, int32_t Hq, int32_t d, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status,
                                    tree_stream_t stream) {
  tree_status_t st = check_attn_shape(T_pad, Hq, 1, d);
  if (st != TREE_OK) return st;
  if (!dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad == 0) return TREE_OK;
  if (!o || !d_o || !lse || !workspace) return TREE_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(d_o) || !aligned16(lse) || !aligned16(workspace))
    return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree::attn_bwd_workspace_bytes(T_pad, Hq, d)) return TREE_ERR_WORKSPACE;
  return cuda_result(tree::launch_attn_bwd_prepare(o, d_o, lse, T_pad, Hq, d, workspace,
                                                   dev_status, stream, num_sms_current(), 0,
                                                   T_pad));
}

tree_status_t tree_attn_bwd_main(const void* q, const void* k, const void* v, const void* d_o,
                                 const int32_t* key_reach, const void* blockmap,
                                 size_t blockmap_bytes, int32_t T_pad, int32_t Hq, int32_t Hkv,
                                 int32_t d, float scale, void* dk, void* dv, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_status,
                                 tree_stream_t stream) {
  tree_status_t st = check_attn_shape(T_pad, Hq, Hkv, d);
  if (st != TREE_OK) return st;
  if (!valid_scale(scale)) return TREE_ERR_INVALID_ARG;
  if (!dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad == 0) return TREE_OK;
  if (!q || !k || !v || !d_o || !key_reach || !blockmap || !dk || !dv || !workspace)
    return TREE_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, d_o, key_reach, blockmap, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree::attn_bwd_workspace_bytes(T_pad, Hq, d)) return TREE_ERR_WORKSPACE;
  if (blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!encode_map(&tq, q, T_pad, Hq, d) || !encode_map(&tk, k, T_pad, Hkv, d) ||
      !encode_map(&tv, v, T_pad, Hkv, d) || !encode_map(&tdo, d_o, T_pad, Hq, d) ||
      !encode_map_acc(&tdq, workspace, T_pad, Hq, d) ||   // the accumulator leads the workspace
      !encode_map(&tdk, dk, T_pad, Hkv, d, 32) || !encode_map(&tdv, dv, T_pad, Hkv, d, 32))
    return TREE_ERR_CUDA;
  return cuda_result(tree::launch_attn_bwd_main(tq, tk, tv, tdo, tdq, tdk, tdv, key_reach,
                                                blockmap, T_pad, Hq, Hkv, d, scale, dk, dv,
                                                workspace, dev_status, stream, num_sms_current(),
                                                0, T_pad, nullptr, nullptr));
}

tree_status_t tree_attn_bwd_finish(int32_t T_pad, int32_t Hq, int32_t d, float scale,
                                   const void* workspace, size_t workspace_bytes, void* dq,
                                   int32_t* dev_status, tree_stream_t stream) {
  tree_status_t st = check_attn_shape(T_pad, Hq, 1, d);
  if (st != TREE_OK) return st;
  if (!valid_scale(scale)) return TREE_ERR_INVALID_ARG;
  if (!dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad == 0) return TREE_OK;
  if (!workspace || !dq) return TREE_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !aligned16(dq)) return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree::attn_bwd_workspace_bytes(T_pad, Hq, d)) return TREE_ERR_WORKSPACE;
  return cuda_result(tree::launch_attn_bwd_finish(T_pad, Hq, d, scale,
                                                  const_cast<void*>(workspace), dq, dev_status,
                                                  stream, num_sms_current(), 0, T_pad));
}

tree_status_t tree_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const void* d_o, const float* lse, const int32_t* key_reach,
                            const void* blockmap, size_t blockmap_bytes, int32_t T_pad,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale, void* dq, void* dk,
                            void* dv, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, tree_stream_t stream) {
  tree_status_t st = check_attn_shape(T_pad, Hq, Hkv, d);
  if (st != TREE_OK) return st;
  if (!valid_scale(scale)) return TREE_ERR_INVALID_ARG;
  if (!dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad == 0) return TREE_OK;
  if (!q || !k || !v || !o || !d_o || !lse || !key_reach || !blockmap || !dq || !dk || !dv ||
      !workspace)
    return TREE_ERR_INVALID_ARG;
  // every argument error is returned before the first launch
  const void* ptrs[] = {q, k, v, o, d_o, lse, key_reach, blockmap, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree::attn_bwd_workspace_bytes(T_pad, Hq, d)) return TREE_ERR_WORKSPACE;
  if (blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  st = tree_attn_bwd_prepare(o, d_o, lse, T_pad, Hq, d, workspace, workspace_bytes, dev_status,
                             stream);
  if (st != TREE_OK) return st;
  st = tree_attn_bwd_main(q, k, v, d_o, key_reach, blockmap, blockmap_bytes, T_pad, Hq, Hkv, d,
                          scale, dk, dv, workspace, workspace_bytes, dev_status, stream);
  if (st != TREE_OK) return st;
  return tree_attn_bwd_finish(T_pad, Hq, d, scale, workspace, workspace_bytes, dq, dev_status,
                              stream);
}

size_t tree_dta_attn_workspace_bytes(int32_t T_pad, int32_t Hq, int32_t Hkv, int32_t d) {
  if (T_pad < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return 0;
  return tree::attn_bwd_workspace_bytes(T_pad, Hq, d) +
         2 * static_cast<size_t>(T_pad) * Hkv * d * sizeof(float);
}

tree_status_t tree_dta_attn(const void* q, const void* k, const void* v, const void* d_o,
                            const int32_t* key_reach, const void* blockmap,
                            size_t blockmap_bytes, int32_t T_pad, int32_t Hq, int32_t Hkv,
                            int32_t d, float scale, const int32_t* ops, int64_t n_ops, void* o,
                            float* lse, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, tree_stream_t stream) {
  tree_status_t st = check_attn_shape(T_pad, Hq, Hkv, d);
  if (st != TREE_OK) return st;
  if (!valid_scale(scale) || !dev_status || n_ops < 0) return TREE_ERR_INVALID_ARG;
  if (T_pad == 0) return TREE_OK;
  if (!q || !k || !v || !d_o || !key_reach || !blockmap || !o || !lse || !dq || !dk || !dv ||
      !workspace || (n_ops > 0 && !ops))
    return TREE_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, d_o, key_reach, blockmap, o, lse, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree_dta_attn_workspace_bytes(T_pad, Hq, Hkv, d))
    return TREE_ERR_WORKSPACE;
  if (blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  for (int64_t i = 0; i < n_ops; ++i) {
    const int32_t kind = ops[3 * i], t0 = ops[3 * i + 1], t1 = ops[3 * i + 2];
    if (kind < TREE_DTA_FWD_PUSH || kind > TREE_DTA_BWD_POP || t0 < 0 || t1 <= t0 || t1 > T_pad)
      return TREE_ERR_INVALID_ARG;
  }
  // the bwd workspace (dQ accumulator, D and LSE rows) leads; the fp32 dK and
  // dV accumulators follow
  const size_t bwd_bytes = tree::attn_bwd_workspace_bytes(T_pad, Hq, d);
  float* dk_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_bytes);
  float* dv_acc = dk_acc + static_cast<size_t>(T_pad) * Hkv * d;
  CUtensorMap tq, tk, tv, to, tdo, tdq, tdk, tdv;
  if (!encode_map(&tq, q, T_pad, Hq, d) || !encode_map(&tk, k, T_pad, Hkv, d) ||
      !encode_map(&tv, v, T_pad, Hkv, d) || !encode_map(&to, o, T_pad, Hq, d, 32) ||
      !encode_map(&tdo, d_o, T_pad, Hq, d) || !encode_map_acc(&tdq, workspace, T_pad, Hq, d) ||
      !encode_map(&tdk, dk, T_pad, Hkv, d, 32) || !encode_map(&tdv, dv, T_pad, Hkv, d, 32))
    return TREE_ERR_CUDA;
  const int sms = num_sms_current();
  cudaError_t e = tree::launch_dta_init(o, dq, lse, workspace,
                                        tree_dta_attn_workspace_bytes(T_pad, Hq, Hkv, d), T_pad,
                                        Hq, d, dev_status, stream, sms);
  for (int64_t i = 0; e == cudaSuccess && i < n_ops; ++i) {
    const int32_t kind = ops[3 * i], t0 = ops[3 * i + 1], t1 = ops[3 * i + 2];
    if (kind != TREE_DTA_BWD_POP)     // forward of the rows against their visible keys
      e = tree::launch_attn_fwd(tq, tk, tv, to, key_reach, blockmap, T_pad, Hq, Hkv, d, scale,
                                o, lse, dev_status, stream, t0, t1);
    if (e == cudaSuccess && kind != TREE_DTA_FWD_PUSH) {   // backward of the rows
      e = tree::launch_attn_bwd_prepare(o, d_o, lse, T_pad, Hq, d, workspace, dev_status,
                                        stream, sms, t0, t1);
      if (e == cudaSuccess)
        e = tree::launch_attn_bwd_main(tq, tk, tv, tdo, tdq, tdk, tdv, key_reach, blockmap,
                                       T_pad, Hq, Hkv, d, scale, dk, dv, workspace, dev_status,
                                       stream, sms, t0, t1, dk_acc, dv_acc);
      if (e == cudaSuccess)
        e = tree::launch_attn_bwd_finish(T_pad, Hq, d, scale, workspace, dq, dev_status, stream,
                                         sms, t0, t1);
    }
  }
  if (e == cudaSuccess)
    e = tree::launch_dta_finish(dk_acc, dv_acc, dk, dv, T_pad, Hkv, d, dev_status, stream, sms);
  return cuda_result(e);
}

uint64_t tree_launch_count(void) { return tree::launches_total(); }

size_t tree_lm_head_workspace_bytes(int32_t T_pad, int32_t V) {
  if (T_pad < 0 || V < 1) return 0;
  return tree::lm_head_workspace_bytes(T_pad, V);
}

tree_status_t tree_lm_head_logprobs_entropy(const void* hidden, const void* weight,
                                            int32_t T_pad, int32_t H, int32_t V,
                                            const int32_t* token_ids, const int32_t* key_reach,
                                            const void* blockmap, size_t blockmap_bytes,
                                            float* lse, float* entropy, float* vocab_min,
                                            float* vocab_max, float* logprob,
                                            int32_t* token_pred, void* workspace,
                                            size_t workspace_bytes, int32_t* dev_status,
                                            tree_stream_t stream) {
  if (T_pad < 0 || H < 1 || V < 1 || !dev_status) return TREE_ERR_INVALID_ARG;
  if (T_pad % tree::kBlock) return TREE_ERR_ALIGNMENT;
  if (H % 64) return TREE_ERR_UNSUPPORTED;
  if (T_pad == 0) return TREE_OK;
  if (!hidden || !weight || !key_reach || !lse || !workspace) return TREE_ERR_INVALID_ARG;
  const bool labels = logprob != nullptr || token_pred != nullptr;
  if (labels && !blockmap) return TREE_ERR_INVALID_ARG;
  if (logprob && !token_ids) return TREE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(workspace))
    return TREE_ERR_ALIGNMENT;
  if (labels && blockmap_bytes < tree_blockmap_bytes(T_pad)) return TREE_ERR_WORKSPACE;
  if (workspace_bytes < tree::lm_head_workspace_bytes(T_pad, V)) return TREE_ERR_WORKSPACE;
  CUtensorMap th, tw;
  if (!encode_map_2d(&th, hidden, T_pad, H, 128) || !encode_map_2d(&tw, weight, V, H, 256))
    return TREE_ERR_CUDA;
  return cuda_result(tree::launch_lm_head(th, tw, hidden, weight, T_pad, H, V, token_ids,
                                          key_reach, blockmap, lse, entropy, vocab_min,
                                          vocab_max, logprob, token_pred, workspace, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream),
                                          num_sms_current()));
}

size_t tree_lm_head_grad_workspace_bytes(int32_t rows) {
  return rows < 0 ? 0 : static_cast<size_t>(rows) * 16;
}

tree_status_t tree_lm_head_logits_grad(const void* hidden, const void* weight, int32_t T_pad,
                                       int32_t H, int32_t V, int32_t row_lo, int32_t row_hi,
                                       const int32_t* token_ids, const int32_t* key_reach,
                                       const float* lse, const float* entropy,
                                       const float* grad_logprob, const float* grad_entropy,
                                       void* grad_logits, int64_t grad_row_stride,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, tree_stream_t stream) {
  if (T_pad < 0 || H < 1 || V < 1 || !dev_status || grad_row_stride < V)
    return TREE_ERR_INVALID_ARG;
  if (row_lo < 0 || row_hi < row_lo || row_hi > T_pad) return TREE_ERR_INVALID_ARG;
  if (T_pad % tree::kBlock || row_lo % tree::kBlock || row_hi % tree::kBlock)
    return TREE_ERR_ALIGNMENT;
  if (H % 64) return TREE_ERR_UNSUPPORTED;
  if (row_hi == row_lo) return TREE_OK;
  if (!hidden || !weight || !key_reach || !lse || !grad_logits || !workspace)
    return TREE_ERR_INVALID_ARG;
  if (grad_logprob && !token_ids) return TREE_ERR_INVALID_ARG;
  if (grad_entropy && !entropy) return TREE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(workspace) ||
      !aligned16(grad_logits) || (grad_row_stride * 2) % 16)
    return TREE_ERR_ALIGNMENT;
  if (workspace_bytes < tree_lm_head_grad_workspace_bytes(row_hi - row_lo))
    return TREE_ERR_WORKSPACE;
  CUtensorMap th, tw, tg;
  if (!encode_map_2d(&th, hidden, T_pad, H, 128) || !encode_map_2d(&tw, weight, V, H, 256) ||
      !encode_map_grad(&tg, grad_logits, row_hi - row_lo, V, grad_row_stride))
    return TREE_ERR_CUDA;
  return cuda_result(tree::launch_lm_head_grad(
      th, tw, tg, hidden, weight, T_pad, H, V, row_lo, row_hi, token_ids, key_reach, lse, entropy,
      grad_logprob, grad_entropy, grad_logits, grad_row_stride, workspace, dev_status,
      reinterpret_cast<cudaStream_t>(stream), num_sms_current()));
}

}  // extern "C"
