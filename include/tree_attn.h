/*
 * tree_attn.h — C ABI of the packed prefix-trie ("tree training") attention
 * library for NVIDIA GB300 (sm_103a).
 *
 * What the library computes.  Sequences that share prefixes (n_samples
 * responses to one prompt, a shared system prompt, a shared multi-turn
 * history) are packed once into a compressed trie laid out in preorder, so
 * every shared token is stored and computed once (AReaL Tree Training guide,
 * sections "什么是 Tree Training" and "树构建流程").  Token i attends to
 * token j iff j <= i and j's node is i's node or one of its ancestors (the
 * guide's packing figure), and the position id of a token is the number of
 * tokens it may attend to minus one (section "打包数据的生成").  Attention is
 * ordinary softmax attention under that mask; its backward pass sums the
 * gradient of a shared-prefix token over every continuation (AREAL-DTA,
 * section 3 "Problem formalisation").
 *
 * Data model at this boundary.
 *   token_node[T_pad]   node of each packed token, -1 for a pad token.
 *   node_entry[N]       preorder rank of each node (a permutation of 0..N-1).
 *   node_exit[N]        largest preorder rank inside the node's subtree.
 *   Node a is an ancestor-or-self of node b iff
 *       node_entry[a] <= node_entry[b] <= node_exit[a].
 *   Tokens are laid out in preorder: each node's tokens are contiguous and
 *   nodes appear in increasing rank (the guide's TrieNode start_idx/end_idx
 *   spans and root-level preorder `nodes` list).  Several tries may share one
 *   buffer (a forest under a virtual root).  Pad tokens may sit only outside
 *   every subtree's token span (between top-level subtrees or at the end).
 *   T_pad is a multiple of the 128-token block (section "FlexAttention +
 *   BlockMask"; block-alignment check of "参数背后的源码校验逻辑").
 *
 *   Q, O, dO, dQ  bf16 [T_pad, Hq, d]   (token-major, d innermost, batch 1)
 *   K, V, dK, dV  bf16 [T_pad, Hkv, d]
 *   LSE           fp32 [Hq, T_pad]      natural-log logsumexp per row
 *   Query head h reads key/value head h / (Hq / Hkv).
 *
 * Pad semantics: a pad token attends to nothing and is attended by nothing;
 * its O and LSE are 0 and -inf, its gradients 0, its position id 0.
 *
 * Conventions for every call.
 *  * Ownership: the caller owns every buffer.  The library never allocates,
 *    frees or synchronises; work is queued on `stream` and runs in stream
 *    order.  Device pointers must be 16-byte aligned.
 *  * Errors detectable from the arguments (null pointer, sizes, alignment,
 *    unsupported shapes, short workspace) are returned synchronously and
 *    nothing is launched.  A launch failure returns TREE_ERR_CUDA.
 *  * Errors that depend on device data (a malformed tree; a device-side wait
 *    that ran out of time) are written to `*dev_status` (device int32).  The
 *    caller zeroes it once; the first error sticks, and later kernels that
 *    find it non-zero skip their work.  Read it after synchronising.
 */
#ifndef TREE_ATTN_H_
#define TREE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TREE_API __attribute__((visibility("default")))
#else
#define TREE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tree_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  TREE_OK = 0,
  TREE_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad head split,
                                  softmax scale not positive and finite */
  TREE_ERR_ALIGNMENT = 2,      /* T_pad or a capacity not a multiple of 128; unaligned pointer */
  TREE_ERR_CAPACITY = 3,       /* a sequence longer than max_tokens_per_mb */
  TREE_ERR_MALFORMED_TREE = 4, /* token_node/node_entry/node_exit inconsistent (device-detected) */
  TREE_ERR_UNSUPPORTED = 5,    /* block != 128, head_dim not in {64,128} */
  TREE_ERR_CUDA = 6,           /* a CUDA call or launch failed */
  TREE_ERR_TIMEOUT = 7,        /* a device-side wait exceeded its limit (device-detected) */
  TREE_ERR_WORKSPACE = 8,      /* workspace or blockmap buffer too small */
  TREE_ERR_BOUNDS = 9          /* an index read from device memory points outside the buffer
                                  it addresses (device-detected; TREE_DEBUG builds) */
} tree_status_t;

/* Human-readable name of a status code (static string). */
TREE_API const char* tree_status_string(int status);

/* Library version as "major.minor.patch". */
TREE_API const char* tree_version(void);

/* ------------------------------------------------------------------------
 * tree_debug_build — 1 for the bounds-checked TREE_DEBUG build, else 0.
 *
 * The library is built twice from the same sources: libtreeattn.so, and
 * libtreeattn_debug.so compiled with TREE_DEBUG.  Indices that a kernel
 * computes from its launch shape and the sizes passed to the call are in
 * range by construction in both.  The debug build also checks, before use,
 * every index a kernel reads from device memory — the blockmap's row order,
 * row offsets, counts and key-block lists, its column order, and key_reach
 * values — against the buffer it addresses.  A failed check writes
 * TREE_ERR_BOUNDS to *dev_status and the work that depends on it is
 * skipped (the CTA returns before its first dependent access); nothing
 * traps or asserts, so the context stays usable.  The release build
 * trusts those buffers to come from tree_pack_positions and
 * tree_blockmap_build.
 * ---------------------------------------------------------------------- */
TREE_API int32_t tree_debug_build(void);

/* ------------------------------------------------------------------------
 * tree_pack_positions — per-key reach and position ids.
 *
 * Source: the guide's section "打包数据的生成" (position id = attendable
 * count - 1) and its packing figure (ancestor mask).  For a preorder layout
 * the mask has the interval form  M(i,j) = (j <= i <= key_reach[j]),  where
 * key_reach[j] is the last token of the subtree of node(j); hence
 * position_ids is an inclusive scan of +1 at j and -1 after key_reach[j].
 *
 *   token_node   [in]  device int32[T_pad]
 *   node_entry   [in]  device int32[n_nodes]   (may be NULL if n_nodes == 0)
 *   node_exit    [in]  device int32[n_nodes]
 *   position_ids [out] device int32[T_pad]; pads get 0
 *   key_reach    [out] device int32[T_pad]; pads get j - 1 (empty interval)
 *   workspace    [tmp] device, >= tree_pack_positions_workspace_bytes()
 *   dev_status   [out] device int32; TREE_ERR_MALFORMED_TREE when a node
 *                      id is out of range, ranks are not a permutation,
 *                      exit < entry, a node is empty or split, nodes are not
 *                      in rank order, subtree intervals cross, or a pad sits
 *                      inside a subtree's span.
 * Returns TREE_ERR_ALIGNMENT if T_pad % 128 != 0.  T_pad == 0 is a no-op.
 * ---------------------------------------------------------------------- */
TREE_API size_t tree_pack_positions_workspace_bytes(int32_t T_pad, int32_t n_nodes);
TREE_API tree_status_t tree_pack_positions(const int32_t* token_node, int32_t T_pad,
                                  const int32_t* node_entry, const int32_t* node_exit,
                                  int32_t n_nodes, int32_t* position_ids, int32_t* key_reach,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                  tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_pack_positions_noalloc — tree_pack_positions without a workspace.
 *
 * The pages have no counterpart; this entry point exists for callers that
 * cannot allocate device memory at all — typically a plugin or custom
 * operator inside a host framework that owns every device allocation and
 * gives the operator only its input and output buffers, so it has no
 * workspace to pass.  The library keeps the scratch in one file-scope device
 * array of 1.75 MiB (held by every GPU that loads the library until the
 * process exits), enough for T_pad <= 65536 and n_nodes <= 65536; larger
 * sizes return TREE_ERR_WORKSPACE and launch nothing.  The call makes no
 * allocation call of any kind (no cudaMalloc, cudaFree or allocating library
 * routine); the array itself is part of the library's CUDA module and is
 * reserved on a device when that module is loaded there — under CUDA's lazy
 * module loading, at the first call on that device.  A caller that needs the
 * reservation made up front can make one call at start-up.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and remembers the CUDA context it found;
 * make that first call before any stream capture.  A call that finds another
 * context current (the primary context was reset and created again) looks
 * the address up again.  Every call re-initialises the scratch it uses before reading it.
 * All calls share the one array, so calls whose work overlaps on the GPU
 * (other streams, other host threads) race and must be serialised.
 * Arguments, outputs and device-side errors are those of tree_pack_positions.
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_pack_positions_noalloc(const int32_t* token_node, int32_t T_pad,
                                                   const int32_t* node_entry,
                                                   const int32_t* node_exit, int32_t n_nodes,
                                                   int32_t* position_ids, int32_t* key_reach,
                                                   int32_t* dev_status, tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_blockmap_build — classify every 128x128 (query block, key block)
 * tile as EMPTY, FULL or PARTIAL and list the non-empty tiles.
 *
 * Source: the guide's sections "树构建流程" step 4 and "FlexAttention +
 * BlockMask" (a block mask over 128-token blocks built from the trie).  From
 * the interval form of the mask, for key block kb with per-block
 * mn = min key_reach, mx = max key_reach (pads included):
 *   tile (qa, kb), kb > qa : EMPTY
 *   tile (kb, kb)          : PARTIAL if the block holds a real key, else EMPTY
 *   tile (qa, kb), kb < qa : EMPTY if mx < 128*qa, FULL if mn >= 128*qa+127,
 *                            else PARTIAL.
 * So each key block's non-empty tiles form one column run
 *   qa = kb (PARTIAL), kb < qa <= col_full_hi (FULL), col_full_hi < qa <= col_hi (PARTIAL).
 *
 *   key_reach [in]  device int32[T_pad] from tree_pack_positions
 *   block     [in]  must be 128 (else TREE_ERR_UNSUPPORTED)
 *   blockmap  [out] device buffer of >= tree_blockmap_bytes(T_pad) bytes,
 *                   int32 words laid out as (nb = T_pad / 128):
 *     [0]                   nb
 *     [1]                   nnz (non-empty tiles)
 *     [2], [3]              reserved (0)
 *     col_full_hi[nb]       at 4
 *     col_hi[nb]            at 4 + nb        (kb - 1 when the column is empty)
 *     row_cnt[nb]           at 4 + 2nb       non-empty tiles of query block qa
 *     row_nfull[nb]         at 4 + 3nb       FULL tiles of query block qa
 *     row_ptr[nb + 1]       at 4 + 4nb       CSR offsets into row_idx
 *     row_order[nb]         at 5 + 5nb       query blocks by row_cnt descending
 *                                            (ties: smaller index first)
 *     col_order[nb]         at 5 + 6nb       key blocks by column length
 *                                            descending (ties: smaller first)
 *     row_idx[nnz]          at 5 + 7nb       per query block: its FULL key
 *                                            blocks ascending, then its
 *                                            PARTIAL key blocks ascending
 * ---------------------------------------------------------------------- */
TREE_API size_t tree_blockmap_bytes(int32_t T_pad);
TREE_API tree_status_t tree_blockmap_build(const int32_t* key_reach, int32_t T_pad, int32_t block,
                                  void* blockmap, size_t blockmap_bytes, int32_t* dev_status,
                                  tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_attn_fwd — tree-masked softmax attention forward.
 *
 * Source: the guide's packing figure and section "两种注意力实现"
 * (attention under the tree mask in 128-token blocks, batch 1).  For each
 * query head h and query row i:
 *   O[i,h] = sum_j P_ij V[j, h/g],  P = softmax_j(scale * Q[i,h].K[j,h/g])
 * over the j with M(i,j); LSE[h,i] = log sum_j exp(scale * Q[i,h].K[j,h/g]).
 * EMPTY tiles are skipped; the mask is evaluated only on PARTIAL tiles.
 * bf16 inputs, fp32 accumulation, P rounded to bf16 before P.V, O rounded
 * to bf16 (nearest even).
 *
 *   q, k, v   [in]  device bf16 (layouts above)
 *   key_reach [in]  device int32[T_pad]
 *   blockmap  [in]  from tree_blockmap_build for the same key_reach
 *   blockmap_bytes  size of the blockmap buffer; less than
 *                   tree_blockmap_bytes(T_pad) is TREE_ERR_WORKSPACE
 *   d         [in]  64 or 128; Hq % Hkv == 0
 *   scale     [in]  softmax scale, positive and finite (1/sqrt(d) is the usual
 *                   choice); anything else is TREE_ERR_INVALID_ARG
 *   o         [out] device bf16 [T_pad, Hq, d]
 *   lse       [out] device fp32 [Hq, T_pad]
 *   dev_status[out] TREE_ERR_TIMEOUT if a device wait ran out of time
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_attn_fwd(const void* q, const void* k, const void* v,
                            const int32_t* key_reach, const void* blockmap,
                            size_t blockmap_bytes, int32_t T_pad, int32_t Hq, int32_t Hkv,
                            int32_t d, float scale, void* o, float* lse, int32_t* dev_status,
                            tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_attn_bwd — backward of tree_attn_fwd.
 *
 * Source: AREAL-DTA section 3 "Problem formalisation" (the loss is a sum over
 * sequences; a shared prefix is processed once and its gradient accumulates
 * every descendant sequence's contribution).  With P recomputed from LSE:
 *   D_i  = sum_d dO[i,h,d] O[i,h,d]
 *   dS   = P * (dO V^T - D)
 *   dQ   = scale * dS K,   dK = scale * dS^T Q (summed over the g heads of a
 *   kv head),             dV = P^T dO          (summed likewise).
 * A shared-prefix key is visible to the queries of every continuation, so
 * its dK/dV sum over all of them by construction.
 *
 *   o, d_o, lse   [in]  forward output, upstream gradient, forward LSE
 *   blockmap, blockmap_bytes  as for tree_attn_fwd
 *   scale         [in]  the forward's scale (positive and finite)
 *   dq            [out] device bf16 [T_pad, Hq, d]
 *   dk, dv        [out] device bf16 [T_pad, Hkv, d]
 *   workspace     [tmp] >= tree_attn_bwd_workspace_bytes(T_pad, Hq, d):
 *                       fp32 dQ accumulator + fp32 D rows
 * ---------------------------------------------------------------------- */
TREE_API size_t tree_attn_bwd_workspace_bytes(int32_t T_pad, int32_t Hq, int32_t d);
TREE_API tree_status_t tree_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const void* d_o, const float* lse, const int32_t* key_reach,
                            const void* blockmap, size_t blockmap_bytes, int32_t T_pad,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale, void* dq, void* dk,
                            void* dv, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, tree_stream_t stream);

/* The three steps of tree_attn_bwd, callable one by one on the same stream
 * (tree_attn_bwd is exactly prepare, main, finish):
 *   prepare  D[h,i] = sum_d dO[i,h,d] O[i,h,d] and LSE*log2(e) into the
 *            workspace; zero the fp32 dQ accumulator.       (HBM-bound)
 *   main     recompute S and P per non-empty tile, dS = P*(dP - D), dK and
 *            dV into dk/dv (bf16, dK scaled), dS K added into the fp32 dQ
 *            accumulator (tensor cores; the dominant step)
 *   finish   dq = bf16(scale * accumulator)                 (HBM-bound)
 * Arguments as for tree_attn_bwd; the workspace must be the same buffer for
 * all three. */
TREE_API tree_status_t tree_attn_bwd_prepare(const void* o, const void* d_o, const float* lse,
                                             int32_t T_pad, int32_t Hq, int32_t d,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, tree_stream_t stream);
TREE_API tree_status_t tree_attn_bwd_main(const void* q, const void* k, const void* v,
                                          const void* d_o, const int32_t* key_reach,
                                          const void* blockmap, size_t blockmap_bytes,
                                          int32_t T_pad, int32_t Hq, int32_t Hkv, int32_t d,
                                          float scale, void* dk, void* dv, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_status,
                                          tree_stream_t stream);
TREE_API tree_status_t tree_attn_bwd_finish(int32_t T_pad, int32_t Hq, int32_t d, float scale,
                                            const void* workspace, size_t workspace_bytes,
                                            void* dq, int32_t* dev_status, tree_stream_t stream);

/* ------------------------------------------------------------------------
 * Host packer: sequences -> tries in the layout above.
 *
 * Source: the guide's section "树构建流程": first-fit-decreasing greedy
 * insertion (longest first; a sequence joins the first trie whose occupied
 * node count plus the nodes it adds stays within max_tokens_per_mb, else
 * opens a new trie), compression of single-child chains whose passing
 * sequences are identical, preorder flattening under a virtual root, and
 * padding to a multiple of `block` (or to max_tokens_per_mb when
 * pad_to_max != 0).  Validation follows "参数背后的源码校验逻辑":
 * max_tokens_per_mb must be positive (TREE_ERR_INVALID_ARG) and a multiple
 * of block (TREE_ERR_ALIGNMENT); a sequence longer than max_tokens_per_mb
 * is TREE_ERR_CAPACITY; an empty sequence is TREE_ERR_INVALID_ARG.
 * Children keep first-insertion order; ties in length keep input order.
 * All pointers are host pointers.  The packing object is owned by the
 * caller and released with tree_packing_free.
 * ---------------------------------------------------------------------- */
typedef struct tree_packing tree_packing_t;

TREE_API tree_status_t tree_packing_build(const int32_t* tokens, const int64_t* seq_offsets,
                                 int32_t n_seqs, int32_t max_tokens_per_mb, int32_t block,
                                 int32_t pad_to_max, tree_packing_t** out);
TREE_API void tree_packing_free(tree_packing_t* packing);
TREE_API int32_t tree_packing_num_tries(const tree_packing_t* packing);

/* Sizes of trie t: real tokens, padded length, nodes, sequences, and the
 * number of visible (i, j) pairs = sum over real tokens of (position + 1). */
TREE_API tree_status_t tree_packing_trie_info(const tree_packing_t* packing, int32_t t,
                                     int32_t* n_tokens, int32_t* T_pad, int32_t* n_nodes,
                                     int32_t* n_seqs, int64_t* visible_pairs);

/* Arrays of trie t (host buffers sized from tree_packing_trie_info; any may
 * be NULL to skip it): token_node[T_pad], token_ids[T_pad] (-1 for pads),
 * node_entry[n_nodes], node_exit[n_nodes], seq_ids[n_seqs] (input indices in
 * insertion order). */
TREE_API tree_status_t tree_packing_trie_arrays(const tree_packing_t* packing, int32_t t,
                                       int32_t* token_node, int32_t* token_ids,
                                       int32_t* node_entry, int32_t* node_exit,
                                       int32_t* seq_ids);

/* Packed token indices of the k-th sequence of trie t, in sequence order
 * (the spans of the nodes it passes, concatenated); `out` holds the
 * sequence's length. */
TREE_API tree_status_t tree_packing_seq_indices(const tree_packing_t* packing, int32_t t, int32_t k,
                                       int32_t* out, int32_t capacity);

/* ------------------------------------------------------------------------
 * tree_partition_sequences — load-balanced split of a batch over K workers.
 *
 * Source: AREAL-DTA, section 4 (load-balanced parallelisation: problem
 * formalisation, partition algorithm, binary-search solution).  Each worker
 * builds one prefix tree from its group; a group's cost is that tree's token
 * count (the sum of its nodes' token lengths).  The sequences are ordered as
 * a DFS of the single prefix tree they would form together (lexicographic
 * order of the token sequences, ties in input order) and cut into at most
 * n_groups contiguous segments whose largest cost is the smallest possible
 * for that order: binary search over the bound tau from the longest sequence
 * to the whole tree's token count, each tau checked by a greedy scan that
 * starts a new segment when the next sequence would push the current one
 * past tau.  Segments are numbered in DFS order; when fewer than n_groups
 * segments are needed, the last groups are empty (cost 0).
 *
 *   tokens        [in]  host int32, the sequences concatenated
 *   seq_offsets   [in]  host int64[n_seqs + 1], sequence s = tokens[off[s], off[s+1])
 *   n_seqs        number of sequences (>= 1)
 *   n_groups      number of workers K (>= 1)
 *   group_of_seq  [out] host int32[n_seqs], the group of every input sequence
 *   group_cost    [out] host int64[n_groups], token count of each group's tree (may be NULL)
 *   max_cost      [out] host int64, the largest group cost (may be NULL)
 * Errors: TREE_ERR_INVALID_ARG for a null required pointer, n_seqs < 1,
 * n_groups < 1 or an empty sequence.  Pure host code; no device work.
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_partition_sequences(const int32_t* tokens, const int64_t* seq_offsets,
                                                int32_t n_seqs, int32_t n_groups,
                                                int32_t* group_of_seq, int64_t* group_cost,
                                                int64_t* max_cost);

/* ------------------------------------------------------------------------
 * tree_logprobs_entropy — log-probabilities and entropies of packed logits.
 *
 * Source: the guide's section "Log Probability 计算：树结构的特殊处理"
 * (gather_packed_tree_logprobs_entropy and gather_packed_tree_vocab_stats).
 * Row r of `logits` holds the next-token logits at packed token r.  Inside a
 * node the row predicts the next token of the node; the last row of a node
 * predicts the first token of each child (the page's transition).  So every
 * real token j has one predicting row
 *     pred(j) = the largest i < j with key_reach[i] >= j   (-1 if none),
 * the last key before j that row j may attend to: j - 1 inside a node, the
 * parent's last token at a node start, -1 at the start of a top-level node.
 * Per row r (a real token):
 *     lse[r]       = log sum_v exp(logits[r, v])
 *     entropy[r]   = -sum_v p_v log p_v,  p = softmax(logits[r])
 *     vocab_min[r] = min_v logits[r, v],  vocab_max[r] = max_v logits[r, v]
 * Per token j:
 *     logprob[j]    = logits[pred(j), token_ids[j]] - lse[pred(j)]  (0 if pred(j) < 0)
 *     token_pred[j] = pred(j)
 * Pads (key_reach[j] < j) get 0 everywhere and token_pred -1.  Every row's
 * distribution is reduced once and every (pred, label) pair gathered once,
 * which is what the page's per-node caches achieve.  fp32 arithmetic; the
 * exponentials use the hardware 2^x approximation.  Logits are assumed to be
 * finite: a -inf logit gives a NaN entropy (0 * log 0 in plain arithmetic),
 * a NaN logit NaN results for its row.
 *
 *   logits        [in]  device [T_pad rows, row_stride elements], the first V
 *                       of each row used; dtype TREE_DTYPE_BF16 or TREE_DTYPE_F32.
 *                       Rows whose start is 16-byte aligned are read in
 *                       16-byte groups, other layouts element by element.
 *   token_ids     [in]  device int32[T_pad], the packed token ids (needed
 *                       when logprob != NULL; pads may hold anything)
 *   key_reach     [in]  device int32[T_pad] from tree_pack_positions
 *   blockmap      [in]  from tree_blockmap_build for the same key_reach
 *                       (needed when logprob or token_pred is requested)
 *   lse           [out] device float[T_pad] (required)
 *   entropy, vocab_min, vocab_max, logprob
 *                 [out] device float[T_pad], each may be NULL to skip it
 *   token_pred    [out] device int32[T_pad], may be NULL
 *   dev_status    [out] TREE_ERR_MALFORMED_TREE if a token with a predicting
 *                       row has an id outside [0, V) (its logprob is NaN)
 * Returns TREE_ERR_UNSUPPORTED for another dtype, TREE_ERR_INVALID_ARG for a
 * missing required pointer, V < 1 or row_stride < V, TREE_ERR_ALIGNMENT if
 * T_pad % 128 != 0, TREE_ERR_WORKSPACE if blockmap_bytes is short.
 * T_pad == 0 is a no-op (checked before the pointers).  Two launches (rows,
 * then labels); one when neither logprob nor token_pred is requested.
 * ---------------------------------------------------------------------- */
typedef enum { TREE_DTYPE_BF16 = 0, TREE_DTYPE_F32 = 1 } tree_dtype_t;

TREE_API tree_status_t tree_logprobs_entropy(const void* logits, int32_t dtype,
                                             int64_t row_stride, int32_t T_pad, int32_t V,
                                             const int32_t* token_ids, const int32_t* key_reach,
                                             const void* blockmap, size_t blockmap_bytes,
                                             float* lse, float* entropy, float* vocab_min,
                                             float* vocab_max, float* logprob,
                                             int32_t* token_pred, int32_t* dev_status,
                                             tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_merge_per_sequence — per-token results into a [n_seqs, max_len] batch.
 *
 * Source: the same section (merge_packed_tree_results: per-sequence results
 * of several micro-batches put back into the original batch layout by
 * sequence id, short sequences padded with padding_value).  Sequence s owns
 * seq_pos[seq_offsets[s] .. seq_offsets[s+1]), the indices into `src` of its
 * tokens in order (for several tries in one buffer: each trie's packed
 * index plus the trie's offset).  With L its length:
 *     out[s, t] = src[seq_pos[seq_offsets[s] + t + shift]]   for t < L - trim
 *     out[s, t] = padding_value                              otherwise.
 * Log-probabilities, which the token they score holds, use shift 1, trim 1
 * (entry t scores token t+1).  Entropies and vocab statistics of the
 * predicting rows use shift 0, trim 1.  Per-token values use 0, 0.
 *
 *   src          [in]  device float[n_src]
 *   seq_pos      [in]  device int32[n_pos]
 *   seq_offsets  [in]  device int64[n_seqs + 1], non-decreasing, last <= n_pos
 *   out          [out] device float[n_seqs * max_len]
 *   dev_status   [out] TREE_ERR_MALFORMED_TREE for an index outside [0, n_src)
 *                      (that entry becomes NaN); TREE_ERR_INVALID_ARG for
 *                      offsets that decrease or pass n_pos (the row is NaN);
 *                      TREE_ERR_CAPACITY if L - trim > max_len.  As everywhere,
 *                      after an error the outputs are undefined (blocks that
 *                      start after it skip their work)
 * Returns TREE_ERR_INVALID_ARG for negative sizes, shift < 0 or trim < shift,
 * or a missing pointer.  n_seqs == 0 or max_len == 0 is a no-op.
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_merge_per_sequence(const float* src, int64_t n_src,
                                               const int32_t* seq_pos, int64_t n_pos,
                                               const int64_t* seq_offsets, int32_t n_seqs,
                                               int32_t max_len, int32_t shift, int32_t trim,
                                               float padding_value, float* out,
                                               int32_t* dev_status, tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_lm_head_logprobs_entropy — the LM head fused with the gather.
 *
 * Source: the guide's section "Log Probability 计算：树结构的特殊处理": the
 * log-probabilities and entropies of a packed tree are taken chunk by chunk
 * so that the [tokens, vocabulary] logits are never held at once.  Here the
 * logits logits[r, v] = sum_k hidden[r, k] * weight[v, k] (fp32 sums of bf16
 * products) exist only one 128 x 256 tile at a time, in tensor memory, and
 * the outputs are those of tree_logprobs_entropy on them:
 *     lse[r], entropy[r], vocab_min[r], vocab_max[r]   per real row
 *     logprob[j] = logits[pred(j), token_ids[j]] - lse[pred(j)],  token_pred[j]
 * with pred(j) as there (pads: 0 and -1).  The label logit is recomputed
 * as a fp32 dot product, so its rounding differs from the tile's by the
 * order of the sum.
 *
 *   hidden        [in]  device bf16 [T_pad, H] row-major, 16-byte aligned
 *   weight        [in]  device bf16 [V, H] row-major (one row per vocabulary
 *                       entry: the LM head / tied embedding), 16-byte aligned
 *   H             hidden size, a multiple of 64 (else TREE_ERR_UNSUPPORTED)
 *   token_ids, key_reach, blockmap, blockmap_bytes, lse, entropy, vocab_min,
 *   vocab_max, logprob, token_pred   as in tree_logprobs_entropy
 *   workspace     [scratch] device, 16-byte aligned,
 *                 >= tree_lm_head_workspace_bytes(T_pad, V) bytes (per-row
 *                 partial statistics of every 2048-column vocabulary chunk)
 *   dev_status    [out] TREE_ERR_MALFORMED_TREE for a label id outside [0, V);
 *                 TREE_ERR_TIMEOUT if a device wait ran out of time
 * Returns TREE_ERR_INVALID_ARG for a missing required pointer, H < 1 or
 * V < 1, TREE_ERR_ALIGNMENT for T_pad % 128 != 0 or an unaligned buffer,
 * TREE_ERR_WORKSPACE for a short workspace or blockmap.  T_pad == 0 is a
 * no-op.  Three launches: the persistent tcgen05 GEMM with the row
 * statistics in its epilogue (one CTA per SM), the combination of the
 * partials, and the labels (skipped when neither logprob nor token_pred is
 * requested).
 * ---------------------------------------------------------------------- */
TREE_API size_t tree_lm_head_workspace_bytes(int32_t T_pad, int32_t V);
TREE_API tree_status_t tree_lm_head_logprobs_entropy(const void* hidden, const void* weight,
                                                     int32_t T_pad, int32_t H, int32_t V,
                                                     const int32_t* token_ids,
                                                     const int32_t* key_reach,
                                                     const void* blockmap, size_t blockmap_bytes,
                                                     float* lse, float* entropy,
                                                     float* vocab_min, float* vocab_max,
                                                     float* logprob, int32_t* token_pred,
                                                     void* workspace, size_t workspace_bytes,
                                                     int32_t* dev_status, tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_lm_head_logits_grad — gradient of the fused gather w.r.t. the logits,
 * one chunk of rows at a time, without the logits.
 *
 * Source: the same section; the page's gather is differentiated by a
 * training step and runs chunk by chunk so that the [tokens, vocabulary]
 * logits are never held at once.  For rows [row_lo, row_hi) this writes
 *     grad_logits[r - row_lo, v] = sum_{pred(j) = r} grad_logprob[j] * ([v == y_j] - p_v)
 *                                - grad_entropy[r] * p_v * (logits[r, v] - lse[r] + H)
 * (the gradient tree_logprobs_entropy_bwd writes from materialised
 * logits), recomputing each 128 x 256 logits tile hidden W^T in tensor
 * memory as tree_lm_head_logprobs_entropy does.  The caller then forms the
 * LM head's own gradients from the chunk with two plain GEMMs:
 *     d hidden[rows] = grad_logits W,   d W += grad_logits^T hidden[rows].
 * fp32 arithmetic, one rounding to bf16 per entry; deterministic.
 *
 *   hidden, weight, T_pad, H, V, token_ids, key_reach
 *                 [in]  as in tree_lm_head_logprobs_entropy
 *   row_lo, row_hi      the chunk: 0 <= row_lo <= row_hi <= T_pad, both
 *                       multiples of 128 (else TREE_ERR_ALIGNMENT)
 *   lse, entropy  [in]  device float[T_pad] from tree_lm_head_logprobs_entropy
 *                       (entropy needed when grad_entropy != NULL)
 *   grad_logprob  [in]  device float[T_pad] per label token, or NULL
 *   grad_entropy  [in]  device float[T_pad] per row, or NULL
 *                       (in the packed layout tree_merge_per_sequence_bwd leaves)
 *   grad_logits   [out] device bf16 [row_hi - row_lo, grad_row_stride], the
 *                       first V entries of each row written (pads: 0); rows
 *                       16-byte aligned (grad_row_stride a multiple of 8)
 *   workspace     [scratch] device, 16-byte aligned,
 *                 >= tree_lm_head_grad_workspace_bytes(row_hi - row_lo)
 *   dev_status    [out] TREE_ERR_MALFORMED_TREE for a child id outside [0, V)
 *                       (its one-hot term is dropped); TREE_ERR_TIMEOUT
 * Returns TREE_ERR_INVALID_ARG for a missing required pointer, H < 1,
 * V < 1, grad_row_stride < V or a chunk outside [0, T_pad),
 * TREE_ERR_ALIGNMENT, TREE_ERR_UNSUPPORTED for H % 64 != 0,
 * TREE_ERR_WORKSPACE.  An empty chunk is a no-op.  Three launches (row
 * coefficients, the GEMM with the gradient epilogue, the one-hot terms;
 * the last skipped without grad_logprob).
 * ---------------------------------------------------------------------- */
TREE_API size_t tree_lm_head_grad_workspace_bytes(int32_t rows);
TREE_API tree_status_t tree_lm_head_logits_grad(const void* hidden, const void* weight,
                                                int32_t T_pad, int32_t H, int32_t V,
                                                int32_t row_lo, int32_t row_hi,
                                                const int32_t* token_ids,
                                                const int32_t* key_reach, const float* lse,
                                                const float* entropy,
                                                const float* grad_logprob,
                                                const float* grad_entropy, void* grad_logits,
                                                int64_t grad_row_stride, void* workspace,
                                                size_t workspace_bytes, int32_t* dev_status,
                                                tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_merge_per_sequence_bwd — the merge's adjoint (its gradient).
 *
 * Source: the same section; the page's merge is part of a differentiable
 * computation, so a training step passes the gradient of its loss with
 * respect to the merged [n_seqs, max_len] batch back to the packed values.
 * With the arguments of the forward call (same seq_pos, seq_offsets, shift,
 * trim, max_len):
 *     src_grad[seq_pos[seq_offsets[s] + t + shift]] += out_grad[s, t]
 *                                                   for t < min(L - trim, max_len).
 * A packed token shared by several sequences (a common prefix) receives the
 * sum over those sequences.  ACCUMULATES into src_grad: zero it first for a
 * plain gradient.  The sums use fp32 atomic adds, so their rounding order,
 * and the last bits of a shared token's sum, may differ run to run.
 *
 *   out_grad     [in]  device float[n_seqs * max_len]
 *   seq_pos, n_pos, seq_offsets, n_seqs, max_len, shift, trim
 *                [in]  as in tree_merge_per_sequence
 *   src_grad     [in,out] device float[n_src]
 *   dev_status   [out] TREE_ERR_MALFORMED_TREE for an index outside
 *                      [0, n_src), TREE_ERR_INVALID_ARG for bad offsets,
 *                      TREE_ERR_CAPACITY if L - trim > max_len (the entries
 *                      that fit are still added); offending entries add nothing
 * Returns TREE_ERR_INVALID_ARG for negative sizes, shift < 0 or
 * trim < shift, or a missing pointer.  n_seqs == 0 or max_len == 0 is a
 * no-op.  One launch.
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_merge_per_sequence_bwd(const float* out_grad, const int32_t* seq_pos,
                                                   int64_t n_pos, const int64_t* seq_offsets,
                                                   int32_t n_seqs, int32_t max_len,
                                                   int32_t shift, int32_t trim, float* src_grad,
                                                   int64_t n_src, int32_t* dev_status,
                                                   tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_logprobs_entropy_bwd — gradient of the gather with respect to the logits.
 *
 * Source: the section "Log Probability 计算：树结构的特殊处理" of the guide;
 * its gather is differentiated by a training step's backward pass.  Inputs
 * are the per-token gradients in the packed layout (as
 * tree_merge_per_sequence_bwd leaves them): grad_logprob[j], the gradient
 * with respect to logprob[j] of tree_logprobs_entropy (label token j), and
 * grad_entropy[r], with respect to entropy[r] (row r).  With p = softmax
 * of row r, H = entropy[r], and the children of r (the tokens j with
 * pred(j) = r, each with its label y_j = token_ids[j]):
 *     grad_logits[r, v] = sum_{pred(j) = r} grad_logprob[j] * ([v == y_j] - p_v)
 *                       - grad_entropy[r] * p_v * (logits[r, v] - lse[r] + H)
 * (d log p_y / d x_v = [v == y] - p_v;  d H / d x_v = -p_v (log p_v + H)).
 * Pad rows get 0.  Overwrites grad_logits (rows [0, T_pad), first V
 * entries each).  fp32 arithmetic with the hardware 2^x approximation,
 * one rounding to the output type per entry; deterministic.  Uses the lse
 * and entropy saved by tree_logprobs_entropy on the same logits; the
 * children of r are found from key_reach (r + 1, then each next sibling
 * at key_reach[j] + 1, while j <= key_reach[r]), so no pred array is needed.
 *
 *   logits        [in]  device, as in tree_logprobs_entropy (same dtype and layout)
 *   token_ids     [in]  device int32[T_pad] (needed when grad_logprob != NULL)
 *   key_reach     [in]  device int32[T_pad] from tree_pack_positions
 *   lse           [in]  device float[T_pad] from tree_logprobs_entropy
 *   entropy       [in]  device float[T_pad] from tree_logprobs_entropy
 *                       (needed when grad_entropy != NULL)
 *   grad_logprob  [in]  device float[T_pad] per label token, or NULL (zero)
 *   grad_entropy  [in]  device float[T_pad] per row, or NULL (zero)
 *   grad_logits   [out] device [T_pad rows, grad_row_stride elements] of
 *                       the logits' dtype; rows 16-byte aligned with the
 *                       logits' rows are written in 16-byte groups
 *   dev_status    [out] TREE_ERR_MALFORMED_TREE if a child's id is outside
 *                       [0, V) (its one-hot term is dropped)
 * Returns TREE_ERR_UNSUPPORTED for another dtype, TREE_ERR_INVALID_ARG for a
 * missing required pointer, V < 1 or a row stride < V, TREE_ERR_ALIGNMENT if
 * T_pad % 128 != 0.  T_pad == 0 is a no-op.  One launch, one CTA per row:
 * reads and writes each row's V values once.
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_logprobs_entropy_bwd(const void* logits, int32_t dtype,
                                                 int64_t row_stride, int32_t T_pad, int32_t V,
                                                 const int32_t* token_ids,
                                                 const int32_t* key_reach, const float* lse,
                                                 const float* entropy,
                                                 const float* grad_logprob,
                                                 const float* grad_entropy, void* grad_logits,
                                                 int64_t grad_row_stride, int32_t* dev_status,
                                                 tree_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_dta_schedule — the depth-first traversal of dynamic tree attention.
 *
 * Source: AREAL-DTA, sections 3.1 (DFS over the prefix tree with a stack of
 * the current path's keys/values: forward and push on the way down, the
 * leaf's backward as soon as its sequence is complete, a node's backward
 * when it is popped, after all its descendants) and 3.2 (chunks of at most
 * `chunk` tokens, 2048 on the page; a leaf's last chunk is never pushed; a
 * greedy DFS order).  Readings: chunks cut each node's span every `chunk`
 * tokens from its first token; children are visited deepest first (longest
 * continuation in tokens below the child's first token), ties by preorder
 * rank.  The op list, one int32 triple (kind, t0, t1) per op over packed rows
 * [t0, t1):
 *   TREE_DTA_FWD_PUSH  forward of the rows against the stack, then push them
 *   TREE_DTA_FWD_BWD   a leaf's last chunk: forward and backward, no push
 *   TREE_DTA_BWD_POP   backward of the rows on top of the stack, then pop
 * At every forward the stack holds exactly the rows' ancestor tokens, so
 * each op is the packed tree attention restricted to its query rows; every
 * real token gets one forward and one backward; a token's backward comes
 * after those of all rows that see it.
 *
 *   token_node, node_entry, node_exit  [in]  host arrays, as for
 *                       tree_pack_positions (T_pad a multiple of 128)
 *   chunk          [in]  >= 1
 *   ops            [out] host int32[capacity][3], may be NULL to count only
 *   n_ops          [out] number of ops (always written)
 *   peak_stack_tokens [out] largest number of tokens on the stack (may be NULL)
 * Returns TREE_ERR_INVALID_ARG (bad sizes, chunk < 1, missing pointer),
 * TREE_ERR_ALIGNMENT (T_pad % 128), TREE_ERR_MALFORMED_TREE (node id out of
 * range, empty or split node, ranks not a permutation, nodes not in rank
 * order, crossing subtree intervals), TREE_ERR_WORKSPACE when ops is given
 * and capacity < n_ops (the first `capacity` ops are written).  Pure host
 * code; no device work.
 * ---------------------------------------------------------------------- */
typedef enum {
  TREE_DTA_FWD_PUSH = 0,
  TREE_DTA_FWD_BWD = 1,
  TREE_DTA_BWD_POP = 2
} tree_dta_op_t;

TREE_API tree_status_t tree_dta_schedule(const int32_t* token_node, int32_t T_pad,
                                         const int32_t* node_entry, const int32_t* node_exit,
                                         int32_t n_nodes, int32_t chunk, int32_t* ops,
                                         int64_t capacity, int64_t* n_ops,
                                         int64_t* peak_stack_tokens);

/* ------------------------------------------------------------------------
 * tree_dta_attn — attention forward and backward executed through the
 * depth-first traversal of dynamic tree attention.
 *
 * Source: AREAL-DTA, sections 3.1 (forward and push on the way down, a
 * leaf's backward as soon as its sequence is complete, a node's backward when
 * it is popped, after all its descendants) and 3.2 (chunked backward, no leaf
 * KV caching).  On the packed layout every key/value row stays resident, so
 * the stack is implicit: at each operation it holds exactly the ancestor
 * tokens of the operation's rows, which are the keys the packed mask lets
 * them see.  Each operation is therefore the packed tree attention
 * restricted to its query rows [t0, t1):
 *   TREE_DTA_FWD_PUSH  forward of the rows (O, LSE of those rows)
 *   TREE_DTA_FWD_BWD   forward, then backward of the rows
 *   TREE_DTA_BWD_POP   backward of the rows
 * A backward writes dQ of its rows and adds its rows' contributions to dK and
 * dV of every key they see into fp32 accumulators (a shared-prefix key thus
 * sums every continuation's rows, in traversal order); after the last
 * operation dK and dV are rounded to bf16.  O, dQ start at 0 and LSE at
 * -inf, so rows no operation covers (pads) keep those values and get zero
 * key gradients.  With a schedule from tree_dta_schedule (every real row in
 * one forward and one backward, forward first) the results equal
 * tree_attn_fwd + tree_attn_bwd up to fp32 summation order.
 *
 *   q, k, v, d_o, key_reach, blockmap, blockmap_bytes, T_pad, Hq, Hkv, d,
 *   scale          as for tree_attn_fwd / tree_attn_bwd
 *   ops            [in]  HOST int32[n_ops][3] of (kind, t0, t1), executed in
 *                        order; kind in {0,1,2}, 0 <= t0 < t1 <= T_pad, else
 *                        TREE_ERR_INVALID_ARG before any launch
 *   o, lse         [out] forward outputs (layouts as for tree_attn_fwd)
 *   dq, dk, dv     [out] gradients (layouts as for tree_attn_bwd)
 *   workspace      [tmp] >= tree_dta_attn_workspace_bytes(T_pad, Hq, Hkv, d):
 *                        the tree_attn_bwd workspace followed by fp32 dK and
 *                        dV accumulators [T_pad, Hkv, d]
 * Launches: 2 + one per FWD_PUSH, four per FWD_BWD, three per BWD_POP, all
 * queued on `stream` with no host synchronisation.
 * ---------------------------------------------------------------------- */
TREE_API size_t tree_dta_attn_workspace_bytes(int32_t T_pad, int32_t Hq, int32_t Hkv, int32_t d);
TREE_API tree_status_t tree_dta_attn(const void* q, const void* k, const void* v, const void* d_o,
                                     const int32_t* key_reach, const void* blockmap,
                                     size_t blockmap_bytes, int32_t T_pad, int32_t Hq,
                                     int32_t Hkv, int32_t d, float scale, const int32_t* ops,
                                     int64_t n_ops, void* o, float* lse, void* dq, void* dk,
                                     void* dv, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, tree_stream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics.
 *
 * tree_debug_wait_timeout — launch one warp that waits on a shared-memory
 * barrier nothing ever arrives on, through the same bounded wait that guards
 * every pipeline wait in tree_attn_fwd/bwd.  After limit_ns (1 ms .. 2 s,
 * else TREE_ERR_INVALID_ARG) the wait gives up and TREE_ERR_TIMEOUT is
 * written to *dev_status (unless it already holds an error); the kernel then
 * returns normally.  This is how the failure-detection path is tested
 * without faulting or hanging a GPU.  The pages have no counterpart.
 * ---------------------------------------------------------------------- */
TREE_API tree_status_t tree_debug_wait_timeout(int32_t* dev_status, int64_t limit_ns,
                                               tree_stream_t stream);

/* tree_launch_count — number of kernels the library has queued in this
 * process, over all entry points (for launch accounting in benchmarks). */
TREE_API uint64_t tree_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* TREE_ATTN_H_ */
