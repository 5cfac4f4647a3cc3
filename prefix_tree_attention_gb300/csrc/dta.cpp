// tree_dta_schedule: the depth-first traversal of dynamic tree attention as a
// list of attention operator calls over packed token rows.
//
// AREAL-DTA, sections 3.1 (depth-first traversal of the prefix tree with a
// stack of the current path's keys/values: a node's new tokens run forward
// against the stack and are pushed; at a leaf the sequence's backward starts
// at once; popping a node runs its backward, after every descendant leaf has
// added to its key/value gradients) and 3.2 (chunked backward: a path is
// handled in chunks of at most `chunk` tokens; a leaf's last chunk is never
// pushed; a greedy DFS order favouring long uninterrupted push/pop runs).
//
// Chunks cut each node's token span every `chunk` tokens from its first
// token.  Children are visited deepest first (the longest root-to-leaf
// continuation below the child's first token, in tokens), ties by preorder
// rank.  Ops:
//   FWD_PUSH (t0, t1)  forward of rows [t0, t1) against the stack, then push
//   FWD_BWD  (t0, t1)  a leaf's last chunk: forward and backward, no push
//   BWD_POP  (t0, t1)  backward of the rows on top of the stack, then pop
// The stack at a chunk's forward holds exactly the chunk's ancestor tokens,
// so each op is the packed tree attention restricted to its query rows.
#include <algorithm>
#include <cstdint>
#include <utility>
#include <vector>

#include "../../include/tree_attn.h"

extern "C" tree_status_t tree_dta_schedule(const int32_t* token_node, int32_t T_pad,
                                           const int32_t* node_entry, const int32_t* node_exit,
                                           int32_t n_nodes, int32_t chunk, int32_t* ops,
                                           int64_t capacity, int64_t* n_ops,
                                           int64_t* peak_stack_tokens) {
  if (T_pad < 0 || n_nodes < 0 || chunk < 1 || capacity < 0 || !n_ops)
    return TREE_ERR_INVALID_ARG;
  if (T_pad % 128) return TREE_ERR_ALIGNMENT;
  if ((T_pad > 0 && !token_node) || (n_nodes > 0 && (!node_entry || !node_exit)))
    return TREE_ERR_INVALID_ARG;
  const int32_t n = n_nodes;
  // token spans: every node non-empty and contiguous
  std::vector<int32_t> start(n, -1), end(n, -1);
  for (int32_t j = 0; j < T_pad; ++j) {
    const int32_t nd = token_node[j];
    if (nd == -1) continue;
    if (nd < -1 || nd >= n) return TREE_ERR_MALFORMED_TREE;
    if (start[nd] == -1) start[nd] = j;
    else if (end[nd] != j - 1) return TREE_ERR_MALFORMED_TREE;
    end[nd] = j;
  }
  std::vector<int32_t> by_rank(n, -1);
  for (int32_t nd = 0; nd < n; ++nd) {
    if (start[nd] == -1) return TREE_ERR_MALFORMED_TREE;
    const int32_t r = node_entry[nd];
    if (r < 0 || r >= n || by_rank[r] != -1) return TREE_ERR_MALFORMED_TREE;
    if (node_exit[nd] < r || node_exit[nd] >= n) return TREE_ERR_MALFORMED_TREE;
    by_rank[r] = nd;
  }
  // preorder layout: nodes appear in rank order; parents from nested intervals
  std::vector<int32_t> parent(n, -1), open, top;
  std::vector<std::vector<int32_t>> kids(n);
  for (int32_t r = 0; r < n; ++r) {
    const int32_t nd = by_rank[r];
    if (r > 0 && start[nd] <= start[by_rank[r - 1]]) return TREE_ERR_MALFORMED_TREE;
    while (!open.empty() && node_exit[open.back()] < r) open.pop_back();
    if (!open.empty()) {
      if (node_exit[nd] > node_exit[open.back()]) return TREE_ERR_MALFORMED_TREE;
      parent[nd] = open.back();
      kids[open.back()].push_back(nd);
    } else {
      top.push_back(nd);
    }
    open.push_back(nd);
  }
  std::vector<int64_t> depth(n, 0);
  for (int32_t r = n - 1; r >= 0; --r) {
    const int32_t nd = by_rank[r];
    int64_t below = 0;
    for (int32_t c : kids[nd]) below = std::max(below, depth[c]);
    depth[nd] = static_cast<int64_t>(end[nd] - start[nd] + 1) + below;
  }
  // greedy order: deepest first; the lists are in rank order, so a stable
  // sort on depth keeps rank order among ties
  auto deepest_first = [&](std::vector<int32_t>& v) {
    std::stable_sort(v.begin(), v.end(),
                     [&](int32_t a, int32_t b) { return depth[a] > depth[b]; });
  };
  for (auto& k : kids) deepest_first(k);
  deepest_first(top);

  int64_t count = 0, cur = 0, peak = 0;
  auto emit = [&](int32_t kind, int32_t t0, int32_t t1) {
    if (ops && count < capacity) {
      ops[3 * count] = kind;
      ops[3 * count + 1] = t0;
      ops[3 * count + 2] = t1;
    }
    ++count;
    if (kind == TREE_DTA_FWD_PUSH) peak = std::max(peak, cur += t1 - t0);
    else if (kind == TREE_DTA_BWD_POP) cur -= t1 - t0;
  };
  // the chunks [a, min(a + chunk, end + 1)) of node nd, forwards or backwards
  auto push_chunks = [&](int32_t nd, int32_t last) {
    for (int64_t a = start[nd]; a < last; a += chunk)
      emit(TREE_DTA_FWD_PUSH, static_cast<int32_t>(a),
           static_cast<int32_t>(std::min<int64_t>(a + chunk, last)));
  };
  auto pop_chunks = [&](int32_t nd, int32_t last) {
    if (last <= start[nd]) return;
    const int64_t k = (static_cast<int64_t>(last) - start[nd] - 1) / chunk;
    for (int64_t c = k; c >= 0; --c) {
      const int64_t a = start[nd] + c * chunk;
      emit(TREE_DTA_BWD_POP, static_cast<int32_t>(a),
           static_cast<int32_t>(std::min<int64_t>(a + chunk, last)));
    }
  };
  // iterative DFS: (node, false) enters a node, (node, true) leaves it
  std::vector<std::pair<int32_t, bool>> work;
  for (auto it = top.rbegin(); it != top.rend(); ++it) work.emplace_back(*it, false);
  while (!work.empty()) {
    const auto [nd, leaving] = work.back();
    work.pop_back();
    const int32_t e1 = end[nd] + 1;
    if (leaving) {
      pop_chunks(nd, e1);
      continue;
    }
    if (kids[nd].empty()) {
      // pushed chunks, the last chunk forward+backward, then the pops
      const int64_t k = (static_cast<int64_t>(e1) - start[nd] - 1) / chunk;
      const int32_t last0 = static_cast<int32_t>(start[nd] + k * chunk);
      push_chunks(nd, last0);
      emit(TREE_DTA_FWD_BWD, last0, e1);
      pop_chunks(nd, last0);
      continue;
    }
    push_chunks(nd, e1);
    work.emplace_back(nd, true);
    for (auto it = kids[nd].rbegin(); it != kids[nd].rend(); ++it) work.emplace_back(*it, false);
  }
  *n_ops = count;
  if (peak_stack_tokens) *peak_stack_tokens = peak;
  if (ops && count > capacity) return TREE_ERR_WORKSPACE;
  return TREE_OK;
}
