// tree_partition_sequences: load-balanced split of a rollout batch over K
// training workers.
//
// AREAL-DTA, section 4 (load-balanced parallelisation: problem
// formalisation, load-balanced partition algorithm, binary-search solution).
// Each worker builds one prefix tree from its group of sequences; the cost of
// a group is the number of tokens of that tree (the sum of its nodes' token
// lengths).  The goal is to minimise the largest group cost.  The sequences
// are put in DFS order of the single prefix tree they would form together
// (lexicographic order of the token sequences), and the ordered list is cut
// into at most K contiguous segments: the smallest feasible bound tau on the
// segment cost is found by binary search between the largest single-sequence
// cost and the cost of the whole tree, each candidate checked by a greedy scan
// that opens a new segment when the next sequence would push the current one
// past tau.  In DFS order the cost of a segment grows by len(s) - lcp(s, the
// previous sequence) per added sequence (its first sequence costs its full
// length), so the scan needs no tree.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/tree_attn.h"

namespace {

// Segments the greedy scan opens when no segment may cost more than tau
// (every single sequence fits: tau >= the longest length).
int64_t segments_for(const std::vector<int64_t>& len, const std::vector<int64_t>& add,
                     int64_t tau) {
  int64_t segs = 1, cur = len[0];
  for (size_t i = 1; i < len.size(); ++i) {
    if (cur + add[i] > tau) {
      ++segs;
      cur = len[i];
    } else {
      cur += add[i];
    }
  }
  return segs;
}

}  // namespace

extern "C" tree_status_t tree_partition_sequences(const int32_t* tokens,
                                                  const int64_t* seq_offsets, int32_t n_seqs,
                                                  int32_t n_groups, int32_t* group_of_seq,
                                                  int64_t* group_cost, int64_t* max_cost) {
  if (n_seqs <= 0 || n_groups <= 0 || !tokens || !seq_offsets || !group_of_seq)
    return TREE_ERR_INVALID_ARG;
  for (int32_t s = 0; s < n_seqs; ++s)
    if (seq_offsets[s + 1] - seq_offsets[s] <= 0) return TREE_ERR_INVALID_ARG;
  // DFS order of the combined prefix tree = lexicographic order (ties: input order).
  std::vector<int32_t> order(n_seqs);
  for (int32_t s = 0; s < n_seqs; ++s) order[s] = s;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return std::lexicographical_compare(tokens + seq_offsets[a], tokens + seq_offsets[a + 1],
                                        tokens + seq_offsets[b], tokens + seq_offsets[b + 1]);
  });
  std::vector<int64_t> len(n_seqs), add(n_seqs);
  int64_t longest = 0, total = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const int32_t s = order[i];
    len[i] = seq_offsets[s + 1] - seq_offsets[s];
    int64_t lcp = 0;
    if (i > 0) {
      const int32_t p = order[i - 1];
      const int64_t lp = seq_offsets[p + 1] - seq_offsets[p];
      const int32_t* a = tokens + seq_offsets[p];
      const int32_t* b = tokens + seq_offsets[s];
      while (lcp < lp && lcp < len[i] && a[lcp] == b[lcp]) ++lcp;
    }
    add[i] = len[i] - lcp;
    longest = std::max(longest, len[i]);
    total += add[i];
  }
  // Smallest tau in [longest, total] for which the greedy scan needs <= K segments.
  int64_t lo = longest, hi = total;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (segments_for(len, add, mid) <= n_groups)
      hi = mid;
    else
      lo = mid + 1;
  }
  const int64_t tau = lo;
  std::vector<int64_t> cost(n_groups, 0);
  int32_t g = 0;
  cost[0] = len[0];
  group_of_seq[order[0]] = 0;
  for (int32_t i = 1; i < n_seqs; ++i) {
    if (cost[g] + add[i] > tau) {
      ++g;
      cost[g] = len[i];
    } else {
      cost[g] += add[i];
    }
    group_of_seq[order[i]] = g;
  }
  if (group_cost)
    for (int32_t k = 0; k < n_groups; ++k) group_cost[k] = cost[k];
  if (max_cost) *max_cost = *std::max_element(cost.begin(), cost.end());
  return TREE_OK;
}
