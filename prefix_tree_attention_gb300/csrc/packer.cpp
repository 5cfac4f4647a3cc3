// Host packer: sequences -> compressed tries in preorder layout.
//
// AReaL Tree Training guide, section "树构建流程":
//  step 2  first-fit-decreasing greedy insertion into tries bounded by
//          max_tokens_per_mb (occupied uncompressed nodes + nodes to add);
//  step 3  compression of single-child chains whose passing-sequence sets are
//          identical;
//  layout  preorder under a virtual root (section "核心数据结构：TrieNode"),
//          padded to the 128-token block (section "FlexAttention + BlockMask").
// Validation follows section "参数背后的源码校验逻辑".
//
// Along any root path the set of sequences passing a child is a subset of
// the set passing its parent, so "identical sets" is tested as "equal
// counts".  Children keep first-insertion order (a linked list appended at
// the tail); FFD ties keep input order.  A child is found by walking its
// parent's list while the parent has few children (most nodes of a trie of
// token sequences have one) and through a hash map once it has many; each
// sequence's node path is recorded as it is inserted, so its packed indices
// need no second walk.
#include <algorithm>
#include <cstdint>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/tree_attn.h"

namespace {

struct UNode {            // uncompressed node: one token
  int32_t tok;
  int32_t parent;
  int32_t first_child = -1;
  int32_t last_child = -1;
  int32_t next_sibling = -1;
  int32_t pass = 0;       // sequences passing this node
  int32_t nkids = 0;
};

// Children of a node with at least this many are also kept in the hash map.
constexpr int32_t kHashKids = 8;

struct UTrie {
  std::vector<UNode> nodes;                    // nodes[0] is the virtual root
  std::unordered_map<uint64_t, int32_t> child; // (parent, tok) -> node, wide nodes only
  int64_t occupied = 0;
  std::vector<int32_t> seqs;                   // input indices, insertion order
  std::vector<int32_t> path;                   // every sequence's nodes, in order
  std::vector<int64_t> path_off{0};            // sequence k: path[path_off[k], path_off[k+1])

  UTrie() { nodes.push_back(UNode{-1, -1}); }

  static uint64_t key(int32_t parent, int32_t tok) {
    return (static_cast<uint64_t>(static_cast<uint32_t>(parent)) << 32) |
           static_cast<uint32_t>(tok);
  }
  int32_t find(int32_t parent, int32_t tok) const {
    if (nodes[parent].nkids >= kHashKids) {
      auto it = child.find(key(parent, tok));
      return it == child.end() ? -1 : it->second;
    }
    for (int32_t c = nodes[parent].first_child; c >= 0; c = nodes[c].next_sibling)
      if (nodes[c].tok == tok) return c;
    return -1;
  }
  int64_t additional(const int32_t* s, int64_t len) const {
    int32_t u = 0;
    int64_t matched = 0;
    while (matched < len) {
      int32_t c = find(u, s[matched]);
      if (c < 0) break;
      u = c;
      ++matched;
    }
    return len - matched;
  }
  void insert(const int32_t* s, int64_t len, int32_t sid) {
    int32_t u = 0;
    for (int64_t i = 0; i < len; ++i) {
      int32_t c = find(u, s[i]);
      if (c < 0) {
        c = static_cast<int32_t>(nodes.size());
        nodes.push_back(UNode{s[i], u});
        UNode& p = nodes[u];
        if (p.last_child < 0) p.first_child = c;
        else nodes[p.last_child].next_sibling = c;
        p.last_child = c;
        if (++p.nkids == kHashKids) {       // the node turns wide: index all its children
          for (int32_t k = p.first_child; k >= 0; k = nodes[k].next_sibling)
            child.emplace(key(u, nodes[k].tok), k);
        } else if (p.nkids > kHashKids) {
          child.emplace(key(u, s[i]), c);
        }
        ++occupied;
      }
      nodes[c].pass += 1;
      path.push_back(c);
      u = c;
    }
    seqs.push_back(sid);
    path_off.push_back(static_cast<int64_t>(path.size()));
  }
};

}  // namespace

struct tree_packing {
  struct Trie {
    int32_t n_tokens = 0, T_pad = 0, n_nodes = 0;
    int64_t pairs = 0;
    std::vector<int32_t> token_node, token_ids, node_entry, node_exit, seq_ids;
    std::vector<std::vector<int32_t>> seq_idx;
  };
  std::vector<Trie> tries;
};

namespace {

void lay_out(const UTrie& u, int32_t block, int32_t pad_to, tree_packing::Trie& out) {
  // Compressed nodes: chains of uncompressed nodes.
  struct CNode {
    std::vector<int32_t> chain;
    std::vector<int32_t> kids;  // compressed children, insertion order
  };
  std::vector<CNode> cn;
  std::vector<int32_t> cn_of(u.nodes.size(), -1);
  // Build compressed nodes top-down (explicit stack of chain heads).
  std::vector<std::pair<int32_t, int32_t>> work;  // (chain head, compressed parent)
  std::vector<int32_t> top;                       // compressed children of the root
  for (int32_t c = u.nodes[0].first_child; c >= 0; c = u.nodes[c].next_sibling)
    work.push_back({c, -1});
  std::reverse(work.begin(), work.end());
  // Process in an order that keeps each kids list in insertion order: pop
  // from the back after pushing siblings reversed.
  while (!work.empty()) {
    auto [head, cpar] = work.back();
    work.pop_back();
    int32_t id = static_cast<int32_t>(cn.size());
    cn.push_back(CNode{});
    int32_t x = head;
    cn[id].chain.push_back(x);
    cn_of[x] = id;
    while (true) {
      const UNode& n = u.nodes[x];
      if (n.first_child < 0 || n.first_child != n.last_child) break;  // not exactly one child
      int32_t c = n.first_child;
      if (u.nodes[c].pass != n.pass) break;
      x = c;
      cn[id].chain.push_back(x);
      cn_of[x] = id;
    }
    if (cpar < 0) top.push_back(id);
    else cn[cpar].kids.push_back(id);
    std::vector<int32_t> kids;
    for (int32_t c = u.nodes[x].first_child; c >= 0; c = u.nodes[c].next_sibling) kids.push_back(c);
    for (auto it = kids.rbegin(); it != kids.rend(); ++it) work.push_back({*it, id});
  }
  // Preorder ranks.
  const int32_t N = static_cast<int32_t>(cn.size());
  std::vector<int32_t> rank(N), order;
  order.reserve(N);
  std::vector<int32_t> stack(top.rbegin(), top.rend());
  while (!stack.empty()) {
    int32_t v = stack.back();
    stack.pop_back();
    rank[v] = static_cast<int32_t>(order.size());
    order.push_back(v);
    for (auto it = cn[v].kids.rbegin(); it != cn[v].kids.rend(); ++it) stack.push_back(*it);
  }
  // Subtree sizes in reverse preorder -> exit ranks; token depth bases.
  std::vector<int32_t> size(N, 1), cparent(N, -1);
  for (int32_t v = 0; v < N; ++v)
    for (int32_t k : cn[v].kids) cparent[k] = v;
  for (int32_t r = N - 1; r >= 0; --r) {
    int32_t v = order[r];
    if (cparent[v] >= 0) size[cparent[v]] += size[v];
  }
  int64_t n_tokens = 0;
  for (const auto& c : cn) n_tokens += static_cast<int64_t>(c.chain.size());
  const int64_t T_pad = pad_to > 0 ? pad_to : (n_tokens + block - 1) / block * block;
  out.n_tokens = static_cast<int32_t>(n_tokens);
  out.T_pad = static_cast<int32_t>(T_pad);
  out.n_nodes = N;
  out.token_node.assign(T_pad, -1);
  out.token_ids.assign(T_pad, -1);
  out.node_entry.resize(N);
  out.node_exit.resize(N);
  std::vector<int32_t> upos(u.nodes.size(), -1);  // packed index of each uncompressed node
  std::vector<int64_t> base(N, 0);                // depth of the node's first token
  int64_t p = 0;
  out.pairs = 0;
  for (int32_t r = 0; r < N; ++r) {
    int32_t v = order[r];
    out.node_entry[r] = r;
    out.node_exit[r] = r + size[v] - 1;
    if (cparent[v] >= 0)
      base[v] = base[cparent[v]] + static_cast<int64_t>(cn[cparent[v]].chain.size());
    for (size_t t = 0; t < cn[v].chain.size(); ++t) {
      int32_t x = cn[v].chain[t];
      out.token_node[p] = r;
      out.token_ids[p] = u.nodes[x].tok;
      upos[x] = static_cast<int32_t>(p);
      out.pairs += base[v] + static_cast<int64_t>(t) + 1;
      ++p;
    }
  }
  out.seq_ids = u.seqs;
  out.seq_idx.resize(u.seqs.size());
  for (size_t k = 0; k < u.seqs.size(); ++k) {
    const int64_t a = u.path_off[k], len = u.path_off[k + 1] - a;
    auto& idx = out.seq_idx[k];
    idx.resize(len);
    for (int64_t i = 0; i < len; ++i) idx[i] = upos[u.path[a + i]];
  }
}

}  // namespace

extern "C" {

tree_status_t tree_packing_build(const int32_t* tokens, const int64_t* seq_offsets,
                                 int32_t n_seqs, int32_t max_tokens_per_mb, int32_t block,
                                 int32_t pad_to_max, tree_packing_t** out) {
  if (!out || n_seqs < 0 || (n_seqs > 0 && (!tokens || !seq_offsets)) || block <= 0)
    return TREE_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_tokens_per_mb <= 0) return TREE_ERR_INVALID_ARG;
  if (max_tokens_per_mb % block) return TREE_ERR_ALIGNMENT;
  for (int32_t s = 0; s < n_seqs; ++s) {
    int64_t len = seq_offsets[s + 1] - seq_offsets[s];
    if (len <= 0) return TREE_ERR_INVALID_ARG;
    if (len > max_tokens_per_mb) return TREE_ERR_CAPACITY;
  }
  std::vector<int32_t> order(n_seqs);
  for (int32_t s = 0; s < n_seqs; ++s) order[s] = s;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return seq_offsets[a + 1] - seq_offsets[a] > seq_offsets[b + 1] - seq_offsets[b];
  });
  std::vector<std::unique_ptr<UTrie>> tries;
  for (int32_t sid : order) {
    const int32_t* s = tokens + seq_offsets[sid];
    int64_t len = seq_offsets[sid + 1] - seq_offsets[sid];
    bool placed = false;
    for (auto& t : tries) {
      if (t->occupied + t->additional(s, len) <= max_tokens_per_mb) {
        t->insert(s, len, sid);
        placed = true;
        break;
      }
    }
    if (!placed) {
      tries.push_back(std::make_unique<UTrie>());
      tries.back()->insert(s, len, sid);
    }
  }
  auto* pk = new (std::nothrow) tree_packing;
  if (!pk) return TREE_ERR_INVALID_ARG;
  pk->tries.resize(tries.size());
  for (size_t t = 0; t < tries.size(); ++t)
    lay_out(*tries[t], block, pad_to_max ? max_tokens_per_mb : 0, pk->tries[t]);
  *out = pk;
  return TREE_OK;
}

void tree_packing_free(tree_packing_t* packing) { delete packing; }

int32_t tree_packing_num_tries(const tree_packing_t* packing) {
  return packing ? static_cast<int32_t>(packing->tries.size()) : 0;
}

tree_status_t tree_packing_trie_info(const tree_packing_t* packing, int32_t t,
                                     int32_t* n_tokens, int32_t* T_pad, int32_t* n_nodes,
                                     int32_t* n_seqs, int64_t* visible_pairs) {
  if (!packing || t < 0 || t >= static_cast<int32_t>(packing->tries.size()))
    return TREE_ERR_INVALID_ARG;
  const auto& tr = packing->tries[t];
  if (n_tokens) *n_tokens = tr.n_tokens;
  if (T_pad) *T_pad = tr.T_pad;
  if (n_nodes) *n_nodes = tr.n_nodes;
  if (n_seqs) *n_seqs = static_cast<int32_t>(tr.seq_ids.size());
  if (visible_pairs) *visible_pairs = tr.pairs;
  return TREE_OK;
}

tree_status_t tree_packing_trie_arrays(const tree_packing_t* packing, int32_t t,
                                       int32_t* token_node, int32_t* token_ids,
                                       int32_t* node_entry, int32_t* node_exit,
                                       int32_t* seq_ids) {
  if (!packing || t < 0 || t >= static_cast<int32_t>(packing->tries.size()))
    return TREE_ERR_INVALID_ARG;
  const auto& tr = packing->tries[t];
  if (token_node) std::copy(tr.token_node.begin(), tr.token_node.end(), token_node);
  if (token_ids) std::copy(tr.token_ids.begin(), tr.token_ids.end(), token_ids);
  if (node_entry) std::copy(tr.node_entry.begin(), tr.node_entry.end(), node_entry);
  if (node_exit) std::copy(tr.node_exit.begin(), tr.node_exit.end(), node_exit);
  if (seq_ids) std::copy(tr.seq_ids.begin(), tr.seq_ids.end(), seq_ids);
  return TREE_OK;
}

tree_status_t tree_packing_seq_indices(const tree_packing_t* packing, int32_t t, int32_t k,
                                       int32_t* out, int32_t capacity) {
  if (!packing || !out || t < 0 || t >= static_cast<int32_t>(packing->tries.size()))
    return TREE_ERR_INVALID_ARG;
  const auto& tr = packing->tries[t];
  if (k < 0 || k >= static_cast<int32_t>(tr.seq_idx.size())) return TREE_ERR_INVALID_ARG;
  const auto& idx = tr.seq_idx[k];
  if (capacity < static_cast<int32_t>(idx.size())) return TREE_ERR_WORKSPACE;
  std::copy(idx.begin(), idx.end(), out);
  return TREE_OK;
}

}  // extern "C"
