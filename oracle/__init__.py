"""Oracle for prefix-tree ("tree training") attention — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct CPU restatement of what the
packed-trie attention path computes.  It exists to check the CUDA library and
nothing else: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product package never imports it, and it imports nothing from the product
package (they share only the seeded input generators in ``workloads/``).

Sources (web pages; cited by title and section):

* "AReaL Tree Training 完全指南" (AReaL Tree Training guide), sections
  "树构建流程" (tree construction: FFD greedy packing, trie compression),
  "核心数据结构：TrieNode" (node spans, preorder ``nodes`` list, virtual root),
  "打包数据的生成" (position ids from the dense mask), the packing figure
  (ancestor mask, worked example [A,B,C,D]/[A,B,E,F]/[A,G,H]),
  "FlexAttention + BlockMask" (128-token blocks),
  "参数背后的源码校验逻辑" (packing validation) and
  "Log Probability 计算：树结构的特殊处理" (per-sequence log-probabilities
  and entropies gathered from packed logits).
* "AREAL-DTA: Dynamic Tree Attention for Efficient Reinforcement Learning of
  Large Language Models", section 3 "Problem formalisation" (total loss is the
  sum of per-sequence losses; a shared prefix is computed once and its
  gradient sums the contributions of every descendant sequence), sections
  3.1-3.2 (depth-first traversal with a key/value stack, chunked backward,
  no leaf KV caching, greedy DFS order) and section 4
  "负载均衡并行化" (load-balanced split of a batch over training workers).

Modules:

* ``oracle.trie``      — trie insertion, first-fit-decreasing packing,
                         compression, preorder layout, 128-padding.
* ``oracle.mask``      — dense ancestor mask by parent-pointer walks,
                         position ids, 128x128 tile classes.
* ``oracle.attention`` — masked softmax attention forward/backward in fp64.
* ``oracle.partition`` — prefix-tree token cost and the optimal contiguous
                         split of the DFS order over K workers.
* ``oracle.dta``       — the depth-first traversal schedule of dynamic tree
                         attention (push / leaf / pop ops over chunks) and
                         attention executed through it with a KV stack.
* ``oracle.logprob``   — node-internal and transition log-probabilities,
                         entropies and vocabulary min/max of packed logits,
                         and the per-sequence merge.

Every floating-point routine accumulates in float64 on inputs that were
already rounded to bf16 by the caller.  Parity status of each function is
stated in its module header.
"""
