"""Oracle tree-aware log-probability / entropy gather — TEST INFRASTRUCTURE ONLY.

Follows the AReaL Tree Training guide, section "Log Probability 计算：树结构的
特殊处理" (log-probabilities of packed trees), in its order:

1. every sequence of the trie is visited (``trie.all_sequence_ids``);
2. for every node on the sequence's path two kinds of log-probability are
   taken:
   * node-internal: the logits at packed rows ``start .. end-1`` of the node
     predict its own tokens at rows ``start+1 .. end``;
   * transition: the logits at the node's last row (``pred_pos = end``)
     predict the first token of the next node on the path
     (``label_pos = next_start``);
3. both are cached, internal pieces by ``(start, end)`` and transitions by
   ``(pred_pos, label_pos)``, so sequences that share a prefix reuse them;
4. the pieces are concatenated in path order into the sequence's own
   log-probability vector.

The same section names the companions: the entropy of the predictive
distributions (``gather_packed_tree_logprobs_entropy``), vocabulary min/max
statistics (``gather_packed_tree_vocab_stats``) and the merge of per-sequence
results of several micro-batches back into a ``[batch, max_len]`` layout
padded with ``padding_value`` (``merge_packed_tree_results``), and a
vocabulary-parallel mode (``tp_group``) in which each rank reduces a slice
of the vocabulary; ``combine_vocab_slices`` restates the combination of the
slices' row statistics.

Readings where the page is silent:
* the input is the packed logits ``[T_pad, V]`` (one row per packed token);
  log-softmax is the plain definition ``x - logsumexp(x)`` in float64 on the
  given values, with no temperature;
* a sequence of length L has L-1 log-probabilities: entry t is the
  log-probability of its token t+1 given the logits at the row of its token
  t.  Its entropy and vocabulary statistics are taken at the same L-1
  predicting rows (entry t: the distribution of the row of token t);
* ``chunk_size`` only bounds the page's peak memory and changes no value,
  so the oracle has no chunking.

Parity: pinned by the worked example of the packing figure (predecessor of
every token), by the unpack invariant (the tree gather equals the textbook
per-sequence computation with labels shifted by one, using scipy's
log_softmax), by closed forms (uniform logits; one dominant logit), by brute
force over small tries (the predecessor from parent pointers is the last
visible key before the token in the dense ancestor mask), and by the cache
count (every non-root-start token is a label exactly once); the slice
combination against scipy's logsumexp and entropy of the whole row.  The
backward (``gather_packed_tree_backward``, the gradient a training step takes
through the gather) is pinned by float64 torch autograd through the
per-sequence computation on the unpacked rows, by central differences of the
forward on tiny tries, and by closed forms (uniform rows; rows of the
gradient sum to zero).  ``lm_head_logits`` is pinned by weights whose
products are known exactly (the identity and a permutation give the hidden
states themselves, a rank-one pair gives H a b^T).  See
tests/test_oracle_logprob.py.
"""
from __future__ import annotations

import numpy as np


def log_softmax(row) -> np.ndarray:
    """``x - logsumexp(x)`` in float64, max-shifted."""
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    return x - (m + np.log(np.exp(x - m).sum()))


def row_stats(row):
    """(logsumexp, entropy, min, max) of one logits row, float64."""
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    lse = m + np.log(np.exp(x - m).sum())
    lp = x - lse
    ent = -(np.exp(lp) * lp).sum()
    return float(lse), float(ent), float(x.min()), float(m)


def path_nodes(packed, sid: int) -> list[int]:
    """Nodes that sequence ``sid`` passes, root side first."""
    idx = packed.seq_index[sid]
    nodes = packed.token_node[idx]
    out = [int(nodes[0])]
    for n in nodes[1:]:
        if int(n) != out[-1]:
            out.append(int(n))
    return out


class _Gather:
    """Steps 1-4 over one packed trie, with the page's two caches."""

    def __init__(self, logits, packed):
        self.logits = logits
        self.packed = packed
        self.internal_cache: dict[tuple[int, int], np.ndarray] = {}
        self.transition_cache: dict[tuple[int, int], float] = {}
        self.row_cache: dict[int, tuple] = {}

    def _row(self, p: int):
        if p not in self.row_cache:
            self.row_cache[p] = (log_softmax(self.logits[p]), row_stats(self.logits[p]))
        return self.row_cache[p]

    def internal(self, start: int, end: int) -> np.ndarray:
        key = (start, end)
        if key not in self.internal_cache:
            tok = self.packed.token_ids
            self.internal_cache[key] = np.array(
                [self._row(p)[0][tok[p + 1]] for p in range(start, end)], dtype=np.float64)
        return self.internal_cache[key]

    def transition(self, pred_pos: int, label_pos: int) -> float:
        key = (pred_pos, label_pos)
        if key not in self.transition_cache:
            self.transition_cache[key] = float(
                self._row(pred_pos)[0][self.packed.token_ids[label_pos]])
        return self.transition_cache[key]

    def sequence(self, sid: int):
        """(logprob[L-1], entropy[L-1], vocab_min[L-1], vocab_max[L-1])."""
        pk = self.packed
        nodes = path_nodes(pk, sid)
        lps: list[np.ndarray] = []
        pred_rows: list[int] = []
        for a, n in enumerate(nodes):
            start, end = int(pk.node_start[n]), int(pk.node_end[n])
            lps.append(self.internal(start, end))
            pred_rows.extend(range(start, end))
            if a + 1 < len(nodes):
                nxt = int(pk.node_start[nodes[a + 1]])
                lps.append(np.array([self.transition(end, nxt)]))
                pred_rows.append(end)
        lp = np.concatenate(lps) if lps else np.zeros(0)
        stats = [self._row(p)[1] for p in pred_rows]
        ent = np.array([s[1] for s in stats], dtype=np.float64)
        vmin = np.array([s[2] for s in stats], dtype=np.float64)
        vmax = np.array([s[3] for s in stats], dtype=np.float64)
        return lp, ent, vmin, vmax


def gather_packed_tree_logprobs_entropy(logits, packed, with_stats: bool = False):
    """Per-sequence log-probabilities and entropies of one packed trie.

    Returns ``{sid: (logprob, entropy)}`` (or ``(logprob, entropy, vmin, vmax)``
    with ``with_stats``) and the gather object, whose caches hold every
    distinct internal and transition piece that was computed.
    """
    g = _Gather(logits, packed)
    out = {}
    for sid in packed.seq_ids:
        lp, ent, vmin, vmax = g.sequence(sid)
        out[sid] = (lp, ent, vmin, vmax) if with_stats else (lp, ent)
    return out, g


def merge_packed_tree_results(results, n_seqs: int, padding_value: float = 0.0,
                              max_len: int | None = None) -> np.ndarray:
    """Per-sequence vectors of several micro-batches (a list of
    ``{sid: vector}``) into ``[n_seqs, max_len]`` by sequence id, short rows
    padded with ``padding_value``."""
    merged: dict[int, np.ndarray] = {}
    for res in results:
        for sid, vec in res.items():
            merged[sid] = np.asarray(vec, dtype=np.float64)
    if max_len is None:
        max_len = max((v.size for v in merged.values()), default=0)
    out = np.full((n_seqs, max_len), padding_value, dtype=np.float64)
    for sid, vec in merged.items():
        n = min(vec.size, max_len)
        out[sid, :n] = vec[:n]
    return out


def token_pred(packed) -> np.ndarray:
    """Packed row whose logits predict each token: the previous token of the
    same node, else the last token of the parent node; -1 for the first token
    of a top-level node and for pads.  Walks parent pointers."""
    pred = np.full(packed.T_pad, -1, np.int32)
    for j in range(packed.T_pad):
        n = int(packed.token_node[j])
        if n < 0:
            continue
        if j > int(packed.node_start[n]):
            pred[j] = j - 1
        else:
            par = int(packed.node_parent[n])
            if par >= 0:
                pred[j] = int(packed.node_end[par])
    return pred


def packed_token_logprobs(logits, packed) -> np.ndarray:
    """Per packed token j: log-probability of its token under the logits of
    its predecessor row (0 where there is none), float64."""
    pred = token_pred(packed)
    out = np.zeros(packed.T_pad, np.float64)
    for j in range(packed.T_pad):
        if pred[j] >= 0:
            out[j] = log_softmax(logits[pred[j]])[packed.token_ids[j]]
    return out


def vocab_slices(V: int, n_slices: int) -> list[tuple[int, int]]:
    """Contiguous vocabulary slices, as even as possible (the first V % n
    slices one entry longer)."""
    base, extra = divmod(V, n_slices)
    out, a = [], 0
    for r in range(n_slices):
        b = a + base + (1 if r < extra else 0)
        out.append((a, b))
        a = b
    return out


def combine_vocab_slices(stats) -> tuple[float, float, float, float]:
    """Row statistics of the whole vocabulary from those of its slices (the
    page's vocabulary-parallel ``tp_group`` mode: each rank reduces its slice
    of V).  ``stats`` holds each slice's (lse_r, entropy_r, min_r, max_r).
    With w_r = exp(lse_r - lse) the share of slice r in the softmax mass:
        lse     = log sum_r exp(lse_r)
        entropy = sum_r w_r * (entropy_r + lse - lse_r)
    (the entropy of the mixture of the slices' softmaxes with weights w_r)."""
    lses = np.array([s[0] for s in stats], dtype=np.float64)
    m = lses.max()
    lse = m + np.log(np.exp(lses - m).sum())
    w = np.exp(lses - lse)
    ent = float((w * (np.array([s[1] for s in stats]) + lse - lses)).sum())
    return float(lse), ent, float(min(s[2] for s in stats)), float(max(s[3] for s in stats))


def lm_head_logits(hidden, weight) -> np.ndarray:
    """The LM head that produces the gather's input: logits[r, v] =
    sum_k hidden[r, k] * weight[v, k] (one weight row per vocabulary entry),
    float64.  The same section's gather then runs on these logits; its
    chunking changes no value, so the oracle takes them whole (or for a
    subset of rows, ``hidden[rows]``)."""
    return np.asarray(hidden, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T


def sequence_pairs(packed, sid: int) -> list[tuple[int, int]]:
    """(predicting row, label row) of every entry of sequence ``sid``, in the
    order of steps 2 and 4: a node's internal pairs (r, r + 1) for r in
    start .. end-1, then the transition (end, next node's start)."""
    pairs: list[tuple[int, int]] = []
    nodes = path_nodes(packed, sid)
    for a, n in enumerate(nodes):
        start, end = int(packed.node_start[n]), int(packed.node_end[n])
        pairs.extend((r, r + 1) for r in range(start, end))
        if a + 1 < len(nodes):
            pairs.append((end, int(packed.node_start[nodes[a + 1]])))
    return pairs


def gather_packed_tree_backward(logits, packed, grads, rows=None):
    """Gradient of the gather with respect to the packed logits, float64.

    ``grads`` maps a sequence id to ``(g_lp, g_ent)``, the gradients of a
    loss with respect to that sequence's log-probability and entropy vectors
    (each of length L-1, or None for zero).  The page's gather is
    differentiable end to end: a piece served from a cache passes back the
    sum over every sequence that used it, so the walk below adds each
    sequence's entries to its predicting rows one by one.  Entry t, taken at
    row p with label y, adds
        g_lp[t]  * (onehot(y) - q)                   d logprob / d x_p
        g_ent[t] * (-q * (log q + H_p))              d entropy / d x_p
    with q = softmax(x_p) and H_p its entropy (the derivative of
    -sum q log q, using sum q = 1).  Rows that predict nothing stay 0.

    Returns the dense ``[T_pad, V]`` gradient; with ``rows`` (row indices)
    only the entries at those predicting rows are taken and a dict
    ``{row: gradient row}`` is returned, and ``logits`` need only support
    ``logits[row]`` for them (so large logits can stay where they are).
    """
    want = None if rows is None else {int(r) for r in rows}
    tok = packed.token_ids
    acc: dict[int, np.ndarray] = {}
    lsm: dict[int, np.ndarray] = {}
    for sid, (g_lp, g_ent) in grads.items():
        for t, (p, lab) in enumerate(sequence_pairs(packed, sid)):
            if want is not None and p not in want:
                continue
            if p not in lsm:
                lsm[p] = log_softmax(np.asarray(logits[p], dtype=np.float64))
            lq = lsm[p]
            q = np.exp(lq)
            out = acc.setdefault(p, np.zeros_like(lq))
            if g_lp is not None:
                out -= g_lp[t] * q
                out[tok[lab]] += g_lp[t]
            if g_ent is not None:
                h = -(q * lq).sum()
                out -= g_ent[t] * q * (lq + h)
    if want is not None:
        return {r: acc.get(r, np.zeros(np.asarray(logits[r]).shape[-1])) for r in sorted(want)}
    dense = np.zeros(np.shape(logits), dtype=np.float64)
    for p, v in acc.items():
        dense[p] = v
    return dense


def merge_packed_tree_results_backward(grad_out, results) -> list[dict]:
    """Adjoint of ``merge_packed_tree_results``: the merged gradient
    ``[n_seqs, max_len]`` back into each micro-batch's ``{sid: vector}``
    (entries past a sequence's length, or past max_len, receive nothing)."""
    g = np.asarray(grad_out, dtype=np.float64)
    out = []
    for res in results:
        part = {}
        for sid, vec in res.items():
            n = np.asarray(vec).size
            v = np.zeros(n, np.float64)
            k = min(n, g.shape[1])
            v[:k] = g[sid, :k]
            part[sid] = v
        out.append(part)
    return out
