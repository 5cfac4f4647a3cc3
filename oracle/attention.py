"""Oracle masked attention, forward and backward, fp64 — TEST INFRASTRUCTURE ONLY.

What it computes (AReaL Tree Training guide, packing figure and section
"两种注意力实现": the attention is ordinary softmax attention under the tree
mask; AREAL-DTA section 3 "Problem formalisation": the total loss is the sum
of per-sequence losses, so the gradient of a shared-prefix token sums the
contributions of all its continuations):

    S = scale * Q K^T            (query head h reads key/value head h // g)
    P = softmax(S masked by M)   (rows with no visible key: P = 0)
    O = P V,  LSE = log sum exp(S masked by M)
    dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D)
    dQ = scale * dS K,  dK = scale * dS^T Q

with dK and dV summed over the g query heads that share a key/value head.

Readings (the pages are silent): ``scale`` defaults to 1/sqrt(d); query head
h maps to key/value head h // (Hq / Hkv); a row with no visible key (a pad)
has O = 0, LSE = -inf and zero gradients.

Inputs are float64 arrays holding bf16-rounded values; nothing is rounded
inside.  Layouts: Q, O, dO, dQ ``[T, Hq, d]``; K, V, dK, dV ``[T, Hkv, d]``;
LSE ``[Hq, T]``.

Parity: pinned against torch's CPU float64 ``scaled_dot_product_attention``
(causal) and CPU autograd through a dense masked softmax, and by the unpack
invariant (each sequence inside the packed trie gets exactly the outputs and,
summed over sequences, the gradients of causal attention on that sequence
alone) — see tests/test_oracle_attention.py.
"""
from __future__ import annotations

import numpy as np

from .mask import ancestors_or_self, mask_rows


def _softmax_rows(s: np.ndarray, mask: np.ndarray):
    """Masked softmax of each row; returns (P, LSE) with empty rows -> 0, -inf."""
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=-1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.where(mask, np.exp(s - m_safe[..., None]), 0.0)
    l = e.sum(axis=-1)
    p = np.where(has[..., None], e / np.where(has, l, 1.0)[..., None], 0.0)
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    return p, lse


def forward(q, k, v, mask, scale=None):
    """Dense forward: returns O ``[T, Hq, d]`` and LSE ``[Hq, T]``."""
    T, Hq, d = q.shape
    g = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o = np.zeros_like(q)
    lse = np.empty((Hq, T))
    for h in range(Hq):
        kv = h // g
        s = scale * (q[:, h, :] @ k[:, kv, :].T)
        p, lse[h] = _softmax_rows(s, mask)
        o[:, h, :] = p @ v[:, kv, :]
    return o, lse


def backward(q, k, v, o, do, mask, scale=None):
    """Dense backward: returns dQ, dK, dV (dK, dV summed over shared heads)."""
    T, Hq, d = q.shape
    g = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        kv = h // g
        s = scale * (q[:, h, :] @ k[:, kv, :].T)
        p, _ = _softmax_rows(s, mask)
        dv[:, kv, :] += p.T @ do[:, h, :]
        dp = do[:, h, :] @ v[:, kv, :].T
        D = (do[:, h, :] * o[:, h, :]).sum(axis=-1)
        ds = p * (dp - D[:, None])
        dq[:, h, :] = scale * (ds @ k[:, kv, :])
        dk[:, kv, :] += scale * (ds.T @ q[:, h, :])
    return dq, dk, dv


def rows_forward_backward(q, k, v, do, packed, rows, heads, scale=None, key_grads=True):
    """Per-row forward and dQ for the listed query rows and query heads.

    Row ``i`` reads exactly the keys of its mask row (ancestor walk), so O,
    LSE and dQ of a row need nothing outside it.  Returns dicts keyed by
    (row, head): ``o``, ``lse``, ``dq``; also (when ``key_grads``) the
    partial dK/dV those rows contribute (``dk_part``/``dv_part``, dict keyed
    by kv head of ``[T, d]`` arrays) — complete only when ``rows`` covers
    every row.
    """
    d = q.shape[2]
    g = q.shape[1] // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    out_o, out_lse, out_dq = {}, {}, {}
    dk_part, dv_part = {}, {}
    for i in rows:
        keys = np.nonzero(mask_rows(packed, i, i + 1)[0])[0]
        gathered = {}                     # kv head -> (K rows, V rows) of this row
        for h in heads:
            kv = h // g
            if keys.size == 0:
                out_o[(i, h)] = np.zeros(d)
                out_lse[(i, h)] = -np.inf
                out_dq[(i, h)] = np.zeros(d)
                continue
            if kv not in gathered:
                gathered[kv] = (k[keys, kv, :], v[keys, kv, :])
            kk, vv = gathered[kv]
            s = scale * (kk @ q[i, h, :])
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            p = e / l
            o_i = p @ vv
            dp = vv @ do[i, h, :]
            D = do[i, h, :] @ o_i
            ds = p * (dp - D)
            out_o[(i, h)] = o_i
            out_lse[(i, h)] = m + np.log(l)
            out_dq[(i, h)] = scale * (ds @ kk)
            if not key_grads:
                continue
            if kv not in dk_part:
                dk_part[kv] = np.zeros((q.shape[0], d))
                dv_part[kv] = np.zeros((q.shape[0], d))
            dk_part[kv][keys] += scale * np.outer(ds, q[i, h, :])
            dv_part[kv][keys] += np.outer(p, do[i, h, :])
    return out_o, out_lse, out_dq, dk_part, dv_part


def rows_seeing_key(packed, j: int) -> np.ndarray:
    """Column ``j`` of the mask: every row i >= j whose ancestor chain holds
    node(j)."""
    nj = int(packed.token_node[j])
    if nj < 0:
        return np.zeros(0, np.int64)
    nodes = [n for n in range(packed.n_nodes)
             if nj in ancestors_or_self(packed, n)]
    rows = [np.arange(packed.node_start[n], packed.node_end[n] + 1) for n in nodes]
    rows = np.concatenate(rows)
    return np.sort(rows[rows >= j])


def key_grads(q, k, v, do, packed, keys, kv_heads, scale=None):
    """dK, dV of the listed keys (per kv head), summing every row that sees
    each key over the g query heads of that kv head.  Cost grows with the
    rows below the key, so callers sample keys from small subtrees."""
    d = q.shape[2]
    g = q.shape[1] // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    dk, dv = {}, {}
    for j in keys:
        rows = rows_seeing_key(packed, j)
        row_keys = {int(i): np.nonzero(mask_rows(packed, int(i), int(i) + 1)[0])[0]
                    for i in rows}
        for kv in kv_heads:
            acc_k = np.zeros(d)
            acc_v = np.zeros(d)
            for i in rows:
                ks = row_keys[int(i)]
                kk = k[ks, kv, :]
                vv = v[ks, kv, :]
                at = int(np.searchsorted(ks, j))
                for h in range(kv * g, (kv + 1) * g):
                    # row i's softmax over its own keys, then key j's share
                    s = scale * (kk @ q[i, h, :])
                    e = np.exp(s - s.max())
                    p = e / e.sum()
                    o_i = p @ vv
                    dp = vv @ do[i, h, :]
                    D = do[i, h, :] @ o_i
                    acc_v += p[at] * do[i, h, :]
                    acc_k += scale * p[at] * (dp[at] - D) * q[i, h, :]
            dk[(j, kv)] = acc_k
            dv[(j, kv)] = acc_v
    return dk, dv
