"""Pins for the oracle's tree-aware log-probability / entropy gather (CPU only).

Each check compares the oracle with something other than itself: the
hand-derived worked example of the packing figure (tests/golden), the
textbook per-sequence computation (scipy's log_softmax and entropy on each
sequence's own rows with labels shifted by one), closed forms, and brute
force over small tries against the dense ancestor mask.
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.special import log_softmax as sp_log_softmax
from scipy.special import logsumexp, softmax
from scipy.stats import entropy as sp_entropy

import workloads as W
from oracle import logprob as OL
from oracle import mask as OM
from oracle import trie as OT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _logits(T, V, seed):
    return W.logits(T, V, seed).float().numpy().astype(np.float64)


def _unpacked_reference(logits, packed, sid):
    """Textbook per-sequence computation: the sequence's own rows, labels =
    its tokens shifted by one, scipy log_softmax / entropy."""
    idx = packed.seq_index[sid]
    rows = logits[idx]
    toks = packed.token_ids[idx]
    lsm = sp_log_softmax(rows[:-1], axis=1)
    lp = lsm[np.arange(len(idx) - 1), toks[1:]]
    ent = sp_entropy(softmax(rows[:-1], axis=1), axis=1)
    return lp, ent, rows[:-1].min(axis=1), rows[:-1].max(axis=1)


def test_worked_example_predecessors_and_pairs():
    g = _golden("worked_example.json")
    gl = _golden("worked_example_logprob.json")
    (p,) = OT.pack_sequences(g["sequences"], g["max_tokens_per_mb"])
    pred = OL.token_pred(p)
    assert pred[:8].tolist() == gl["token_pred"]
    assert (pred[8:] == -1).all()
    V = 16
    logits = _logits(p.T_pad, V, 3)
    res, gat = OL.gather_packed_tree_logprobs_entropy(logits, p)
    for sid, pairs in gl["sequence_pairs"].items():
        lp, ent = res[int(sid)]
        want = [sp_log_softmax(logits[a])[p.token_ids[b]] for a, b in pairs]
        np.testing.assert_allclose(lp, want, rtol=0, atol=1e-13)
        assert ent.shape == (len(pairs),)
    internal = sorted(k for k, v in gat.internal_cache.items() if v.size)
    assert [list(k) for k in internal] == gl["internal_keys_with_labels"]
    assert sorted(map(list, gat.transition_cache)) == sorted(gl["transition_keys"])
    n_labels = sum(v.size for v in gat.internal_cache.values()) + len(gat.transition_cache)
    assert n_labels == gl["distinct_labels"]


def test_unpack_invariant_random_tries():
    rng = W.SplitMix64(2024)
    for trial in range(8):
        seqs = W.random_sequences(rng, rng.randint(2, 9), 40, 3)
        V = 37 + 11 * trial
        for t in OT.pack_sequences(seqs, 1024):
            logits = _logits(t.T_pad, V, trial)
            res, _ = OL.gather_packed_tree_logprobs_entropy(logits, t, with_stats=True)
            for sid in t.seq_ids:
                lp, ent, vmin, vmax = res[sid]
                rlp, rent, rmin, rmax = _unpacked_reference(logits, t, sid)
                assert lp.shape == (len(seqs[sid]) - 1,)
                np.testing.assert_allclose(lp, rlp, rtol=0, atol=1e-12)
                np.testing.assert_allclose(ent, rent, rtol=0, atol=1e-12)
                assert (vmin == rmin).all() and (vmax == rmax).all()


def test_packed_token_logprobs_match_sequences():
    rng = W.SplitMix64(77)
    seqs = W.random_sequences(rng, 7, 60, 2)
    (t,) = OT.pack_sequences(seqs, 2048)
    logits = _logits(t.T_pad, 29, 5)
    per_tok = OL.packed_token_logprobs(logits, t)
    res, _ = OL.gather_packed_tree_logprobs_entropy(logits, t)
    for sid in t.seq_ids:
        idx = t.seq_index[sid]
        np.testing.assert_allclose(per_tok[idx[1:]], res[sid][0], rtol=0, atol=0)
        assert per_tok[idx[0]] == 0.0


def test_row_stats_closed_forms():
    V = 1000
    lse, ent, mn, mx = OL.row_stats(np.full(V, 3.25))
    assert abs(lse - (3.25 + np.log(V))) < 1e-12 and abs(ent - np.log(V)) < 1e-12
    assert mn == mx == 3.25
    np.testing.assert_allclose(OL.log_softmax(np.full(V, -7.0)), -np.log(V), atol=1e-13)
    row = np.zeros(V)
    row[17] = 1000.0
    lse, ent, mn, mx = OL.row_stats(row)
    assert abs(lse - 1000.0) < 1e-12 and 0 <= ent < 1e-300 + 1e-12
    assert abs(OL.log_softmax(row)[17]) < 1e-12
    # two-point distribution [0, ln 3]: p = (1/4, 3/4)
    lse, ent, _, _ = OL.row_stats([0.0, np.log(3.0)])
    assert abs(lse - np.log(4.0)) < 1e-15
    assert abs(ent - (0.25 * np.log(4.0) + 0.75 * np.log(4.0 / 3.0))) < 1e-15
    # shift invariance of log_softmax and entropy; lse shifts
    x = _logits(1, 513, 9)[0]
    a, b = OL.row_stats(x), OL.row_stats(x + 5.5)
    assert abs(b[0] - a[0] - 5.5) < 1e-12 and abs(b[1] - a[1]) < 1e-12
    assert abs(a[0] - logsumexp(x)) < 1e-12


def _reach_from_mask(M):
    T = M.shape[0]
    reach = np.arange(T) - 1
    for j in range(T):
        rows = np.nonzero(M[:, j])[0]
        if rows.size:
            reach[j] = rows.max()
    return reach


def _check_pred_small(seqs):
    for t in OT.pack_sequences(seqs, 2048):
        M = OM.ancestor_mask(t)
        pred = OL.token_pred(t)
        reach = _reach_from_mask(M)
        for j in range(t.T_pad):
            if t.token_node[j] < 0:
                assert pred[j] == -1
                continue
            vis = np.nonzero(M[j, :j])[0]
            # the last visible key before j in the dense mask
            assert pred[j] == (vis.max() if vis.size else -1)
            # interval form: the largest i < j whose reach covers j
            cand = [i for i in range(j) if reach[i] >= j]
            assert pred[j] == (max(cand) if cand else -1)
        # each sequence's consecutive tokens are (pred, label) pairs
        for sid in t.seq_ids:
            idx = t.seq_index[sid]
            assert pred[idx[0]] == -1
            assert (pred[idx[1:]] == idx[:-1]).all()


def test_brute_force_predecessors_exhaustive_pairs():
    pool = []
    for L in range(1, 4):
        pool.extend([list(s) for s in itertools.product((1, 2, 3), repeat=L)])
    for a, b in itertools.product(pool, repeat=2):
        _check_pred_small([a, b])


def test_brute_force_predecessors_sampled_sets():
    rng = W.SplitMix64(4321)
    for _ in range(200):
        _check_pred_small(W.random_sequences(rng, rng.randint(1, 6), 6, 3))


def test_every_label_computed_once():
    rng = W.SplitMix64(555)
    for _ in range(20):
        seqs = W.random_sequences(rng, rng.randint(1, 10), 30, 2)
        for t in OT.pack_sequences(seqs, 2048):
            logits = _logits(t.T_pad, 5, 1)
            _, gat = OL.gather_packed_tree_logprobs_entropy(logits, t)
            labels = sum(v.size for v in gat.internal_cache.values()) + len(gat.transition_cache)
            top_level = int((t.node_parent == -1).sum())
            assert labels == t.n_tokens - top_level


def test_merge_across_micro_batches():
    seqs = [[1, 2, 3, 4], [1, 2, 5], [9, 8], [1, 2, 3, 4, 5, 6]]
    # two micro-batches: sequences 0-1 and 2-3 packed separately
    t0 = OT.pack_sequences([seqs[0], seqs[1]], 128)[0]
    t1 = OT.pack_sequences([seqs[2], seqs[3]], 128)[0]
    l0, l1 = _logits(t0.T_pad, 11, 0), _logits(t1.T_pad, 11, 1)
    r0, _ = OL.gather_packed_tree_logprobs_entropy(l0, t0)
    r1, _ = OL.gather_packed_tree_logprobs_entropy(l1, t1)
    lp = [{sid: v[0] for sid, v in r0.items()},
          {sid + 2: v[0] for sid, v in r1.items()}]
    out = OL.merge_packed_tree_results(lp, 4, padding_value=-5.0)
    assert out.shape == (4, 5)
    want = [None, None, None, None]
    for sid, (a, b) in [(0, (t0, l0)), (1, (t0, l0)), (2, (t1, l1)), (3, (t1, l1))]:
        local = sid if sid < 2 else sid - 2
        want[sid] = _unpacked_reference(b, a, local)[0]
    for sid in range(4):
        n = len(seqs[sid]) - 1
        np.testing.assert_allclose(out[sid, :n], want[sid], rtol=0, atol=1e-12)
        assert (out[sid, n:] == -5.0).all()
    capped = OL.merge_packed_tree_results(lp, 4, padding_value=0.0, max_len=2)
    assert capped.shape == (4, 2)
    np.testing.assert_allclose(capped[3], want[3][:2], atol=1e-12)


@pytest.mark.parametrize("V,n", [(1000, 1), (1000, 2), (1001, 3), (151936, 8), (37, 5)])
def test_vocab_parallel_combine_equals_whole_row(V, n):
    x = _logits(1, V, V + n)[0]
    x[3] += 12.0                      # one slice holds most of the mass
    slices = OL.vocab_slices(V, n)
    assert slices[0][0] == 0 and slices[-1][1] == V
    assert all(b - a in (V // n, V // n + 1) for a, b in slices)
    parts = [OL.row_stats(x[a:b]) for a, b in slices]
    got = OL.combine_vocab_slices(parts)
    want = (logsumexp(x), sp_entropy(softmax(x)), x.min(), x.max())
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ backward
def _seq_grads(packed, seed, lp=True, ent=True):
    """Random gradients of a loss with respect to every sequence's
    log-probability and entropy vectors."""
    rng = np.random.default_rng(seed)
    out = {}
    for sid in packed.seq_ids:
        n = len(packed.seq_index[sid]) - 1
        out[sid] = (rng.standard_normal(n) if lp else None,
                    rng.standard_normal(n) if ent else None)
    return out


def _autograd_unpacked(logits, packed, grads):
    """d loss / d logits by float64 torch autograd through the per-sequence
    computation on the sequence's own rows (torch's log_softmax and the
    Categorical entropy), with loss = sum over sequences of
    g_lp . logprob + g_ent . entropy."""
    import torch
    X = torch.tensor(logits, dtype=torch.float64, requires_grad=True)
    loss = X.new_zeros(())
    for sid, (g_lp, g_ent) in grads.items():
        idx = np.asarray(packed.seq_index[sid])
        rows = X[torch.as_tensor(idx[:-1])]
        labels = torch.as_tensor(packed.token_ids[idx[1:]].astype(np.int64))
        if g_lp is not None:
            lp = torch.log_softmax(rows, dim=1).gather(1, labels[:, None])[:, 0]
            loss = loss + (torch.as_tensor(g_lp) * lp).sum()
        if g_ent is not None:
            ent = torch.distributions.Categorical(logits=rows).entropy()
            loss = loss + (torch.as_tensor(g_ent) * ent).sum()
    loss.backward()
    return X.grad.numpy()


def test_backward_equals_autograd_of_unpacked_sequences():
    rng = W.SplitMix64(99)
    for trial in range(6):
        seqs = W.random_sequences(rng, rng.randint(2, 9), 40, 3)
        V = 23 + 7 * trial
        for t in OT.pack_sequences(seqs, 1024):
            logits = _logits(t.T_pad, V, trial + 40)
            for lp, ent in ((True, True), (True, False), (False, True)):
                grads = _seq_grads(t, trial, lp, ent)
                got = OL.gather_packed_tree_backward(logits, t, grads)
                want = _autograd_unpacked(logits, t, grads)
                np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def _loss(logits, packed, grads):
    res, _ = OL.gather_packed_tree_logprobs_entropy(logits, packed)
    tot = 0.0
    for sid, (g_lp, g_ent) in grads.items():
        lp, ent = res[sid]
        tot += float(np.dot(g_lp, lp)) + float(np.dot(g_ent, ent))
    return tot


def test_backward_central_differences():
    seqs = [[1, 2, 3, 4], [1, 2, 5], [1, 6], [7, 3]]
    (t,) = OT.pack_sequences(seqs, 128)
    V = 7
    logits = _logits(t.T_pad, V, 11)
    grads = _seq_grads(t, 5)
    got = OL.gather_packed_tree_backward(logits, t, grads)
    h = 1e-5
    for r in range(t.n_tokens):
        for v in range(V):
            a, b = logits.copy(), logits.copy()
            a[r, v] += h
            b[r, v] -= h
            fd = (_loss(a, t, grads) - _loss(b, t, grads)) / (2 * h)
            assert abs(fd - got[r, v]) < 1e-8, (r, v, fd, got[r, v])


def test_backward_closed_forms():
    # one sequence [1, 2, 3] over uniform rows: softmax is 1/V and the
    # entropy is at its maximum, so its gradient vanishes
    V = 9
    (t,) = OT.pack_sequences([[1, 2, 3]], 128)
    logits = np.full((t.T_pad, V), 0.75)
    g = {0: (np.array([2.0, -3.0]), np.array([5.0, 7.0]))}
    got = OL.gather_packed_tree_backward(logits, t, g)
    want = np.zeros_like(logits)
    want[0] = -2.0 / V
    want[0, 2] += 2.0
    want[1] = 3.0 / V
    want[1, 3] -= 3.0
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
    # rows of the gradient sum to zero (softmax sums to 1) and pads and
    # rows that predict nothing get nothing
    rng = W.SplitMix64(8)
    seqs = W.random_sequences(rng, 6, 30, 2)
    (t,) = OT.pack_sequences(seqs, 2048)
    logits = _logits(t.T_pad, 31, 2)
    got = OL.gather_packed_tree_backward(logits, t, _seq_grads(t, 3))
    np.testing.assert_allclose(got.sum(axis=1), 0.0, atol=1e-12)
    predicting = np.zeros(t.T_pad, bool)
    predicting[OL.token_pred(t)[OL.token_pred(t) >= 0]] = True
    assert (got[~predicting] == 0).all()
    # the two-point row [0, ln 3] (p = 1/4, 3/4): d H / d x_0 = p0 p1 ln(p1/p0)
    (t,) = OT.pack_sequences([[0, 1]], 128)
    logits = np.zeros((t.T_pad, 2))
    logits[0, 1] = np.log(3.0)
    got = OL.gather_packed_tree_backward(logits, t, {0: (None, np.array([1.0]))})
    assert abs(got[0, 0] - 0.1875 * np.log(3.0)) < 1e-15
    assert abs(got[0, 1] + 0.1875 * np.log(3.0)) < 1e-15


def test_merge_backward_is_the_adjoint():
    rng = np.random.default_rng(4)
    res = [{0: rng.standard_normal(3), 1: rng.standard_normal(2)},
           {2: rng.standard_normal(1), 3: rng.standard_normal(5)}]
    for max_len in (None, 3):
        fwd = OL.merge_packed_tree_results(res, 4, padding_value=1.5, max_len=max_len)
        g = rng.standard_normal(fwd.shape)
        back = OL.merge_packed_tree_results_backward(g, res)
        # <merge(x) - merge(0), g> = sum over parts <x, merge^T g>
        zero = [{s: np.zeros_like(v) for s, v in part.items()} for part in res]
        lin = fwd - OL.merge_packed_tree_results(zero, 4, padding_value=1.5, max_len=max_len)
        lhs = float((lin * g).sum())
        rhs = sum(float(np.dot(part[s], bp[s])) for part, bp in zip(res, back) for s in part)
        assert abs(lhs - rhs) < 1e-12



# ------------------------------------------------------------------ LM head
def test_lm_head_logits_exact_products():
    rng = np.random.default_rng(3)
    hidden = rng.standard_normal((37, 16))
    # the identity: logits are the hidden states themselves
    np.testing.assert_array_equal(OL.lm_head_logits(hidden, np.eye(16)), hidden)
    # a permutation of vocabulary rows permutes the logits' columns
    perm = rng.permutation(16)
    np.testing.assert_array_equal(OL.lm_head_logits(hidden, np.eye(16)[perm]), hidden[:, perm])
    # rank one: hidden = a 1^T, weight = b 1^T gives H a b^T (small integers: exact)
    a, b = rng.integers(-8, 9, 37).astype(float), rng.integers(-8, 9, 11).astype(float)
    got = OL.lm_head_logits(np.outer(a, np.ones(16)), np.outer(b, np.ones(16)))
    np.testing.assert_array_equal(got, 16 * np.outer(a, b))
    # the gather on LM-head logits of identity weights is the gather on the
    # hidden states
    seqs = [[1, 2, 3, 4], [1, 2, 5], [6, 7]]
    (t,) = OT.pack_sequences(seqs, 128)
    h = rng.standard_normal((t.T_pad, 16))
    r1, _ = OL.gather_packed_tree_logprobs_entropy(OL.lm_head_logits(h, np.eye(16)), t)
    r2, _ = OL.gather_packed_tree_logprobs_entropy(h, t)
    for sid in t.seq_ids:
        np.testing.assert_array_equal(r1[sid][0], r2[sid][0])
