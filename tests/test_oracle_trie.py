"""Pins for the oracle's trie packing and mask (CPU only).

Each check compares the oracle with something other than itself: the worked
example of the packing figure (hand-derived, tests/golden), a hand-worked FFD
example, and brute force over small sequence sets where the answer follows
from the definitions (distinct prefixes, unpacked causal order).
"""
import itertools
import json
import os

import numpy as np
import pytest

import workloads as W
from oracle import mask as OM
from oracle import trie as OT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _membership_mask(packed, seqs):
    """M[i, j] from the unpacked semantics: some sequence passes both i and j
    with j at or before i in that sequence's own order."""
    T = packed.T_pad
    m = np.zeros((T, T), bool)
    for sid in packed.seq_ids:
        idx = packed.seq_index[sid]
        for a in range(len(idx)):
            m[idx[a], idx[: a + 1]] = True
    return m


def test_worked_example_compressed():
    g = _golden("worked_example.json")
    (p,) = OT.pack_sequences(g["sequences"], g["max_tokens_per_mb"])
    assert p.n_tokens == g["n_tokens"] and p.T_pad == g["T_pad"]
    n = g["n_tokens"]
    assert p.token_ids[:n].tolist() == g["token_ids"]
    assert (p.token_ids[n:] == -1).all() and (p.token_node[n:] == -1).all()
    assert p.token_node[:n].tolist() == g["token_node"]
    assert p.node_entry.tolist() == g["node_entry"]
    assert p.node_exit.tolist() == g["node_exit"]
    assert p.node_parent.tolist() == g["node_parent"]
    toks = [p.token_ids[p.node_start[r]:p.node_end[r] + 1].tolist() for r in range(p.n_nodes)]
    assert toks == g["compressed_nodes_tokens"]
    pos = OM.position_ids(p)
    assert pos[:n].tolist() == g["position_ids"] and (pos[n:] == 0).all()
    M = OM.ancestor_mask(p)
    for i, row in enumerate(g["mask_rows"]):
        assert np.nonzero(M[i])[0].tolist() == row
    assert not M[n:].any() and not M[:, n:].any()
    assert OM.visible_pairs(p) == g["visible_pairs"]
    assert sum(len(s) * (len(s) + 1) // 2 for s in g["sequences"]) == g["unpacked_causal_pairs"]
    num, den = g["tree_token_ratio"]
    assert OT.tree_token_ratio([p], g["sequences"]) == pytest.approx(num / den)
    assert OM.tile_classes(p).tolist() == g["tile_classes"]


def test_worked_example_uncompressed_same_mask():
    g = _golden("worked_example.json")
    (pc,) = OT.pack_sequences(g["sequences"], 2048)
    (pu,) = OT.pack_sequences(g["sequences"], 2048, compress_nodes=False)
    assert pu.token_node[:8].tolist() == g["uncompressed_token_node"]
    assert (pu.token_ids == pc.token_ids).all()
    assert (OM.ancestor_mask(pu) == OM.ancestor_mask(pc)).all()
    assert (OM.position_ids(pu) == OM.position_ids(pc)).all()


def test_ffd_hand_example():
    # Worked by hand, capacity 8 tokens, block 4.  FFD order: a(5) d(4) b(3)
    # c(3).  a opens trie 0 (5); d shares [1,2,3] -> +1 = 6; b shares [1,2]
    # -> +1 = 7; c shares nothing -> 10 > 8 -> opens trie 1.
    a, b, c, d = [1, 2, 3, 4, 5], [1, 2, 6], [7, 8, 9], [1, 2, 3, 10]
    tries = OT.pack_sequences([a, b, c, d], 8, block=4)
    assert [t.seq_ids for t in tries] == [[0, 3, 1], [2]]
    assert [t.n_tokens for t in tries] == [7, 3]
    assert [t.T_pad for t in tries] == [8, 4]
    # trie 0 preorder: [1,2] {3 {4,5} {10}} {6}: chain 4-5 compresses
    t0 = tries[0]
    toks = [t0.token_ids[t0.node_start[r]:t0.node_end[r] + 1].tolist() for r in range(t0.n_nodes)]
    assert toks == [[1, 2], [3], [4, 5], [10], [6]]
    assert t0.node_exit.tolist() == [4, 3, 2, 3, 4]


def test_validation_errors():
    with pytest.raises(ValueError):
        OT.pack_sequences([[1, 2]], 0)
    with pytest.raises(ValueError):
        OT.pack_sequences([[1, 2]], 100)          # not a multiple of 128
    with pytest.raises(ValueError):
        OT.pack_sequences([list(range(1, 200))], 128)   # longer than the cap
    with pytest.raises(ValueError):
        OT.pack_sequences([[]], 128)


def _all_seqs(alphabet, max_len):
    out = []
    for L in range(1, max_len + 1):
        out.extend([list(t) for t in itertools.product(range(1, alphabet + 1), repeat=L)])
    return out


def _check_small_set(seqs, cap=2048):
    tries = OT.pack_sequences(seqs, cap)
    assert sorted(s for t in tries for s in t.seq_ids) == list(range(len(seqs)))
    for t in tries:
        assert t.n_tokens <= cap
        members = [seqs[s] for s in t.seq_ids]
        prefixes = {tuple(s[:k]) for s in members for k in range(1, len(s) + 1)}
        assert t.n_tokens == len(prefixes)                    # one token per prefix
        pos = OM.position_ids(t)
        M = OM.ancestor_mask(t)
        assert (M == _membership_mask(t, seqs)).all()
        for sid in t.seq_ids:
            idx = t.seq_index[sid]
            assert t.token_ids[idx].tolist() == seqs[sid]    # span round trip
            assert pos[idx].tolist() == list(range(len(seqs[sid])))
        # closed form: position = depth of the token below the virtual root
        for i in range(t.n_tokens):
            n = int(t.token_node[i])
            depth = (i - t.node_start[n]) + sum(
                t.node_end[a] - t.node_start[a] + 1 for a in OM.ancestors_or_self(t, n)[1:])
            assert pos[i] == depth
        # compression does not change the mask
        (u,) = [x for x in OT.pack_sequences(members, cap, compress_nodes=False)]
        assert (OM.ancestor_mask(u) == _membership_mask(u, members)).all()


def test_brute_force_pairs_exhaustive():
    pool = _all_seqs(3, 3)                    # 39 sequences
    for a, b in itertools.product(pool, repeat=2):
        _check_small_set([a, b])


def test_brute_force_sets_sampled():
    pool = _all_seqs(3, 4)                    # 120 sequences
    rng = W.SplitMix64(1234)
    for _ in range(600):
        k = rng.randint(1, 4)
        _check_small_set([pool[rng.randint(0, len(pool) - 1)] for _ in range(k)])


def test_brute_force_tile_classes():
    rng = W.SplitMix64(99)
    for _ in range(6):
        seqs = [[rng.randint(1, 2) for _ in range(rng.randint(40, 300))] for _ in range(5)]
        for t in OT.pack_sequences(seqs, 1024):
            M = _membership_mask(t, seqs)
            nb = t.T_pad // 128
            cls = OM.tile_classes(t)
            for qa in range(nb):
                for kb in range(nb):
                    c = M[qa * 128:(qa + 1) * 128, kb * 128:(kb + 1) * 128].sum()
                    want = OM.EMPTY if c == 0 else (OM.FULL if c == 128 * 128 else OM.PARTIAL)
                    assert cls[qa, kb] == want


def test_pad_to_max_same_real_rows():
    seqs = W.sequences("tiny")
    (a,) = OT.pack_sequences(seqs, 2048)
    (b,) = OT.pack_sequences(seqs, 2048, pad_to_max=True)
    assert b.T_pad == 2048
    n = a.n_tokens
    assert (a.token_node[:n] == b.token_node[:n]).all()
    assert (OM.position_ids(a)[:n] == OM.position_ids(b)[:n]).all()
