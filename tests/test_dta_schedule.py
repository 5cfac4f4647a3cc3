"""The library's DFS traversal schedule (tree_dta_schedule, host code)
against the oracle's, op for op (CPU only)."""
import json
import os

import numpy as np
import pytest

import prefix_tree_attention_gb300 as ptg
import workloads as W
from oracle import dta as OD
from oracle import trie as OT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lib_schedule(p, chunk):
    ops, peak = ptg.dta_schedule(p.token_node, p.node_entry, p.node_exit, chunk)
    return [tuple(int(x) for x in o) for o in ops], peak


def test_worked_example():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    with open(os.path.join(GOLDEN, "worked_example_dta.json")) as f:
        gd = json.load(f)
    (p,) = OT.pack_sequences(g["sequences"], g["max_tokens_per_mb"])
    for chunk, ops in gd["schedules"].items():
        got, peak = _lib_schedule(p, int(chunk))
        assert [list(o) for o in got] == ops
        assert peak == gd["peak_stack_tokens"][chunk]


@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 128, 2048])
def test_matches_oracle_on_random_tries(chunk):
    rng = W.SplitMix64(4000 + chunk)
    for _ in range(25):
        seqs = W.random_sequences(rng, rng.randint(1, 10), 60, 3)
        for p in OT.pack_sequences(seqs, 512):
            want = OD.schedule(p, chunk)
            got, peak = _lib_schedule(p, chunk)
            assert got == want
            assert peak == OD.peak_stack_tokens(want)


@pytest.mark.parametrize("key,chunk", [("tiny", 64), ("tiny", 2048), ("fanout", 2048),
                                       ("fanout", 1000)])
def test_matches_oracle_on_workloads(key, chunk):
    wl = W.WORKLOADS[key]
    for p in OT.pack_sequences(W.sequences(key), wl.max_tokens_per_mb):
        want = OD.schedule(p, chunk)
        got, peak = _lib_schedule(p, chunk)
        assert got == want and peak == OD.peak_stack_tokens(want)


def test_library_packer_tries_and_counts():
    # the library packer's arrays give the same schedule; op counts follow
    # from the chunking (every chunk is forwarded once and, unless it is a
    # leaf's last chunk, popped once)
    seqs = W.sequences("tiny")
    (tr,) = ptg.pack_sequences(seqs, W.WORKLOADS["tiny"].max_tokens_per_mb)
    (p,) = OT.pack_sequences(seqs, W.WORKLOADS["tiny"].max_tokens_per_mb)
    for chunk in (5, 100, 4096):
        a, pa = ptg.dta_schedule(tr.token_node, tr.node_entry, tr.node_exit, chunk)
        b, pb = _lib_schedule(p, chunk)
        assert [tuple(o) for o in a.tolist()] == b and pa == pb
        kinds = a[:, 0]
        n_chunks = sum(-(-(int(p.node_end[n]) - int(p.node_start[n]) + 1) // chunk)
                       for n in range(p.n_nodes))
        leaves = sum(1 for n in range(p.n_nodes) if not (p.node_parent == n).any())
        assert (kinds == OD.FWD_BWD).sum() == leaves
        assert (kinds == OD.FWD_PUSH).sum() == (kinds == OD.BWD_POP).sum() == n_chunks - leaves


def test_errors():
    (p,) = OT.pack_sequences([[1, 2, 3], [1, 4]], 128)
    tn, en, ex = p.token_node, p.node_entry, p.node_exit
    with pytest.raises(ptg.TreeError) as e:
        ptg.dta_schedule(tn, en, ex, 0)
    assert e.value.status == 1
    with pytest.raises(ptg.TreeError) as e:
        ptg.dta_schedule(tn[:100], en, ex, 8)
    assert e.value.status == 2
    bad = tn.copy()
    bad[1] = 7                                  # node id out of range
    with pytest.raises(ptg.TreeError) as e:
        ptg.dta_schedule(bad, en, ex, 8)
    assert e.value.status == 4
    bad = tn.copy()
    bad[[0, 1]] = bad[[1, 0]]                   # nodes out of rank order
    with pytest.raises(ptg.TreeError) as e:
        ptg.dta_schedule(bad, en, ex, 8)
    assert e.value.status == 4
    ex_bad = ex.copy()
    ex_bad[0] = len(ex)                         # exit past the last rank
    with pytest.raises(ptg.TreeError) as e:
        ptg.dta_schedule(tn, en, ex_bad, 8)
    assert e.value.status == 4
    # an empty trie (all pads) schedules nothing
    ops, peak = ptg.dta_schedule(np.full(128, -1, np.int32), np.zeros(0, np.int32),
                                 np.zeros(0, np.int32), 8)
    assert ops.shape == (0, 3) and peak == 0
