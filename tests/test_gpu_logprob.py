"""GPU parity of the tree-aware log-probability / entropy gather against the
fp64 oracle, through the C ABI.

Bit-exact: every token's predicting row (``token_pred``), pads' zeros, the
vocabulary min / max (a max of bf16 or fp32 values is exact).

Floating point: the kernel reduces a row in fp32 with the hardware 2^x
approximation (relative error about 2^-22 per term).  Each thread sums about
V / 256 terms before a 256-way tree, every term at most 1 after rebasing,
so the sum s carries a relative rounding error below (V/256 + 16) * 2^-24,
about 4e-5 at V = 151936.  lse = m + ln s and logprob = x - lse then sit
within about 4e-5 of the exact values: the bound used is ``LSE_TOL`` = 2e-4.
The entropy ln 2 * (log2 s - t / s) also carries t / s, whose magnitude
(the mean of (m - x) log2 e under p) stays below about 20 for these logits,
so ``ENT_TOL`` = 2e-3.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import logprob as OL
from oracle import trie as OT

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefix_tree_attention_gb300 as ptg  # noqa: E402

LSE_TOL, ENT_TOL = 2e-4, 2e-3
QWEN3_VOCAB = 151936
DEV = "cuda"


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype).to(DEV)


def _positions_blockmap(packed):
    bufs = ptg.TrieBuffers(packed.T_pad, packed.n_nodes, 1, 64)
    ptg.tree_pack_positions(_dev(packed.token_node), _dev(packed.node_entry),
                            _dev(packed.node_exit), bufs.position_ids, bufs.key_reach,
                            bufs.pos_ws, bufs.status)
    ptg.tree_blockmap_build(bufs.key_reach, bufs.blockmap, bufs.status)
    return bufs


class _Out:
    def __init__(self, T):
        f = dict(dtype=torch.float32, device=DEV)
        self.lse = torch.full((T,), 7.0, **f)
        self.entropy = torch.full((T,), 7.0, **f)
        self.vmin = torch.full((T,), 7.0, **f)
        self.vmax = torch.full((T,), 7.0, **f)
        self.logprob = torch.full((T,), 7.0, **f)
        self.pred = torch.full((T,), 7, dtype=torch.int32, device=DEV)


def _run(packed, logits, with_min=True):
    bufs = _positions_blockmap(packed)
    out = _Out(packed.T_pad)
    ptg.tree_logprobs_entropy(logits, bufs.key_reach, out.lse, bufs.status,
                              token_ids=_dev(packed.token_ids), blockmap=bufs.blockmap,
                              entropy=out.entropy, vocab_min=out.vmin if with_min else None,
                              vocab_max=out.vmax, logprob=out.logprob, token_pred=out.pred)
    torch.cuda.synchronize()
    return bufs, out


def _check(packed, logits, out, bufs, rows=None, with_min=True):
    st = int(bufs.status.item())
    assert st == 0, ptg.status_string(st)
    T = packed.T_pad
    real = packed.token_node >= 0
    pred = out.pred.cpu().numpy()
    assert np.array_equal(pred, OL.token_pred(packed))
    host = logits.float().cpu().numpy().astype(np.float64) if rows is None else None
    rows = np.nonzero(real)[0] if rows is None else rows
    lse, ent = out.lse.cpu().numpy(), out.entropy.cpu().numpy()
    vmin, vmax, lp = out.vmin.cpu().numpy(), out.vmax.cpu().numpy(), out.logprob.cpu().numpy()
    for r in rows:
        x = host[r] if host is not None else logits[r].float().cpu().numpy().astype(np.float64)
        w_lse, w_ent, w_min, w_max = OL.row_stats(x)
        assert abs(lse[r] - w_lse) <= LSE_TOL, (r, lse[r], w_lse)
        assert abs(ent[r] - w_ent) <= ENT_TOL, (r, ent[r], w_ent)
        assert vmax[r] == w_max, r
        assert vmin[r] == w_min if with_min else vmin[r] == 7.0, r
    pads = ~real
    for a in (lse, ent, vmax, lp) + ((vmin,) if with_min else ()):
        assert (a[pads] == 0).all()
    if not with_min:                        # an output passed as NULL is not written
        assert (vmin == 7.0).all()
    assert (pred[pads] == -1).all()
    if host is not None:
        want = OL.packed_token_logprobs(host, packed)
        np.testing.assert_allclose(lp, want, rtol=0, atol=LSE_TOL)
    return lse, ent, lp, pred


def test_tiny_workload_qwen3_vocab_bf16():
    (packed,) = OT.pack_sequences(W.sequences("tiny"), W.WORKLOADS["tiny"].max_tokens_per_mb)
    assert packed.token_ids.max() < QWEN3_VOCAB
    logits = W.logits(packed.T_pad, QWEN3_VOCAB, seed=1, device=DEV)
    bufs, out = _run(packed, logits)
    _check(packed, logits, out, bufs)


@pytest.mark.parametrize("V,dtype,stride", [
    (1001, torch.bfloat16, None),       # 125 16-byte groups + a ragged tail of 1
    (50257, torch.float32, None),       # fp32, ragged tail of 1
    (4096, torch.float32, 4099),        # rows not 16-byte aligned: element-wise path
    (333, torch.bfloat16, 341),         # unaligned bf16 rows
    (7, torch.bfloat16, None),          # fewer logits than one 16-byte group
])
def test_dtypes_strides_and_ragged_vocab(V, dtype, stride):
    rng = W.SplitMix64(V)
    seqs = W.random_sequences(rng, 12, 90, 3)
    (packed,) = OT.pack_sequences(seqs, 2048)
    logits = W.logits(packed.T_pad, V, seed=V, device=DEV, dtype=dtype, row_stride=stride)
    assert logits.stride(0) == (V if stride is None else stride)
    with_min = V % 2 == 1
    bufs, out = _run(packed, logits, with_min=with_min)
    _check(packed, logits, out, bufs, with_min=with_min)


def test_long_sibling_skips_and_forest():
    # one 10-token prefix with 8 children of 300 tokens: child k's first token
    # must skip k - 1 earlier subtrees (several 128-token blocks each); then
    # 3 unrelated top-level sequences whose first tokens have no predecessor
    rng = W.SplitMix64(8)
    prefix = [rng.randint(1, 50) for _ in range(10)]
    seqs = [prefix + [1000 * (k + 1) + i for i in range(300)] for k in range(8)]
    seqs += [[90000 + 500 * k + i for i in range(rng.randint(1, 200))] for k in range(3)]
    (packed,) = OT.pack_sequences(seqs, 4096)
    logits = W.logits(packed.T_pad, 2048, seed=8, device=DEV)
    # token ids above the vocabulary are remapped so every label is in range
    packed.token_ids = np.where(packed.token_ids >= 0, packed.token_ids % 2048, -1).astype(np.int32)
    bufs, out = _run(packed, logits)
    _check(packed, logits, out, bufs)
    pred = out.pred.cpu().numpy()
    top_level = [int(packed.node_start[n]) for n in range(packed.n_nodes)
                 if packed.node_parent[n] == -1]
    assert len(top_level) == 4 and (pred[top_level] == -1).all()


def test_merge_over_micro_batches_matches_oracle():
    rng = W.SplitMix64(31)
    seqs = W.random_sequences(rng, 20, 150, 2)
    tries = OT.pack_sequences(seqs, 256)
    assert len(tries) > 1
    V = 512
    offs_t = np.cumsum([0] + [t.T_pad for t in tries]).tolist()
    total = offs_t[-1]
    lp_all = torch.zeros(total, dtype=torch.float32, device=DEV)
    ent_all = torch.zeros(total, dtype=torch.float32, device=DEV)
    want_lp, want_ent = [], []
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for i, t in enumerate(tries):
        logits = W.logits(t.T_pad, V, seed=100 + i, device=DEV)
        bufs = _positions_blockmap(t)
        sl = slice(offs_t[i], offs_t[i + 1])
        lse = torch.empty(t.T_pad, dtype=torch.float32, device=DEV)
        ptg.tree_logprobs_entropy(logits, bufs.key_reach, lse, bufs.status,
                                  token_ids=_dev(t.token_ids), blockmap=bufs.blockmap,
                                  entropy=ent_all[sl], logprob=lp_all[sl])
        torch.cuda.synchronize()
        assert int(bufs.status.item()) == 0
        res, _ = OL.gather_packed_tree_logprobs_entropy(
            logits.float().cpu().numpy().astype(np.float64), t)
        want_lp.append({sid: v[0] for sid, v in res.items()})
        want_ent.append({sid: v[1] for sid, v in res.items()})
    pos, offs = ptg.sequence_index_arrays(tries, len(seqs), offs_t[:-1])
    max_len = max(len(s) for s in seqs) - 1
    pos_d, offs_d = _dev(pos), _dev(offs, torch.int64)
    out_lp = torch.empty((len(seqs), max_len), dtype=torch.float32, device=DEV)
    out_ent = torch.empty_like(out_lp)
    ptg.tree_merge_per_sequence(lp_all, pos_d, offs_d, out_lp, status, shift=1, trim=1,
                                padding_value=-3.5)
    ptg.tree_merge_per_sequence(ent_all, pos_d, offs_d, out_ent, status, shift=0, trim=1,
                                padding_value=0.0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    e_lp = OL.merge_packed_tree_results(want_lp, len(seqs), -3.5, max_len)
    e_ent = OL.merge_packed_tree_results(want_ent, len(seqs), 0.0, max_len)
    got_lp, got_ent = out_lp.cpu().numpy(), out_ent.cpu().numpy()
    for sid, s in enumerate(seqs):
        n = len(s) - 1
        assert (got_lp[sid, n:] == -3.5).all() and (got_ent[sid, n:] == 0.0).all()
    np.testing.assert_allclose(got_lp, e_lp, rtol=0, atol=LSE_TOL)
    np.testing.assert_allclose(got_ent, e_ent, rtol=0, atol=ENT_TOL)
    # a max_len shorter than the longest sequence is reported as CAPACITY
    short = torch.empty((len(seqs), 3), dtype=torch.float32, device=DEV)
    ptg.tree_merge_per_sequence(lp_all, pos_d, offs_d, short, status, shift=1, trim=1)
    torch.cuda.synchronize()
    assert int(status.item()) == 3


def test_edge_cases_single_token_and_bad_ids():
    (packed,) = OT.pack_sequences([[5]], 128)
    logits = W.logits(packed.T_pad, 64, seed=2, device=DEV)
    bufs, out = _run(packed, logits)
    _check(packed, logits, out, bufs)
    assert out.pred.cpu().numpy()[0] == -1 and out.logprob.cpu().numpy()[0] == 0.0
    # a label id outside [0, V): MALFORMED_TREE and a NaN log-probability
    (packed,) = OT.pack_sequences([[1, 2, 3]], 128)
    packed.token_ids = packed.token_ids.copy()
    packed.token_ids[2] = 64
    logits = W.logits(packed.T_pad, 64, seed=3, device=DEV)
    bufs, out = _run(packed, logits)
    assert int(bufs.status.item()) == 4
    assert np.isnan(out.logprob.cpu().numpy()[2])
    # T_pad == 0: nothing is launched, nothing written
    empty = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    z = torch.empty(0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ptg.tree_logprobs_entropy(empty, torch.empty(0, dtype=torch.int32, device=DEV), z, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_grpo_trie0_full_size_sampled():
    """The bench's configuration: the first grpo trie (T_pad 32640) against
    the Qwen3 vocabulary in bf16 (9.9 GB of logits).  Every predecessor is
    checked by the sequence property; sampled rows against the oracle."""
    wl = W.WORKLOADS["grpo"]
    seqs = W.sequences("grpo")
    tr = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)[0]
    logits = W.logits(tr.T_pad, QWEN3_VOCAB, seed=0, device=DEV)
    # the workload's fresh token ids run past the vocabulary: fold them into it
    tok = np.where(tr.token_ids >= 0, tr.token_ids % QWEN3_VOCAB, -1).astype(np.int32)
    bufs = ptg.TrieBuffers(tr.T_pad, tr.n_nodes, 1, 64)
    ptg.tree_pack_positions(_dev(tr.token_node), _dev(tr.node_entry), _dev(tr.node_exit),
                            bufs.position_ids, bufs.key_reach, bufs.pos_ws, bufs.status)
    ptg.tree_blockmap_build(bufs.key_reach, bufs.blockmap, bufs.status)
    out = _Out(tr.T_pad)
    ptg.tree_logprobs_entropy(logits, bufs.key_reach, out.lse, bufs.status,
                              token_ids=_dev(tok), blockmap=bufs.blockmap,
                              entropy=out.entropy, vocab_max=out.vmax, logprob=out.logprob,
                              token_pred=out.pred)
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == 0
    pred = out.pred.cpu().numpy()
    for sid, idx in tr.seq_index.items():
        assert pred[idx[0]] == -1
        assert np.array_equal(pred[idx[1:]], idx[:-1])
    assert (pred[tr.n_tokens:] == -1).all()
    lse, ent, lp = out.lse.cpu().numpy(), out.entropy.cpu().numpy(), out.logprob.cpu().numpy()
    rng = W.SplitMix64(5)
    starts = sorted({int(idx[0]) for idx in tr.seq_index.values()})
    sample = {rng.randint(0, tr.n_tokens - 1) for _ in range(40)} | set(starts[:8])
    sample |= {tr.n_tokens - 1}
    for j in sorted(sample):
        x = logits[j].float().cpu().numpy().astype(np.float64)
        w_lse, w_ent, _, w_max = OL.row_stats(x)
        assert abs(lse[j] - w_lse) <= LSE_TOL and abs(ent[j] - w_ent) <= ENT_TOL, j
        assert out.vmax[j].item() == w_max
        p = pred[j]
        if p >= 0:
            xp = logits[p].float().cpu().numpy().astype(np.float64)
            want = OL.log_softmax(xp)[tok[j]]
            assert abs(lp[j] - want) <= LSE_TOL, j
        else:
            assert lp[j] == 0.0
