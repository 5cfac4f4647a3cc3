"""GPU parity of the LM head fused with the log-prob gather
(``tree_lm_head_logprobs_entropy``) against the fp64 oracle
(``lm_head_logits`` then the gather), through the C ABI.

Bit-exact: every token's predicting row, and the zeros of pads.

Floating point.  The kernel's logits are fp32 sums of bf16 products: the
tensor cores add H/16 blocks of 16 exact products into an fp32 accumulator,
one rounding per block, so |x~ - x| <= (H/16) 2^-24 sum_k |h_k w_k| <=
2^-24 (H/16) ||h_r|| max_v ||w_v|| =: delta_r (Cauchy-Schwarz).  The label
logit's fp32 dot product (H/256 fused multiply-adds per lane, a 32-lane
tree) stays inside the same bound.  On top of the row-reduction error of
the materialised path (LSE_TOL 2e-4, ENT_TOL 2e-3, see test_gpu_logprob):
lse within LSE_TOL + delta_r, entropy within ENT_TOL + 2 delta_r, the
vocabulary min / max within delta_r, logprob within LSE_TOL + 2 delta_r.
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
QWEN3_VOCAB, QWEN3_HIDDEN = 151936, 4096
DEV = "cuda"


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype).to(DEV)


class _Run:
    def __init__(self, packed, hidden, weight, labels=True, stats=True):
        T = packed.T_pad
        V = weight.shape[0]
        self.bufs = ptg.TrieBuffers(T, packed.n_nodes, 1, 64)
        b = self.bufs
        ptg.tree_pack_positions(_dev(packed.token_node), _dev(packed.node_entry),
                                _dev(packed.node_exit), b.position_ids, b.key_reach, b.pos_ws,
                                b.status)
        ptg.tree_blockmap_build(b.key_reach, b.blockmap, b.status)
        f = dict(dtype=torch.float32, device=DEV)
        self.lse, self.ent = torch.full((T,), 7.0, **f), torch.full((T,), 7.0, **f)
        self.vmin, self.vmax = torch.full((T,), 7.0, **f), torch.full((T,), 7.0, **f)
        self.lp = torch.full((T,), 7.0, **f)
        self.pred = torch.full((T,), 7, dtype=torch.int32, device=DEV)
        ws = torch.empty(ptg.lm_head_workspace_bytes(T, V) // 4 + 4, **f)
        tok = np.where(packed.token_ids >= 0, packed.token_ids % V, -1).astype(np.int32)
        self.tok = tok
        ptg.tree_lm_head_logprobs_entropy(
            hidden, weight, b.key_reach, self.lse, ws, b.status, token_ids=_dev(tok),
            blockmap=b.blockmap, entropy=self.ent if stats else None,
            vocab_min=self.vmin if stats else None, vocab_max=self.vmax if stats else None,
            logprob=self.lp if labels else None, token_pred=self.pred if labels else None)
        torch.cuda.synchronize()


def _check(packed, hidden, weight, run, rows=None, stats=True, labels=True):
    st = int(run.bufs.status.item())
    assert st == 0, ptg.status_string(st)
    T = packed.T_pad
    real = packed.token_node >= 0
    h = hidden.float().cpu().numpy()
    w = weight.float().cpu().numpy()                 # exact bf16 values
    H = h.shape[1]
    slices = [(a, min(a + 16384, w.shape[0])) for a in range(0, w.shape[0], 16384)]
    w_norm = max(np.sqrt((w[a:b].astype(np.float64) ** 2).sum(axis=1)).max()
                 for a, b in slices)
    pred_want = OL.token_pred(packed)
    lse, ent = run.lse.cpu().numpy(), run.ent.cpu().numpy()
    vmin, vmax, lp = run.vmin.cpu().numpy(), run.vmax.cpu().numpy(), run.lp.cpu().numpy()
    pred = run.pred.cpu().numpy()
    rows = np.nonzero(real)[0] if rows is None else np.asarray(rows)
    need = sorted(set(int(r) for r in rows) | {int(pred_want[j]) for j in rows
                                               if pred_want[j] >= 0})
    hn = h[need].astype(np.float64)
    x = np.concatenate([OL.lm_head_logits(hn, w[a:b]) for a, b in slices], axis=1)
    xrow = {r: x[i] for i, r in enumerate(need)}
    delta = {r: 2.0 ** -24 * (H / 16) * np.sqrt((hn[i] ** 2).sum()) * w_norm
             for i, r in enumerate(need)}
    for r in rows:
        r = int(r)
        if not real[r]:
            continue
        w_lse, w_ent, w_min, w_max = OL.row_stats(xrow[r])
        d = delta[r]
        assert abs(lse[r] - w_lse) <= LSE_TOL + d, (r, lse[r], w_lse, d)
        if stats:
            assert abs(ent[r] - w_ent) <= ENT_TOL + 2 * d, (r, ent[r], w_ent)
            assert abs(vmin[r] - w_min) <= d and abs(vmax[r] - w_max) <= d, r
        if labels:
            assert pred[r] == pred_want[r], r
            p = pred_want[r]
            if p >= 0:
                want = OL.log_softmax(xrow[p])[run.tok[r]]
                assert abs(lp[r] - want) <= LSE_TOL + 2 * delta[p], (r, lp[r], want)
            else:
                assert lp[r] == 0.0
    pads = ~real
    for a in (lse,) + ((ent, vmin, vmax) if stats else ()):
        assert (a[pads] == 0).all()
    if labels:
        assert (lp[pads] == 0).all() and (pred[pads] == -1).all()
    else:
        assert (lp == 7.0).all() and (pred == 7).all()
    if not stats:
        assert (ent == 7.0).all() and (vmin == 7.0).all() and (vmax == 7.0).all()


@pytest.mark.parametrize("H,V", [
    (64, 256),        # one vocabulary tile, one hidden stage
    (128, 1000),      # ragged last tile (232 of 256 columns; its second half 104)
    (256, 2048 + 7),  # crosses a 2048-column chunk by 7 columns
    (1024, 5000),     # several chunks, 16 hidden stages
    (192, 129),       # fewer columns than one tile half plus one
])
def test_fused_matches_oracle(H, V):
    rng = W.SplitMix64(H + V)
    seqs = W.random_sequences(rng, 12, 120, 3)
    (packed,) = OT.pack_sequences(seqs, 4096)
    hidden, weight = W.lm_head(packed.T_pad, H, V, seed=H, device=DEV)
    run = _Run(packed, hidden, weight)
    _check(packed, hidden, weight, run)


def test_fused_without_labels_or_stats():
    rng = W.SplitMix64(5)
    seqs = W.random_sequences(rng, 6, 100, 2)
    (packed,) = OT.pack_sequences(seqs, 2048)
    hidden, weight = W.lm_head(packed.T_pad, 128, 777, seed=5, device=DEV)
    run = _Run(packed, hidden, weight, labels=False)
    _check(packed, hidden, weight, run, labels=False)
    run = _Run(packed, hidden, weight, stats=False)
    _check(packed, hidden, weight, run, stats=False)


def test_fused_many_row_blocks_and_forest():
    # more row blocks than one group of 16, so the work order wraps groups;
    # several top-level subtrees and a 40-child fan-out
    rng = W.SplitMix64(77)
    prefix = [rng.randint(1, 30) for _ in range(10)]
    seqs = [prefix + [100 + k] + [rng.randint(1, 900) for _ in range(rng.randint(0, 90))]
            for k in range(40)]
    seqs += W.random_sequences(rng, 30, 200, 2)
    (packed,) = OT.pack_sequences(seqs, 8192)
    assert packed.T_pad // 128 > 16
    hidden, weight = W.lm_head(packed.T_pad, 256, 3000, seed=7, device=DEV)
    run = _Run(packed, hidden, weight)
    _check(packed, hidden, weight, run)


def test_fused_edge_cases():
    # a single token: no label
    (packed,) = OT.pack_sequences([[5]], 128)
    hidden, weight = W.lm_head(packed.T_pad, 64, 300, seed=1, device=DEV)
    run = _Run(packed, hidden, weight)
    _check(packed, hidden, weight, run)
    assert run.pred.cpu().numpy()[0] == -1
    # a label id outside [0, V): MALFORMED_TREE and a NaN log-probability
    (packed,) = OT.pack_sequences([[1, 2, 3]], 128)
    hidden, weight = W.lm_head(packed.T_pad, 64, 300, seed=2, device=DEV)
    bufs = ptg.TrieBuffers(packed.T_pad, packed.n_nodes, 1, 64)
    ptg.tree_pack_positions(_dev(packed.token_node), _dev(packed.node_entry),
                            _dev(packed.node_exit), bufs.position_ids, bufs.key_reach,
                            bufs.pos_ws, bufs.status)
    ptg.tree_blockmap_build(bufs.key_reach, bufs.blockmap, bufs.status)
    tok = packed.token_ids.copy()
    tok[2] = 300
    f = dict(dtype=torch.float32, device=DEV)
    lse, lp = torch.empty(packed.T_pad, **f), torch.empty(packed.T_pad, **f)
    ws = torch.empty(ptg.lm_head_workspace_bytes(packed.T_pad, 300) // 4, **f)
    ptg.tree_lm_head_logprobs_entropy(hidden, weight, bufs.key_reach, lse, ws, bufs.status,
                                      token_ids=_dev(tok), blockmap=bufs.blockmap, logprob=lp)
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == 4 and np.isnan(lp.cpu().numpy()[2])
    # T_pad == 0 launches nothing
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    e = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    z = torch.empty(0, **f)
    ptg.tree_lm_head_logprobs_entropy(e, weight, torch.empty(0, dtype=torch.int32, device=DEV),
                                      z, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def _sample(packed, n, seed):
    rng = W.SplitMix64(seed)
    starts = sorted({int(idx[0]) for idx in packed.seq_index.values()})
    pred = OL.token_pred(packed)
    branch = [int(j) for j in np.nonzero((pred >= 0) & (pred != np.arange(packed.T_pad) - 1))[0]]
    rows = {rng.randint(0, packed.n_tokens - 1) for _ in range(n)}
    rows |= set(starts[:4]) | set(branch[:8]) | {packed.n_tokens - 1, packed.T_pad - 1}
    return sorted(rows)


@pytest.mark.parametrize("name", ["tiny", "grpo"])
def test_fused_qwen3_head_sampled(name):
    """Qwen3-8B's LM head (H = 4096, V = 151,936) on the tiny workload and on
    the bench's first grpo trie (T_pad 32,640: 40.8 TFLOP); sampled rows —
    random rows, node starts whose predicting row is a parent's last token,
    the last real row and a pad — against the oracle."""
    wl = W.WORKLOADS[name]
    (packed,) = OT.pack_sequences(W.sequences(name), wl.max_tokens_per_mb)[:1]
    hidden, weight = W.lm_head(packed.T_pad, QWEN3_HIDDEN, QWEN3_VOCAB, seed=3, device=DEV)
    run = _Run(packed, hidden, weight)
    _check(packed, hidden, weight, run, rows=_sample(packed, 24, 9))


# ------------------------------------------------------------------ gradient
HALF_ULP_BF16 = 2.0 ** -8   # unit roundoff of bf16


def _seq_grads(packed, seed, lp=True, ent=True):
    rng = np.random.default_rng(seed)
    return {s: (rng.standard_normal(len(packed.seq_index[s]) - 1) if lp else None,
                rng.standard_normal(len(packed.seq_index[s]) - 1) if ent else None)
            for s in packed.seq_ids}


def _packed_grads(packed, grads):
    T = packed.T_pad
    tok, row, tok_abs = np.zeros(T), np.zeros(T), np.zeros(T)
    for s, (a, b) in grads.items():
        idx = np.asarray(packed.seq_index[s])
        if a is not None:
            np.add.at(tok, idx[1:], a)
            np.add.at(tok_abs, idx[1:], np.abs(a))
        if b is not None:
            np.add.at(row, idx[:-1], b)
    return tok, row, tok_abs


class _HostLogits:
    """Rows of the LM-head logits, float64, computed on demand."""

    def __init__(self, h, w):
        self.h, self.w = h, w

    def __getitem__(self, r):
        return OL.lm_head_logits(self.h[int(r):int(r) + 1].astype(np.float64), self.w)[0]


def _run_grad(packed, hidden, weight, grads, chunks, with_lp=True, with_ent=True):
    """Fused forward, the merge adjoints on the device, then the chunked
    logits gradient; returns {row: gradient row (float64)} and the run."""
    run = _Run(packed, hidden, weight)
    assert int(run.bufs.status.item()) == 0
    T, V = packed.T_pad, weight.shape[0]
    n_seqs = max(packed.seq_ids) + 1
    pos, offs = ptg.sequence_index_arrays([packed], n_seqs, [0])
    max_len = max(len(packed.seq_index[s]) for s in packed.seq_ids) - 1
    g_lp = np.full((n_seqs, max_len), np.nan, np.float32)
    g_ent = np.full((n_seqs, max_len), np.nan, np.float32)
    for s, (a, b) in grads.items():
        n = len(packed.seq_index[s]) - 1
        g_lp[s, :n] = 0.0 if a is None else a
        g_ent[s, :n] = 0.0 if b is None else b
    f = dict(dtype=torch.float32, device=DEV)
    tok_g, row_g = torch.zeros(T, **f), torch.zeros(T, **f)
    st = run.bufs.status
    pos_d, offs_d = _dev(pos), _dev(offs, torch.int64)
    ptg.tree_merge_per_sequence_bwd(_dev(g_lp, torch.float32), pos_d, offs_d, tok_g, st, 1, 1)
    ptg.tree_merge_per_sequence_bwd(_dev(g_ent, torch.float32), pos_d, offs_d, row_g, st, 0, 1)
    out = {}
    width = (V + 7) // 8 * 8                  # rows 16-byte aligned, as the call requires
    for lo, hi in chunks:
        gbuf = torch.full((hi - lo, width), float("nan"), dtype=torch.bfloat16, device=DEV)
        grad = gbuf[:, :V]
        ws = torch.empty(ptg.lm_head_grad_workspace_bytes(hi - lo) // 4, **f)
        ptg.tree_lm_head_logits_grad(
            hidden, weight, run.bufs.key_reach, run.lse, grad, ws, st, lo, hi,
            token_ids=_dev(run.tok), entropy=run.ent,
            grad_logprob=tok_g if with_lp else None, grad_entropy=row_g if with_ent else None)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, ptg.status_string(int(st.item()))
        assert torch.isnan(gbuf[:, V:].float()).all()       # past V: untouched
        g = grad.float().cpu().numpy().astype(np.float64)
        for r in range(lo, hi):
            out[r] = g[r - lo]
    return out, run


def _check_grad(packed, hidden, weight, grads, got, rows):
    """Kernel gradient rows against the oracle within the derived bound:
    p (|w| (2 delta + LSE_TOL + 1e-5) + 1e-6 Gabs + |E| (ENT_TOL + LSE_TOL + 4 delta)
       + 1e-6 (|A| + |E x|)) + a bf16 unit roundoff of |d|, delta as for the forward."""
    h = hidden.float().cpu().numpy()
    w = weight.float().cpu().numpy().astype(np.float64)
    H = h.shape[1]
    w_norm = np.sqrt((w * w).sum(axis=1)).max()
    tok, row, tok_abs = _packed_grads(packed, grads)
    pred = OL.token_pred(packed)
    tok_ids = np.where(packed.token_ids >= 0, packed.token_ids % w.shape[0], -1)
    pk = _Relabel(packed, tok_ids)
    want_rows = OL.gather_packed_tree_backward(_HostLogits(h, w), pk, grads, rows=rows)
    for r in rows:
        g = got[r]
        if packed.token_node[r] < 0:
            assert (g == 0).all(), r
            continue
        x = _HostLogits(h, w)[r]
        lq = OL.log_softmax(x)
        p = np.exp(lq)
        lse = float(x.max() + np.log(np.exp(x - x.max()).sum()))
        Hr = float(-(p * lq).sum())
        kids = np.nonzero(pred == r)[0]
        G, Gabs, E = float(tok[kids].sum()), float(tok_abs[kids].sum()), float(row[r])
        A = G + E * (Hr - lse)
        wv = -(A + E * x)
        d = 2.0 ** -24 * (H / 16) * np.sqrt((h[r].astype(np.float64) ** 2).sum()) * w_norm
        tol = p * (np.abs(wv) * (2 * d + LSE_TOL + 1e-5) + 1e-6 * Gabs
                   + abs(E) * (ENT_TOL + LSE_TOL + 4 * d) + 1e-6 * (abs(A) + np.abs(E * x)))
        want = want_rows[r]
        tol += 1.01 * HALF_ULP_BF16 * np.abs(want) + 1e-30
        for j in kids:
            tol[int(tok_ids[j])] += 1e-7 * abs(tok[j]) + 1e-6 * tok_abs[j]
        bad = np.abs(g - want) > tol
        assert not bad.any(), (r, np.nonzero(bad)[0][:5], g[bad][:5], want[bad][:5])


class _Relabel:
    """The packed trie with its token ids folded into the vocabulary."""

    def __init__(self, packed, tok):
        self.__dict__.update(packed.__dict__)
        self.token_ids = tok


@pytest.mark.parametrize("H,V,with_lp,with_ent", [
    (128, 1000, True, True),
    (256, 2055, True, True),
    (64, 300, True, False),
    (64, 300, False, True),
])
def test_logits_grad_matches_oracle(H, V, with_lp, with_ent):
    rng = W.SplitMix64(H * 7 + V)
    seqs = W.random_sequences(rng, 10, 90, 3)
    (packed,) = OT.pack_sequences(seqs, 4096)
    hidden, weight = W.lm_head(packed.T_pad, H, V, seed=V, device=DEV)
    grads = _seq_grads(packed, seed=H, lp=with_lp, ent=with_ent)
    got, _ = _run_grad(packed, hidden, weight, grads, [(0, packed.T_pad)], with_lp, with_ent)
    _check_grad(packed, hidden, weight, grads, got, list(range(packed.T_pad)))


def test_logits_grad_in_chunks_and_fanout():
    # chunks that start past row 0 and end before T_pad; a 40-child fan-out
    # whose branch row sits in the first chunk while its children do not
    rng = W.SplitMix64(19)
    prefix = [rng.randint(1, 30) for _ in range(100)]
    seqs = [prefix + [100 + k] + [rng.randint(1, 900) for _ in range(rng.randint(0, 30))]
            for k in range(40)]
    seqs += W.random_sequences(rng, 8, 120, 2)
    (packed,) = OT.pack_sequences(seqs, 4096)
    T = packed.T_pad
    assert T >= 384
    hidden, weight = W.lm_head(T, 192, 1500, seed=4, device=DEV)
    grads = _seq_grads(packed, seed=5)
    chunks = [(0, 128), (128, 384), (384, T)] if T > 384 else [(0, 128), (128, 384)]
    got, _ = _run_grad(packed, hidden, weight, grads, chunks)
    _check_grad(packed, hidden, weight, grads, got, list(range(T)))


def test_logits_grad_qwen3_head_sampled():
    """Qwen3-8B's head (H = 4096, V = 151,936) on the tiny workload: the
    gradient of rows [0, 512) and [1024, T_pad), sampled rows against the
    oracle (the widest branch rows, random rows, a pad)."""
    wl = W.WORKLOADS["tiny"]
    (packed,) = OT.pack_sequences(W.sequences("tiny"), wl.max_tokens_per_mb)
    T = packed.T_pad
    hidden, weight = W.lm_head(T, QWEN3_HIDDEN, QWEN3_VOCAB, seed=6, device=DEV)
    grads = _seq_grads(packed, seed=7)
    got, _ = _run_grad(packed, hidden, weight, grads, [(0, 512), (1024, T)])
    pred = OL.token_pred(packed)
    kids = np.bincount(pred[pred >= 0], minlength=T)
    rng = W.SplitMix64(8)
    rows = {int(r) for r in np.argsort(-kids)[:3]} | {rng.randint(0, 511) for _ in range(6)}
    rows |= {rng.randint(1024, packed.n_tokens - 1) for _ in range(4)} | {T - 1}
    rows = sorted(r for r in rows if r < 512 or r >= 1024)
    _check_grad(packed, hidden, weight, grads, got, rows)
