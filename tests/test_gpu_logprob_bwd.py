"""GPU parity of the gradient of the log-probability / entropy gather
(``tree_merge_per_sequence_bwd`` then ``tree_logprobs_entropy_bwd``) against
the fp64 oracle, through the C ABI.

A loss with random per-sequence gradients ``g_lp[s, t]`` and ``g_ent[s, t]``
(the merged [n_seqs, max_len] layout) flows back through the two merges and
the row pass to the packed logits; the oracle walks each sequence's
(predicting row, label) pairs in float64.

Tolerances, derived from the kernel's arithmetic.  The row pass forms
d_v = p_v * w_v with p_v = 2^((x_v - lse) log2 e), w_v = -(G + E (x_v - lse
+ H)), using the forward's fp32 lse (within LSE_TOL = 2e-4 of exact) and
entropy (within ENT_TOL = 2e-3), and G, the fp32 sum of the children's
gradients (relative rounding below 1e-6 of the sum of their magnitudes).  So
    |d~ - d| <= p (|w| (LSE_TOL + 1e-5) + 1e-6 Gabs + |E| (ENT_TOL + LSE_TOL)
                   + 1e-6 (|A| + |E x|)) + half an output ulp of |d|,
plus 1e-7 of the label gradient at the label entry.  The merge's adjoint is
a sum of fp32 values in atomic order: within 1e-6 of the sum of their
magnitudes.
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
HALF_ULP = {torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -24}   # unit roundoff


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype).to(DEV)


def _seq_grads(seq_ids, lens, seed, lp=True, ent=True):
    rng = np.random.default_rng(seed)
    return {s: (rng.standard_normal(lens[s] - 1) if lp else None,
                rng.standard_normal(lens[s] - 1) if ent else None) for s in seq_ids}


class _Case:
    """One trie on the device with its forward outputs."""

    def __init__(self, packed, logits, tok=None):
        self.packed, self.logits = packed, logits
        T = packed.T_pad
        self.tok_host = packed.token_ids if tok is None else tok
        self.tok = _dev(self.tok_host)
        self.bufs = ptg.TrieBuffers(T, packed.n_nodes, 1, 64)
        b = self.bufs
        ptg.tree_pack_positions(_dev(packed.token_node), _dev(packed.node_entry),
                                _dev(packed.node_exit), b.position_ids, b.key_reach, b.pos_ws,
                                b.status)
        ptg.tree_blockmap_build(b.key_reach, b.blockmap, b.status)
        f = dict(dtype=torch.float32, device=DEV)
        self.lse, self.ent = torch.empty(T, **f), torch.empty(T, **f)
        ptg.tree_logprobs_entropy(logits, b.key_reach, self.lse, b.status, entropy=self.ent)
        torch.cuda.synchronize()
        assert int(b.status.item()) == 0


def _merge_bwd(case, grads, n_seqs, pad_value=np.nan):
    """Per-sequence gradients -> packed per-token / per-row gradients on the
    device through tree_merge_per_sequence_bwd.  Entries past a sequence's
    length hold ``pad_value`` and must not be read."""
    tr = case.packed
    pos, offs = ptg.sequence_index_arrays([tr], n_seqs, [0])
    max_len = max(len(tr.seq_index[s]) for s in grads) - 1
    g_lp = np.full((n_seqs, max_len), pad_value, np.float32)
    g_ent = np.full((n_seqs, max_len), pad_value, np.float32)
    for s, (a, b) in grads.items():
        n = len(tr.seq_index[s]) - 1
        g_lp[s, :n] = 0.0 if a is None else a
        g_ent[s, :n] = 0.0 if b is None else b
    f = dict(dtype=torch.float32, device=DEV)
    tok_g, row_g = torch.zeros(tr.T_pad, **f), torch.zeros(tr.T_pad, **f)
    st = case.bufs.status
    pos_d, offs_d = _dev(pos), _dev(offs, torch.int64)
    ptg.tree_merge_per_sequence_bwd(_dev(g_lp, torch.float32), pos_d, offs_d, tok_g, st, 1, 1)
    ptg.tree_merge_per_sequence_bwd(_dev(g_ent, torch.float32), pos_d, offs_d, row_g, st, 0, 1)
    return tok_g, row_g


def _packed_grads(tr, grads):
    """float64 per-token / per-row sums and sums of magnitudes (numpy)."""
    T = tr.T_pad
    tok, row, tok_abs, row_abs = (np.zeros(T) for _ in range(4))
    for s, (a, b) in grads.items():
        idx = np.asarray(tr.seq_index[s])
        if a is not None:
            np.add.at(tok, idx[1:], a)
            np.add.at(tok_abs, idx[1:], np.abs(a))
        if b is not None:
            np.add.at(row, idx[:-1], b)
            np.add.at(row_abs, idx[:-1], np.abs(b))
    return tok, row, tok_abs, row_abs


def _row_bwd(case, tok_g, row_g, with_lp=True, with_ent=True, stride=None, fill=np.nan):
    lg = case.logits
    T, V = lg.shape
    width = V if stride is None else stride
    gbuf = torch.full((T, width), fill, dtype=lg.dtype, device=DEV)
    grad = gbuf[:, :V]
    ptg.tree_logprobs_entropy_bwd(lg, case.bufs.key_reach, case.lse, grad, case.bufs.status,
                                  token_ids=case.tok if with_lp else None,
                                  entropy=case.ent if with_ent else None,
                                  grad_logprob=tok_g if with_lp else None,
                                  grad_entropy=row_g if with_ent else None)
    torch.cuda.synchronize()
    return gbuf, grad


def _check_rows(case, got, want_rows, grads, dtype):
    """Compare kernel gradient rows with the oracle's within the derived bound."""
    tr = case.packed
    tok, row, tok_abs, _ = _packed_grads(tr, grads)
    pred = OL.token_pred(tr)
    for r, want in want_rows.items():
        g = got[r].float().cpu().numpy().astype(np.float64)
        if tr.token_node[r] < 0:
            assert (g == 0).all(), r
            continue
        x = case.logits[r].float().cpu().numpy().astype(np.float64)
        lq = OL.log_softmax(x)
        p = np.exp(lq)
        lse = float(x.max() + np.log(np.exp(x - x.max()).sum()))
        H = float(-(p * lq).sum())
        kids = np.nonzero(pred == r)[0]
        G, Gabs = float(tok[kids].sum()), float(tok_abs[kids].sum())
        E = float(row[r])
        A = G + E * (H - lse)
        w = -(A + E * x)
        tol = p * (np.abs(w) * (LSE_TOL + 1e-5) + 1e-6 * Gabs + abs(E) * (ENT_TOL + LSE_TOL)
                   + 1e-6 * (abs(A) + np.abs(E * x)))
        tol += 1.01 * HALF_ULP[dtype] * np.abs(want) + 1e-30
        for j in kids:
            tol[int(case.tok_host[j])] += 1e-7 * abs(tok[j]) + 1e-6 * tok_abs[j]
        bad = np.abs(g - want) > tol
        assert not bad.any(), (r, np.nonzero(bad)[0][:5], g[bad][:5], want[bad][:5])


def _full_case(seqs, V, dtype, seed, stride=None, max_tokens=2048):
    (packed,) = OT.pack_sequences(seqs, max_tokens)
    logits = W.logits(packed.T_pad, V, seed=seed, device=DEV, dtype=dtype, row_stride=stride)
    tok = np.where(packed.token_ids >= 0, packed.token_ids % V, -1).astype(np.int32)
    packed.token_ids = tok
    return _Case(packed, logits)


@pytest.mark.parametrize("V,dtype,stride", [
    (1001, torch.bfloat16, None),       # 125 16-byte groups + a ragged tail of 1
    (5003, torch.float32, None),        # fp32, ragged tail of 3
    (4096, torch.float32, 4099),        # rows not 16-byte aligned: element-wise path
    (333, torch.bfloat16, 341),         # unaligned bf16 rows
    (2048, torch.bfloat16, 2056),       # padded but 16-byte aligned rows
    (7, torch.bfloat16, None),          # fewer logits than one 16-byte group
])
def test_gradient_matches_oracle(V, dtype, stride):
    rng = W.SplitMix64(V + 1)
    seqs = W.random_sequences(rng, 12, 90, 3)
    case = _full_case(seqs, V, dtype, seed=V, stride=stride)
    tr = case.packed
    grads = _seq_grads(tr.seq_ids, {s: len(seqs[s]) for s in tr.seq_ids}, seed=V)
    tok_g, row_g = _merge_bwd(case, grads, len(seqs))
    gbuf, got = _row_bwd(case, tok_g, row_g, stride=stride)
    assert int(case.bufs.status.item()) == 0
    host = case.logits.float().cpu().numpy().astype(np.float64)
    want = OL.gather_packed_tree_backward(host, tr, grads)
    _check_rows(case, got, {r: want[r] for r in range(tr.T_pad)}, grads, dtype)
    if stride is not None:                 # entries past V are not touched
        assert torch.isnan(gbuf[:, V:].float()).all()


def test_merge_adjoint_matches_scatter_and_ignores_padding():
    rng = W.SplitMix64(17)
    seqs = W.random_sequences(rng, 16, 120, 2)
    case = _full_case(seqs, 64, torch.bfloat16, seed=3)
    tr = case.packed
    grads = _seq_grads(tr.seq_ids, {s: len(seqs[s]) for s in tr.seq_ids}, seed=4)
    tok_g, row_g = _merge_bwd(case, grads, len(seqs), pad_value=np.nan)   # NaN past lengths
    torch.cuda.synchronize()
    assert int(case.bufs.status.item()) == 0
    tok, row, tok_abs, row_abs = _packed_grads(tr, grads)
    g_tok, g_row = tok_g.cpu().numpy(), row_g.cpu().numpy()
    assert np.isfinite(g_tok).all() and np.isfinite(g_row).all()
    assert (np.abs(g_tok - tok) <= 1e-6 * tok_abs + 1e-30).all()
    assert (np.abs(g_row - row) <= 1e-6 * row_abs + 1e-30).all()
    # tokens that no entry reads (first tokens, pads) receive nothing
    firsts = [int(tr.seq_index[s][0]) for s in tr.seq_ids]
    assert (g_tok[firsts] == 0).all() and (g_tok[tr.n_tokens:] == 0).all()
    # the adjoint identity <merge(src), g> = <src, merge^T g> on the device
    n_seqs = len(seqs)
    pos, offs = ptg.sequence_index_arrays([tr], n_seqs, [0])
    src = torch.randn(tr.T_pad, device=DEV, dtype=torch.float32)
    adj = torch.zeros(tr.T_pad, device=DEV, dtype=torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pos_d, offs_d = _dev(pos), _dev(offs, torch.int64)
    for shift, trim in ((1, 1), (0, 1), (0, 0)):
        max_len = max(len(s) for s in seqs) - trim
        g = torch.randn((n_seqs, max_len), device=DEV, dtype=torch.float32)
        out = torch.empty_like(g)
        ptg.tree_merge_per_sequence(src, pos_d, offs_d, out, st, shift, trim, 0.0)
        adj.zero_()
        ptg.tree_merge_per_sequence_bwd(g, pos_d, offs_d, adj, st, shift, trim)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        lhs = float((out.double() * g.double()).sum())
        rhs = float((src.double() * adj.double()).sum())
        assert abs(lhs - rhs) <= 1e-5 * float((out.abs().double() * g.abs().double()).sum())
    # accumulation: a second call adds the same amount again
    adj2 = adj.clone()
    ptg.tree_merge_per_sequence_bwd(g, pos_d, offs_d, adj2, st, 0, 0)
    torch.cuda.synchronize()
    torch.testing.assert_close(adj2, 2 * adj, rtol=1e-6, atol=1e-6)
    # a max_len shorter than a sequence: CAPACITY (the entries that fit are added)
    short = torch.zeros((n_seqs, 2), device=DEV, dtype=torch.float32)
    ptg.tree_merge_per_sequence_bwd(short, pos_d, offs_d, adj, st, 1, 1)
    torch.cuda.synchronize()
    assert int(st.item()) == 3


@pytest.mark.parametrize("with_lp,with_ent", [(True, False), (False, True), (False, False)])
def test_gradient_with_one_or_no_term(with_lp, with_ent):
    rng = W.SplitMix64(5)
    seqs = W.random_sequences(rng, 8, 70, 2)
    case = _full_case(seqs, 777, torch.bfloat16, seed=6)
    tr = case.packed
    grads = _seq_grads(tr.seq_ids, {s: len(seqs[s]) for s in tr.seq_ids}, seed=7,
                       lp=with_lp, ent=with_ent)
    tok_g, row_g = _merge_bwd(case, grads, len(seqs))
    _, got = _row_bwd(case, tok_g, row_g, with_lp=with_lp, with_ent=with_ent)
    assert int(case.bufs.status.item()) == 0
    host = case.logits.float().cpu().numpy().astype(np.float64)
    want = OL.gather_packed_tree_backward(host, tr, grads)
    _check_rows(case, got, {r: want[r] for r in range(tr.T_pad)}, grads, torch.bfloat16)
    if not (with_lp or with_ent):
        assert (got.float() == 0).all()


def test_gradient_wide_fanout_and_forest():
    # a 10-token prefix with 40 children (distinct first tokens) of 1-60
    # tokens, children with their own branches, and single-token and
    # unrelated top-level sequences
    rng = W.SplitMix64(41)
    prefix = [rng.randint(1, 30) for _ in range(10)]
    seqs = [prefix + [100 + k] + [rng.randint(1, 900) for _ in range(rng.randint(0, 60))]
            for k in range(40)]
    seqs += [prefix + [100, 7, 7], prefix + [100, 7, 8], [3], [4], [5, 6, 7]]
    case = _full_case(seqs, 1024, torch.bfloat16, seed=9, max_tokens=4096)
    tr = case.packed
    grads = _seq_grads(tr.seq_ids, {s: len(seqs[s]) for s in tr.seq_ids}, seed=10)
    tok_g, row_g = _merge_bwd(case, grads, len(seqs))
    _, got = _row_bwd(case, tok_g, row_g)
    assert int(case.bufs.status.item()) == 0
    host = case.logits.float().cpu().numpy().astype(np.float64)
    want = OL.gather_packed_tree_backward(host, tr, grads)
    _check_rows(case, got, {r: want[r] for r in range(tr.T_pad)}, grads, torch.bfloat16)
    # the prefix's last row predicts 40 distinct first tokens
    assert (OL.token_pred(tr) == 9).sum() == 40


def test_gradient_is_deterministic_and_edge_cases():
    rng = W.SplitMix64(12)
    seqs = W.random_sequences(rng, 10, 80, 3)
    case = _full_case(seqs, 999, torch.bfloat16, seed=12)
    tr = case.packed
    grads = _seq_grads(tr.seq_ids, {s: len(seqs[s]) for s in tr.seq_ids}, seed=13)
    tok_g, row_g = _merge_bwd(case, grads, len(seqs))
    _, a = _row_bwd(case, tok_g, row_g)
    _, b = _row_bwd(case, tok_g, row_g)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # a single-token sequence predicts nothing: its row's gradient is 0
    one = _full_case([[5]], 64, torch.bfloat16, seed=2)
    g = {0: (np.zeros(0), np.zeros(0))}
    tok_g, row_g = _merge_bwd(one, g, 1)
    _, got = _row_bwd(one, tok_g, row_g)
    assert int(one.bufs.status.item()) == 0 and (got.float() == 0).all()
    # a child's id outside [0, V): MALFORMED_TREE
    bad = _full_case([[1, 2, 3]], 64, torch.bfloat16, seed=3)
    bad.tok_host = bad.tok_host.copy()
    bad.tok_host[2] = 64
    bad.tok = _dev(bad.tok_host)
    g = {0: (np.ones(2), np.ones(2))}
    tok_g, row_g = _merge_bwd(bad, g, 1)
    _row_bwd(bad, tok_g, row_g)
    assert int(bad.bufs.status.item()) == 4
    # T_pad == 0: nothing is launched
    empty = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    z = torch.empty(0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ptg.tree_logprobs_entropy_bwd(empty, torch.empty(0, dtype=torch.int32, device=DEV), z,
                                  torch.empty_like(empty), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


class _HostRows:
    """Rows of a device logits tensor fetched one at a time, float64."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, r):
        return self.t[int(r)].float().cpu().numpy().astype(np.float64)


def _sampled_rows(tr, n, seed):
    rng = W.SplitMix64(seed)
    pred = OL.token_pred(tr)
    kids = np.bincount(pred[pred >= 0], minlength=tr.T_pad)
    branch = [int(r) for r in np.argsort(-kids)[:4]]           # the widest branch rows
    leaves = [int(tr.seq_index[s][-1]) for s in list(tr.seq_ids)[:3]]   # predict nothing
    rows = {rng.randint(0, tr.n_tokens - 1) for _ in range(n)} | set(branch) | set(leaves)
    rows |= {tr.T_pad - 1} if tr.T_pad > tr.n_tokens else set()
    return sorted(rows)


@pytest.mark.parametrize("name", ["tiny", "grpo"])
def test_gradient_workload_qwen3_vocab_sampled(name):
    """The tiny workload and the bench's first grpo trie (T_pad 32640,
    9.9 GB of bf16 logits at the Qwen3 vocabulary): the whole gradient is
    computed on the device, sampled rows (the widest branch rows, leaf rows
    that predict nothing, random rows, a pad) against the oracle."""
    wl = W.WORKLOADS[name]
    seqs = W.sequences(name)
    tr = OT.pack_sequences(seqs, wl.max_tokens_per_mb)[0]     # the library's packer agrees
    logits = W.logits(tr.T_pad, QWEN3_VOCAB, seed=0, device=DEV)
    tr.token_ids = np.where(tr.token_ids >= 0, tr.token_ids % QWEN3_VOCAB, -1).astype(np.int32)
    case = _Case(tr, logits)
    grads = _seq_grads(tr.seq_ids, {s: len(tr.seq_index[s]) for s in tr.seq_ids}, seed=1)
    tok_g, row_g = _merge_bwd(case, grads, len(seqs))
    gbuf, got = _row_bwd(case, tok_g, row_g)
    del gbuf
    assert int(case.bufs.status.item()) == 0
    rows = _sampled_rows(tr, 24 if name == "grpo" else 40, seed=2)
    want = OL.gather_packed_tree_backward(_HostRows(logits), tr, grads, rows=rows)
    _check_rows(case, got, want, grads, torch.bfloat16)
