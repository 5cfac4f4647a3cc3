"""Pins for the oracle's masked attention (CPU only, float64).

The oracle's forward and backward are compared with library routines it does
not use (torch CPU float64 ``scaled_dot_product_attention`` and autograd),
and with the unpack invariant of the tree-training pages: every sequence of a
packed trie must see exactly the outputs of causal attention on that sequence
alone, and the packed gradients must equal the per-sequence gradients summed
over the sequences passing each token (AREAL-DTA, section 3 "Problem
formalisation": shared prefixes are computed once and their gradients sum the
contributions of all continuations).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import mask as OM
from oracle import trie as OT


def _rand(shape, rng):
    x = torch.from_numpy(rng.standard_normal(shape)).to(torch.bfloat16)
    return x.to(torch.float64).numpy()


def _expand_kv(x, g):
    """Query head h reads kv head h // g (the head-map reading)."""
    return np.repeat(x, g, axis=1)


def _sdpa_causal(q, k, v, scale):
    """torch float64 causal SDPA over one sequence, [L, H, d] layouts."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def _trie_case(seed=0, n_seqs=6, g=2, Hkv=2, d=32):
    rng = W.SplitMix64(seed)
    base = [rng.randint(1, 3) for _ in range(40)]
    seqs = []
    for _ in range(n_seqs):
        cut = rng.randint(1, 40)
        seqs.append(base[:cut] + [rng.randint(4, 9) for _ in range(rng.randint(1, 70))])
    (p,) = OT.pack_sequences(seqs, 4096)
    nrng = np.random.default_rng(seed)
    T = p.T_pad
    q = _rand((T, g * Hkv, d), nrng)
    k = _rand((T, Hkv, d), nrng)
    v = _rand((T, Hkv, d), nrng)
    do = _rand((T, g * Hkv, d), nrng)
    return seqs, p, q, k, v, do


def test_single_sequence_equals_causal_sdpa():
    nrng = np.random.default_rng(3)
    seq = list(range(1, 200))
    (p,) = OT.pack_sequences([seq], 2048)
    T, L = p.T_pad, len(seq)
    q, k, v = _rand((T, 4, 64), nrng), _rand((T, 2, 64), nrng), _rand((T, 2, 64), nrng)
    o, lse = OA.forward(q, k, v, OM.ancestor_mask(p), scale=0.125)
    want = _sdpa_causal(q[:L], _expand_kv(k[:L], 2), _expand_kv(v[:L], 2), 0.125)
    assert np.abs(o[:L] - want).max() < 1e-12
    assert (o[L:] == 0).all() and np.isneginf(lse[:, L:]).all()


def test_backward_equals_autograd_dense_mask():
    seqs, p, q, k, v, do = _trie_case(seed=5)
    M = OM.ancestor_mask(p)
    scale = 1 / np.sqrt(q.shape[2])
    o, _ = OA.forward(q, k, v, M, scale)
    dq, dk, dv = OA.backward(q, k, v, o, do, M, scale)
    g = q.shape[1] // k.shape[1]
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    ke = kt.repeat_interleave(g, dim=1)
    ve = vt.repeat_interleave(g, dim=1)
    s = torch.einsum("ihd,jhd->hij", qt, ke) * scale
    Mt = torch.from_numpy(M)[None]
    s = s.masked_fill(~Mt, float("-inf"))
    pt = torch.softmax(s, dim=-1).nan_to_num(0.0)         # pad rows -> 0
    ot = torch.einsum("hij,jhd->ihd", pt, ve)
    (ot * torch.from_numpy(do)).sum().backward()
    assert np.abs(ot.detach().numpy() - o).max() < 1e-12
    assert np.abs(qt.grad.numpy() - dq).max() < 1e-11
    assert np.abs(kt.grad.numpy() - dk).max() < 1e-11
    assert np.abs(vt.grad.numpy() - dv).max() < 1e-11


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_unpack_invariant_forward_and_backward(seed):
    seqs, p, q, k, v, do_unused = _trie_case(seed=seed)
    M = OM.ancestor_mask(p)
    d = q.shape[2]
    g = q.shape[1] // k.shape[1]
    scale = 1 / np.sqrt(d)
    o, lse = OA.forward(q, k, v, M, scale)
    nrng = np.random.default_rng(100 + seed)
    # per-sequence upstream gradients and their packed sum
    do = np.zeros_like(q)
    dos = {}
    for sid in p.seq_ids:
        idx = p.seq_index[sid]
        dos[sid] = _rand((len(idx), q.shape[1], d), nrng)
        np.add.at(do, idx, dos[sid])
    dq, dk, dv = OA.backward(q, k, v, o, do, M, scale)
    want_q = np.zeros_like(q)
    want_k = np.zeros_like(k)
    want_v = np.zeros_like(v)
    for sid in p.seq_ids:
        idx = p.seq_index[sid]
        qs = torch.tensor(q[idx], requires_grad=True)
        ks = torch.tensor(k[idx], requires_grad=True)
        vs = torch.tensor(v[idx], requires_grad=True)
        os_ = torch.nn.functional.scaled_dot_product_attention(
            qs.permute(1, 0, 2)[None], ks.repeat_interleave(g, 1).permute(1, 0, 2)[None],
            vs.repeat_interleave(g, 1).permute(1, 0, 2)[None], is_causal=True, scale=scale
        )[0].permute(1, 0, 2)
        assert np.abs(os_.detach().numpy() - o[idx]).max() < 1e-12
        (os_ * torch.from_numpy(dos[sid])).sum().backward()
        np.add.at(want_q, idx, qs.grad.numpy())
        np.add.at(want_k, idx, ks.grad.numpy())
        np.add.at(want_v, idx, vs.grad.numpy())
    assert np.abs(dq - want_q).max() < 1e-11
    assert np.abs(dk - want_k).max() < 1e-11
    assert np.abs(dv - want_v).max() < 1e-11
    pad = p.token_node < 0
    assert (o[pad] == 0).all() and (dq[pad] == 0).all()
    assert (dk[pad] == 0).all() and (dv[pad] == 0).all()
    assert np.isneginf(lse[:, pad]).all()


def test_rows_and_key_grads_match_dense():
    seqs, p, q, k, v, do = _trie_case(seed=7)
    M = OM.ancestor_mask(p)
    scale = 1 / np.sqrt(q.shape[2])
    o, lse = OA.forward(q, k, v, M, scale)
    dq, dk, dv = OA.backward(q, k, v, o, do, M, scale)
    rows = [0, 3, p.n_tokens - 1, p.n_tokens, p.T_pad - 1]
    ro, rl, rdq, _, _ = OA.rows_forward_backward(q, k, v, do, p, rows, range(q.shape[1]), scale)
    for i in rows:
        for h in range(q.shape[1]):
            assert np.abs(ro[(i, h)] - o[i, h]).max() < 1e-12
            assert np.abs(rdq[(i, h)] - dq[i, h]).max() < 1e-12
            assert rl[(i, h)] == lse[h, i] or abs(rl[(i, h)] - lse[h, i]) < 1e-12
    keys = [p.n_tokens - 1, p.n_tokens - 5, 2]
    kdk, kdv = OA.key_grads(q, k, v, do, p, keys, range(k.shape[1]), scale)
    for j in keys:
        for kv in range(k.shape[1]):
            assert np.abs(kdk[(j, kv)] - dk[j, kv]).max() < 1e-11
            assert np.abs(kdv[(j, kv)] - dv[j, kv]).max() < 1e-11
