"""GPU parity of attention executed through the depth-first traversal of
dynamic tree attention (``tree_dta_attn``, AREAL-DTA sections 3.1-3.2).

The library runs the schedule op by op (row-windowed forward and backward
kernels, dK/dV added into fp32 accumulators across ops) and is compared
element by element with the oracle's attention through the same schedule
(``oracle/dta.py`` ``run_attention``: an explicit key/value stack, float64).
Bounds are those of the packed tests: every element within 2e-2 plus half a
bf16 ulp of the reference, mean error within 2e-3, LSE within 5e-3.  The
forward outputs must also equal the packed forward's bit for bit (the same
kernel computes the same blocks; only the rows written differ), and the
gradients the packed backward's within the same bounds.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import dta as OD
from oracle import trie as OT

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefix_tree_attention_gb300 as ptg  # noqa: E402

from test_gpu_parity import (LSE_ERR, assert_close, pack_both, run_attention,  # noqa: E402
                             run_positions_blockmap)

DEV = "cuda"


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_dta(bufs, t, ops):
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    o = torch.full_like(q, 7.0)          # garbage the init must overwrite
    lse = torch.full((Hq, T), 7.0, dtype=torch.float32, device=DEV)
    dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    ws = torch.full(((ptg.dta_attn_workspace_bytes(T, Hq, Hkv, d) + 3) // 4,), float("nan"),
                    dtype=torch.float32, device=DEV)
    ptg.tree_dta_attn(q, k, v, do, bufs.key_reach, bufs.blockmap, ops, o, lse, dq, dk, dv, ws,
                      bufs.status)
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == 0, ptg.status_string(int(bufs.status.item()))
    return o, lse, dq, dk, dv


def check_dta(p, Hq, Hkv, d, chunk, seed, kv_group=None):
    """Library schedule = oracle schedule; the DTA execution against the
    oracle's (optionally on one kv head's query heads only) and against the
    packed path."""
    ops, peak = ptg.dta_schedule(p.token_node, p.node_entry, p.node_exit, chunk)
    want_ops = OD.schedule(p, chunk)
    assert [tuple(o) for o in ops.tolist()] == [tuple(o) for o in want_ops]
    assert peak == OD.peak_stack_tokens(want_ops)
    t = W.tensors(p.T_pad, Hq, Hkv, d, seed=seed, device=DEV)
    bufs = run_positions_blockmap(p.token_node, p.node_entry, p.node_exit)
    o, lse, dq, dk, dv = run_dta(bufs, t, ops)
    real = p.token_node >= 0
    pad = torch.from_numpy(~real).to(DEV)
    # pads are never scheduled: they keep O = 0, LSE = -inf, zero gradients
    for name, x in (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)):
        assert (x[pad] == 0).all(), f"{name} pads"
    assert torch.isneginf(lse[:, pad]).all()
    # the oracle through the same schedule
    g = Hq // Hkv
    if kv_group is None:
        hs, ks = list(range(Hq)), list(range(Hkv))
    else:
        hs, ks = list(range(kv_group * g, (kv_group + 1) * g)), [kv_group]
    sel = lambda x, idx: _f64(x[:, torch.tensor(idx, device=DEV)])  # noqa: E731
    o_r, lse_r, dq_r, dk_r, dv_r = OD.run_attention(
        sel(t["q"], hs), sel(t["k"], ks), sel(t["v"], ks), sel(t["do"], hs), p, chunk)
    hsel = torch.tensor(hs, device=DEV)
    ksel = torch.tensor(ks, device=DEV)
    assert_close("O", _f64(o[:, hsel]), o_r, real)
    assert_close("dQ", _f64(dq[:, hsel]), dq_r, real)
    assert_close("dK", _f64(dk[:, ksel]), dk_r, real)
    assert_close("dV", _f64(dv[:, ksel]), dv_r, real)
    assert np.abs(lse[hsel].cpu().numpy()[:, real] - lse_r[:, real]).max() <= LSE_ERR
    # against the packed path on the same inputs, every head
    po, plse, pdq, pdk, pdv = run_attention(bufs, t["q"], t["k"], t["v"], t["do"])
    assert torch.equal(o, po), "O differs from the packed forward"
    assert torch.equal(lse[:, torch.from_numpy(real).to(DEV)],
                       plse[:, torch.from_numpy(real).to(DEV)]), "LSE differs"
    for name, a, b in (("dQ", dq, pdq), ("dK", dk, pdk), ("dV", dv, pdv)):
        assert_close(name + " vs packed", _f64(a), _f64(b), np.ones(p.T_pad, bool))
    return len(ops)


@pytest.mark.parametrize("chunk", [1, 64, 2048])
def test_dta_tiny_workload(chunk):
    wl = W.WORKLOADS["tiny"]
    _, (p,) = pack_both(W.sequences("tiny"), wl.max_tokens_per_mb)
    check_dta(p, wl.Hq, wl.Hkv, wl.d, chunk, seed=chunk)


def test_dta_worked_example():
    _, (p,) = pack_both([[1, 2, 3, 4], [1, 2, 5, 6], [1, 7, 8]], 2048)
    for chunk in (1, 2, 2048):
        check_dta(p, 4, 2, 64, chunk, seed=3)


@pytest.mark.parametrize("Hq,Hkv,d,chunk", [(4, 2, 128, 64), (6, 3, 64, 200), (2, 1, 128, 2048)])
def test_dta_random_tries(Hq, Hkv, d, chunk):
    rng = W.SplitMix64(500 + chunk)
    base = [rng.randint(1, 2) for _ in range(600)]
    seqs = [base[:rng.randint(1, 600)] + [rng.randint(3, 6) for _ in range(rng.randint(1, 400))]
            for _ in range(7)]
    _, refs = pack_both(seqs, 4096)
    for p in refs:
        check_dta(p, Hq, Hkv, d, chunk, seed=chunk + 1)


def test_dta_full_size_agent_trie():
    # one 32K-token agent trie at the page's chunk of 2048 tokens; the oracle
    # runs the query heads of kv head 0
    wl = W.WORKLOADS["agent"]
    p = OT.pack_sequences(W.sequences("agent"), wl.max_tokens_per_mb)[0]
    mine = ptg.pack_sequences(W.sequences("agent"), wl.max_tokens_per_mb)[0]
    assert np.array_equal(mine.token_node, p.token_node)
    n_ops = check_dta(p, wl.Hq, wl.Hkv, wl.d, 2048, seed=11, kv_group=0)
    assert n_ops > 10
