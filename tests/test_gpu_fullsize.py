"""GPU parity at full size: every real row and every real key of key/value
heads 0 and 7 (with their query heads), element by element, on one trie of
each Qwen3-8B-head workload (grpo, agent, long, fanout).

The reference is the oracle's dense masked attention (``oracle/attention.py``
``forward`` / ``backward``) evaluated on blocks of query rows: a block of
rows R reads its rows of the parent-walk mask (``oracle/mask.py``
``mask_rows``), keeps the key columns C that any row of R sees, and calls
the oracle on (Q[R], K[C], V[C], mask[R, C]).  This is the oracle's own
definition restricted to those rows — a row's softmax involves only its own
row of the mask, and every masked-out column contributes exactly zero — so
O, LSE and dQ of R are complete, and dK/dV of C receive exactly the terms
of the rows of R; summing those partials over all blocks gives the full
dK/dV (the gradient of a shared-prefix key over every continuation, AREAL-DTA
section 3).  The backward is evaluated at the oracle's O rounded to bf16, the
value the forward stores (see test_gpu_parity.stored_o).

Bounds, as in the dense tests: every element within 2e-2 plus half a bf16 ulp
of the reference value, and the mean error over all compared elements of each
output within 2e-3.  Key reach (the last row that sees each key) and position
ids are compared bit for bit, reach from the same mask blocks.

Each test prints, per output, the largest error, its margin to the literal
2e-2 bound (negative = inside it) and the mean error; with PARITY_REPORT set
to a file path the same figures are appended there as JSON lines.
"""
import json
import os
import time

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import mask as OM
from oracle import trie as OT

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefix_tree_attention_gb300 as ptg  # noqa: E402

from test_gpu_parity import (LSE_ERR, MAX_ERR, MEAN_ERR, check_integer_outputs,  # noqa: E402
                             half_ulp_bf16, run_attention, run_positions_blockmap, stored_o)

ROW_BLOCK = 256
KV_HEADS = (0, 7)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _reference_block(p, q, k, v, do, nh, g, scale, r0, r1):
    """The oracle on query rows r0..r1-1 against the key columns they see."""
    M = OM.mask_rows(p, r0, r1)
    cols = np.nonzero(M.any(axis=0))[0]
    if cols.size == 0:
        return None
    last = r1 - 1 - np.argmax(M[::-1][:, cols], axis=0)   # last row seeing each column
    Mc = M[:, cols]
    out = []
    for a in range(nh):
        hs = slice(a * g, (a + 1) * g)
        qa, doa = q[r0:r1, hs], do[r0:r1, hs]
        ka, va = k[cols, a:a + 1], v[cols, a:a + 1]
        o_b, lse_b = OA.forward(qa, ka, va, Mc, scale)
        dq_b, dk_b, dv_b = OA.backward(qa, ka, va, stored_o(o_b), doa, Mc, scale)
        out.append((o_b, lse_b, dq_b, dk_b[:, 0], dv_b[:, 0]))
    return cols, last, out


def blockwise_reference(p, q, k, v, do, kv_heads, g, scale):
    """Oracle O, LSE, dQ (query heads of ``kv_heads``) and dK, dV, plus the
    key reach, from row blocks of the parent-walk mask.  q/do hold only those
    query heads (in kv-head order), k/v only those kv heads.  Blocks run on
    host threads (numpy releases the GIL in its array loops); their dK/dV
    partials are summed afterwards in block order."""
    from concurrent.futures import ThreadPoolExecutor
    T = p.T_pad
    nh = len(kv_heads)
    o = np.zeros((T, nh * g, q.shape[2]))
    lse = np.full((nh * g, T), -np.inf)
    dq = np.zeros_like(o)
    dk = np.zeros((T, nh, q.shape[2]))
    dv = np.zeros_like(dk)
    reach = np.arange(T, dtype=np.int64) - 1
    starts = list(range(0, T, ROW_BLOCK))
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(
            lambda r0: _reference_block(p, q, k, v, do, nh, g, scale, r0,
                                        min(T, r0 + ROW_BLOCK)), starts))
    for r0, res in zip(starts, results):
        if res is None:
            continue
        r1 = min(T, r0 + ROW_BLOCK)
        cols, last, out = res
        reach[cols] = np.maximum(reach[cols], last)
        for a, (o_b, lse_b, dq_b, dk_b, dv_b) in enumerate(out):
            hs = slice(a * g, (a + 1) * g)
            o[r0:r1, hs] = o_b
            lse[hs, r0:r1] = lse_b
            dq[r0:r1, hs] = dq_b
            dk[cols, a] += dk_b
            dv[cols, a] += dv_b
    return o, lse, dq, dk, dv, reach


def _report(record):
    path = os.environ.get("PARITY_REPORT")
    print(json.dumps(record))
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")


def compare(name, got, want, real, rec):
    err = np.abs(got[real] - want[real])
    excess = err - (MAX_ERR + half_ulp_bf16(want[real]))
    rec[name] = {"max_err": float(err.max()), "max_minus_2e-2": float(err.max() - MAX_ERR),
                 "max_excess_over_bound": float(excess.max()), "mean_err": float(err.mean()),
                 "elements": int(err.size)}
    return excess.max() <= 0 and err.mean() <= MEAN_ERR


def check_full_trie(key, trie_index, kv_heads=KV_HEADS):
    wl = W.WORKLOADS[key]
    seqs = W.sequences(key)
    mine = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)
    ref = OT.pack_sequences(seqs, wl.max_tokens_per_mb)
    a, p = mine[trie_index], ref[trie_index]
    assert np.array_equal(a.token_node, p.token_node)
    assert np.array_equal(a.node_exit, p.node_exit)
    bufs = run_positions_blockmap(p.token_node, p.node_entry, p.node_exit)
    check_integer_outputs(p, bufs, full_reach=False)
    t = W.tensors(p.T_pad, wl.Hq, wl.Hkv, wl.d, seed=100 + trie_index, device="cuda")
    o, lse, dq, dk, dv = run_attention(bufs, t["q"], t["k"], t["v"], t["do"])
    g = wl.Hq // wl.Hkv
    heads = [h for kv in kv_heads for h in range(kv * g, (kv + 1) * g)]
    hidx = torch.tensor(heads, device="cuda")
    kidx = torch.tensor(list(kv_heads), device="cuda")
    q, do = _f64(t["q"][:, hidx]), _f64(t["do"][:, hidx])
    k, v = _f64(t["k"][:, kidx]), _f64(t["v"][:, kidx])
    t0 = time.perf_counter()
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref, reach_ref = blockwise_reference(
        p, q, k, v, do, kv_heads, g, wl.d ** -0.5)
    host_s = time.perf_counter() - t0
    assert np.array_equal(bufs.key_reach.cpu().numpy(), reach_ref), "key reach"
    real = p.token_node >= 0
    rec = {"workload": key, "trie": trie_index, "T_pad": p.T_pad,
           "real_tokens": int(real.sum()), "kv_heads": list(kv_heads),
           "query_heads": heads, "oracle_host_s": round(host_s, 1)}
    ok = {}
    ok["O"] = compare("O", _f64(o[:, hidx]), o_ref, real, rec)
    ok["dQ"] = compare("dQ", _f64(dq[:, hidx]), dq_ref, real, rec)
    ok["dK"] = compare("dK", _f64(dk[:, kidx]), dk_ref, real, rec)
    ok["dV"] = compare("dV", _f64(dv[:, kidx]), dv_ref, real, rec)
    lse_err = np.abs(lse.cpu().numpy()[heads][:, real] - lse_ref[:, real])
    rec["LSE"] = {"max_err": float(lse_err.max()), "bound": LSE_ERR}
    ok["LSE"] = lse_err.max() <= LSE_ERR
    pad = torch.from_numpy(~real).to("cuda")
    for name, x in (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)):
        ok[name + " pads"] = bool((x[pad] == 0).all())
    _report(rec)
    bad = [n for n, v_ in ok.items() if not v_]
    assert not bad, f"{key} trie {trie_index}: {bad} out of bounds: {rec}"


def test_fullsize_elementwise_fanout():
    # one 16384-token prefix seen by all 512 leaves: its keys' dK/dV sum the
    # rows of every leaf
    check_full_trie("fanout", 0)


def test_fullsize_elementwise_grpo():
    check_full_trie("grpo", 0)


def test_fullsize_elementwise_agent():
    check_full_trie("agent", 0)


def test_fullsize_elementwise_long():
    check_full_trie("long", 0)
