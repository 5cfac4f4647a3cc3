"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Integer outputs (position ids, key reach, blockmap) must match bit for bit.
Float outputs (O, dQ, dK, dV over real tokens) are compared with the oracle,
which computes in float64 from the same bf16 inputs: mean |err| <= 2e-3, and
every element within ``max_bound``: 2e-2 on top of half a bf16
ulp of the reference value, because an output stored in bf16 cannot sit
closer to the exact value than that (at |x| >= 4 half an ulp is already
0.0156, at |x| >= 8 it is 0.031).  LSE within 5e-3.  Pads must give exactly
O = 0, LSE = -inf and zero gradients.
"""
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

MAX_ERR, MEAN_ERR, LSE_ERR = 2e-2, 2e-3, 5e-3
DEV = "cuda"


# ---------------------------------------------------------------- helpers
def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype).to(DEV)


def run_positions_blockmap(token_node, entry, exit_):
    T = len(token_node)
    N = len(entry)
    tn = _dev(token_node)
    en = _dev(entry) if N else torch.zeros(1, dtype=torch.int32, device=DEV)
    ex = _dev(exit_) if N else torch.zeros(1, dtype=torch.int32, device=DEV)
    bufs = ptg.TrieBuffers(T, N, 1, 64)
    ptg.tree_pack_positions(tn, en[:N], ex[:N], bufs.position_ids, bufs.key_reach, bufs.pos_ws,
                            bufs.status)
    ptg.tree_blockmap_build(bufs.key_reach, bufs.blockmap, bufs.status)
    torch.cuda.synchronize()
    return bufs


def expected_reach(packed):
    """Last row that sees key j (mask column maximum); pads j - 1."""
    M = OM.ancestor_mask(packed)
    T = packed.T_pad
    out = np.arange(T, dtype=np.int64) - 1
    for j in range(T):
        rows = np.nonzero(M[:, j])[0]
        if rows.size:
            out[j] = rows.max()
    return out


def expected_blockmap_fields(cls):
    nb = cls.shape[0]
    row_cnt = (cls != 0).sum(axis=1)
    row_nfull = (cls == 1).sum(axis=1)
    rows = []
    for qa in range(nb):
        rows += [kb for kb in range(nb) if cls[qa, kb] == 1]
        rows += [kb for kb in range(nb) if cls[qa, kb] == 2]
    col_len = (cls != 0).sum(axis=0)
    row_order = sorted(range(nb), key=lambda q: (-row_cnt[q], q))
    col_order = sorted(range(nb), key=lambda k: (-col_len[k], k))
    return dict(row_cnt=row_cnt, row_nfull=row_nfull, row_idx=np.array(rows, np.int64),
                row_order=np.array(row_order), col_order=np.array(col_order))


def check_integer_outputs(packed, bufs, full_reach=True):
    status = int(bufs.status.item())
    assert status == 0, ptg.status_string(status)
    pos = bufs.position_ids.cpu().numpy()
    assert np.array_equal(pos, OM.position_ids(packed))
    reach = bufs.key_reach.cpu().numpy()
    if full_reach:
        assert np.array_equal(reach, expected_reach(packed))
    view = ptg.blockmap_view(bufs.blockmap.cpu().numpy())
    cls = OM.tile_classes(packed)
    assert np.array_equal(ptg.tile_classes_from_blockmap(view), cls)
    want = expected_blockmap_fields(cls)
    for key in ("row_cnt", "row_nfull", "row_idx", "row_order", "col_order"):
        assert np.array_equal(np.asarray(view[key]), want[key]), key
    assert view["nnz"] == int((cls != 0).sum())
    return view


def run_attention(bufs, q, k, v, do):
    T, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=DEV)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((ptg.attn_bwd_workspace_bytes(T, Hq, d) + 3) // 4, dtype=torch.float32,
                     device=DEV)
    ptg.tree_attn_fwd(q, k, v, bufs.key_reach, bufs.blockmap, o, lse, bufs.status)
    ptg.tree_attn_bwd(q, k, v, o, do, lse, bufs.key_reach, bufs.blockmap, dq, dk, dv, ws,
                      bufs.status)
    torch.cuda.synchronize()
    status = int(bufs.status.item())
    assert status == 0, ptg.status_string(status)
    return o, lse, dq, dk, dv


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def half_ulp_bf16(x):
    """Half a bf16 ulp of |x| (bf16 keeps 8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def stored_o(o_ref):
    """The forward output as the backward receives it: rounded to bf16.

    The backward's D = rowsum(dO * O) term is a function of the O it is
    given, so the reference backward is evaluated at the oracle's own O
    rounded to bf16 (round to nearest even), not at the exact O.  With keys
    of large norm the two differ visibly: a row dominated by one key has
    dP - D close to zero, and the rounding of O moves D by up to ~0.2.
    """
    return torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy()


def max_bound(want):
    return MAX_ERR + half_ulp_bf16(want)


def assert_close(name, got, want, real):
    err = np.abs(got[real] - want[real])
    excess = err - max_bound(want[real])
    assert excess.max() <= 0, (f"{name}: max err {err.max():.3e} exceeds 2e-2 + half-ulp by "
                               f"{excess.max():.3e}")
    assert err.mean() <= MEAN_ERR, f"{name}: mean err {err.mean():.3e}"


def check_attention_dense(packed, Hq, Hkv, d, seed=0, tensors=None):
    T = packed.T_pad
    t = tensors if tensors is not None else W.tensors(T, Hq, Hkv, d, seed=seed, device=DEV)
    bufs = run_positions_blockmap(packed.token_node, packed.node_entry, packed.node_exit)
    o, lse, dq, dk, dv = run_attention(bufs, t["q"], t["k"], t["v"], t["do"])
    q, k, v, do = (_f64(t[n]) for n in ("q", "k", "v", "do"))
    M = OM.ancestor_mask(packed)
    scale = d ** -0.5
    o_ref, lse_ref = OA.forward(q, k, v, M, scale)
    dq_ref, dk_ref, dv_ref = OA.backward(q, k, v, stored_o(o_ref), do, M, scale)
    real = packed.token_node >= 0
    pad = ~real
    assert_close("O", _f64(o), o_ref, real)
    assert_close("dQ", _f64(dq), dq_ref, real)
    assert_close("dK", _f64(dk), dk_ref, real)
    assert_close("dV", _f64(dv), dv_ref, real)
    lse_np = lse.cpu().numpy()
    assert np.abs(lse_np[:, real] - lse_ref[:, real]).max() <= LSE_ERR
    assert np.isneginf(lse_np[:, pad]).all()
    for name, x in (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv)):
        assert (x[torch.from_numpy(pad).to(DEV)] == 0).all(), f"{name} pads not zero"
    return bufs


def pack_both(seqs, cap, **kw):
    mine = ptg.pack_sequences(seqs, cap, **kw)
    ref = OT.pack_sequences(seqs, cap, **kw)
    assert len(mine) == len(ref)
    for a, b in zip(mine, ref):
        assert np.array_equal(a.token_node, b.token_node)
        assert np.array_equal(a.node_exit, b.node_exit)
    return mine, ref


# ---------------------------------------------------------------- small cases
def test_wait_timeout_is_reported_not_hung():
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ptg.tree_debug_wait_timeout(st, 5_000_000)
    torch.cuda.synchronize()
    assert st.item() == 7
    # the context is still healthy
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum().item()) == 8.0


def test_worked_example_integer_outputs():
    seqs = [[1, 2, 3, 4], [1, 2, 5, 6], [1, 7, 8]]
    _, (p,) = pack_both(seqs, 2048)
    bufs = run_positions_blockmap(p.token_node, p.node_entry, p.node_exit)
    check_integer_outputs(p, bufs)
    reach = bufs.key_reach.cpu().numpy()
    assert reach[:8].tolist() == [7, 5, 3, 3, 5, 5, 7, 7]


def test_worked_example_attention_gqa():
    _, (p,) = pack_both([[1, 2, 3, 4], [1, 2, 5, 6], [1, 7, 8]], 2048)
    check_attention_dense(p, Hq=4, Hkv=2, d=64)


def test_all_pad_trie():
    T = 256
    bufs = run_positions_blockmap(np.full(T, -1, np.int32), np.zeros(0, np.int32),
                                  np.zeros(0, np.int32))
    assert bufs.status.item() == 0
    assert (bufs.position_ids.cpu() == 0).all()
    assert np.array_equal(bufs.key_reach.cpu().numpy(), np.arange(T) - 1)
    view = ptg.blockmap_view(bufs.blockmap.cpu().numpy())
    assert view["nnz"] == 0
    t = W.tensors(T, 2, 1, 128, seed=3, device=DEV)
    o, lse, dq, dk, dv = run_attention(bufs, t["q"], t["k"], t["v"], t["do"])
    for x in (o, dq, dk, dv):
        assert (x == 0).all()
    assert torch.isneginf(lse).all()


def test_single_token():
    _, (p,) = pack_both([[5]], 128)
    check_attention_dense(p, Hq=2, Hkv=2, d=128)


def test_tiny_workload_integer_and_attention():
    seqs = W.sequences("tiny")
    _, (p,) = pack_both(seqs, 2048)
    wl = W.WORKLOADS["tiny"]
    bufs = check_attention_dense(p, wl.Hq, wl.Hkv, wl.d, seed=0)
    check_integer_outputs(p, bufs)


def test_tiny_workload_padded_to_max():
    seqs = W.sequences("tiny")
    _, (p,) = pack_both(seqs, 2048, pad_to_max=True)
    assert p.T_pad == 2048
    bufs = check_attention_dense(p, 4, 4, 64, seed=1)
    check_integer_outputs(p, bufs)


def _random_case(seed, n_seqs, prefix, tail):
    rng = W.SplitMix64(seed)
    base = [rng.randint(1, 2) for _ in range(prefix)]
    seqs = []
    for _ in range(n_seqs):
        cut = rng.randint(1, prefix)
        seqs.append(base[:cut] + [rng.randint(3, 6) for _ in range(rng.randint(1, tail))])
    return seqs


@pytest.mark.parametrize("Hq,Hkv,d,seed", [(8, 2, 128, 11), (4, 2, 128, 12), (2, 2, 128, 13),
                                          (6, 3, 64, 14), (4, 1, 64, 15)])
def test_random_tries_dense(Hq, Hkv, d, seed):
    seqs = _random_case(seed, n_seqs=7, prefix=700, tail=300)
    _, refs = pack_both(seqs, 4096)
    for p in refs:
        bufs = check_attention_dense(p, Hq, Hkv, d, seed=seed)
        check_integer_outputs(p, bufs)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 128), (2, 2, 64)])
def test_key_block_with_many_reach_values(Hq, Hkv, d):
    # A chain of twenty 5-token nodes, each also the parent of a 200-token
    # leaf: the first key block holds twenty distinct reach values, more
    # than 4 in every 32-key group, so the forward's visibility bits of its
    # PARTIAL tiles take the key-by-key fallback instead of the run list.
    seqs = [list(range(1, 5 * k + 1)) + [1000 * k + t for t in range(200)] for k in range(1, 21)]
    _, (p,) = pack_both(seqs, 8192)
    reach = expected_reach(p)
    groups = [len(set(reach[g * 32:g * 32 + 32].tolist())) for g in range(3)]
    assert min(groups) > 4
    bufs = check_attention_dense(p, Hq, Hkv, d, seed=6)
    check_integer_outputs(p, bufs)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 1, 128), (2, 2, 64)])
def test_top_level_boundaries_inside_blocks(Hq, Hkv, d):
    # Several top-level subtrees whose boundaries fall inside 128-token
    # blocks: rows just past a boundary see nothing in the first listed
    # tiles of their block and meet their first visible key later on.
    rng = W.SplitMix64(77)
    seqs = []
    for s in range(6):
        L = rng.randint(150, 700)
        seqs.append([1000 * (s + 1) + t for t in range(L)])
    seqs.append(seqs[1][:200] + [99000 + t for t in range(rng.randint(50, 300))])
    _, refs = pack_both(seqs, 8192)
    for p in refs:
        starts = [p.node_start[n] for n in range(p.n_nodes) if p.node_parent[n] < 0]
        assert any(s_ % 128 for s_ in starts[1:])
        bufs = check_attention_dense(p, Hq, Hkv, d, seed=9)
        check_integer_outputs(p, bufs)


def test_full_tiles_long_prefix():
    rng = W.SplitMix64(21)
    prefix = [rng.randint(1, 50) for _ in range(900)]
    seqs = [prefix + [100 + i] * rng.randint(100, 700) for i in range(4)]
    _, (p,) = pack_both(seqs, 4096)
    assert (OM.tile_classes(p) == 1).sum() > 10
    bufs = check_attention_dense(p, 4, 2, 128, seed=2)
    check_integer_outputs(p, bufs)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 128), (2, 1, 64)])
def test_score_jumps_force_rescale(Hq, Hkv, d):
    # Every query shares the all-ones direction and a few keys point along
    # it, so rows that see those keys have their running max jump by about
    # 17, 24, 33, 140 and 33 log2 units at later tiles: in the first and in
    # the second 64-column half of a tile, in FULL and PARTIAL tiles, and once
    # by so much that the earlier terms underflow to zero.  This drives the
    # forward's O and P rescale paths, which random scores never reach.
    rng = W.SplitMix64(21)
    prefix = [rng.randint(1, 50) for _ in range(900)]
    seqs = [prefix + [100 + i] * rng.randint(100, 700) for i in range(4)]
    _, (p,) = pack_both(seqs, 4096)
    T = p.T_pad
    t = W.tensors(T, Hq, Hkv, d, seed=3, device=DEV)
    g = (128 / d) ** 0.5
    k = t["k"].clone()
    for j, beta in ((200, 1.5), (300, 2.5), (650, 3.5), (870, 12.0), (1000, 14.0)):
        k[j] = beta * g
    t = dict(t, q=(t["q"].float() + 1.0).to(torch.bfloat16), k=k)
    bufs = run_positions_blockmap(p.token_node, p.node_entry, p.node_exit)
    check_integer_outputs(p, bufs)
    o, lse, _, _, _ = run_attention(bufs, t["q"], t["k"], t["v"], t["do"])
    q, k, v, do = (_f64(t[n]) for n in ("q", "k", "v", "do"))
    M = OM.ancestor_mask(p)
    scale = d ** -0.5
    o_ref, lse_ref = OA.forward(q, k, v, M, scale)
    real = p.token_node >= 0
    assert_close("O", _f64(o), o_ref, real)
    assert np.abs(lse.cpu().numpy()[:, real] - lse_ref[:, real]).max() <= LSE_ERR
    # The backward on its own, at the oracle's O (rounded to bf16, as the
    # forward stores it) and LSE: with keys this large, D = rowsum(dO * O)
    # is sensitive to the last bit of O.
    o_in = torch.from_numpy(stored_o(o_ref)).to(torch.bfloat16).to(DEV)
    lse_in = torch.from_numpy(lse_ref).float().to(DEV)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    ws = torch.empty((ptg.attn_bwd_workspace_bytes(T, Hq, d) + 3) // 4, dtype=torch.float32,
                     device=DEV)
    ptg.tree_attn_bwd(t["q"], t["k"], t["v"], o_in, t["do"], lse_in, bufs.key_reach,
                      bufs.blockmap, dq, dk, dv, ws, bufs.status)
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == 0
    o_st = stored_o(o_ref)
    dq_ref, dk_ref, dv_ref = OA.backward(q, k, v, o_st, do, M, scale)
    assert_close("dV", _f64(dv), dv_ref, real)
    # dQ and dK take dS rounded to bf16 (relative error <= 2^-9) times keys
    # and queries of norm up to 14*sqrt(d): allow one bf16 ulp of dS on
    # every term of their sums on top of the usual bound.
    bq, bk = np.zeros_like(dq_ref), np.zeros_like(dk_ref)
    g_ = Hq // Hkv
    for h in range(Hq):
        hk = h // g_
        S = np.where(M, q[:, h] @ k[:, hk].T * scale, -np.inf)
        P = np.exp(S - np.where(np.isfinite(lse_ref[h]), lse_ref[h], 0.0)[:, None])
        dS = np.abs(P * (do[:, h] @ v[:, hk].T - (do[:, h] * o_st[:, h]).sum(1)[:, None]))
        bq[:, h] = 2.0 ** -8 * scale * dS @ np.abs(k[:, hk])
        bk[:, hk] += 2.0 ** -8 * scale * dS.T @ np.abs(q[:, h])
    for name, got, want, extra in (("dQ", dq, dq_ref, bq), ("dK", dk, dk_ref, bk)):
        err = np.abs(_f64(got)[real] - want[real])
        excess = err - max_bound(want[real]) - extra[real]
        assert excess.max() <= 0, f"{name}: max err {err.max():.3e}, excess {excess.max():.3e}"
        assert err.mean() <= MEAN_ERR, f"{name}: mean err {err.mean():.3e}"


def test_forest_of_two_tries_in_one_buffer():
    a = _random_case(31, 4, 300, 200)
    b = [[s_ + 1000 for s_ in seq] for seq in _random_case(32, 4, 300, 200)]
    _, (pa,) = pack_both(a, 4096)
    _, (pb,) = pack_both(b, 4096)
    # concatenate: pb's nodes re-ranked after pa's
    Na, Nb = pa.n_nodes, pb.n_nodes
    tn = np.concatenate([pa.token_node, np.where(pb.token_node >= 0, pb.token_node + Na, -1)])
    entry = np.concatenate([pa.node_entry, pb.node_entry + Na]).astype(np.int32)
    exit_ = np.concatenate([pa.node_exit, pb.node_exit + Na]).astype(np.int32)
    forest = OT.PackedTrie(seq_ids=[], n_tokens=pa.n_tokens + pb.n_tokens,
                           T_pad=pa.T_pad + pb.T_pad, token_node=tn.astype(np.int32),
                           token_ids=np.concatenate([pa.token_ids, pb.token_ids]),
                           node_entry=entry, node_exit=exit_,
                           node_parent=np.concatenate([pa.node_parent, np.where(
                               pb.node_parent >= 0, pb.node_parent + Na, -1)]).astype(np.int32),
                           node_start=np.concatenate([pa.node_start, pb.node_start + pa.T_pad]),
                           node_end=np.concatenate([pa.node_end, pb.node_end + pa.T_pad]))
    bufs = check_attention_dense(forest, 4, 2, 128, seed=5)
    check_integer_outputs(forest, bufs)


MALFORMED = 4


def _status_of(token_node, entry, exit_):
    bufs = run_positions_blockmap(np.asarray(token_node, np.int32), np.asarray(entry, np.int32),
                                  np.asarray(exit_, np.int32))
    return int(bufs.status.item())


def test_malformed_inputs_flagged():
    good_tn = [0, 1, 2, 2, 3, 3, 4, 4] + [-1] * 120
    good_en, good_ex = [0, 1, 2, 3, 4], [4, 3, 2, 3, 4]
    assert _status_of(good_tn, good_en, good_ex) == 0
    split = [0, 1, 2, 3, 2, 3, 4, 4] + [-1] * 120                 # node 2 split in two runs
    assert _status_of(split, good_en, good_ex) == MALFORMED
    assert _status_of([0, 1, 2, 2, 3, 3, 4, 9] + [-1] * 120, good_en, good_ex) == MALFORMED
    assert _status_of(good_tn, [0, 1, 2, 3, 3], good_ex) == MALFORMED   # duplicate rank
    assert _status_of(good_tn, good_en, [4, 3, 2, 4, 4]) == MALFORMED   # crossing subtrees
    assert _status_of(good_tn, good_en, [4, 3, 1, 3, 4]) == MALFORMED   # exit < entry
    pad_inside = [0, 1, -1, 2, 2, 3, 3, 4, 4] + [-1] * 119          # pad inside the span of 0
    assert _status_of(pad_inside, good_en, good_ex) == MALFORMED
    order = [0, 1, 3, 3, 2, 2, 4, 4] + [-1] * 120                 # ranks out of order
    assert _status_of(order, good_en, good_ex) == MALFORMED
    empty = [0, 1, 2, 2, 4, 4, 4, 4] + [-1] * 120                 # node 3 has no token
    assert _status_of(empty, good_en, good_ex) == MALFORMED


# ---------------------------------------------------------------- full sizes
def _sampled_rows(packed, n, rng):
    real = np.nonzero(packed.token_node >= 0)[0]
    pick = [int(real[0]), int(real[-1])] + [int(real[rng.randint(0, len(real) - 1)])
                                            for _ in range(n)]
    return sorted(set(pick))


def check_full_size(key, trie_indices, n_rows=6, n_keys=3):
    wl = W.WORKLOADS[key]
    seqs = W.sequences(key)
    mine = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)
    ref = OT.pack_sequences(seqs, wl.max_tokens_per_mb)
    rng = W.SplitMix64(7 + wl.index)
    for ti in trie_indices:
        a, p = mine[ti], ref[ti]
        assert np.array_equal(a.token_node, p.token_node)
        bufs = run_positions_blockmap(p.token_node, p.node_entry, p.node_exit)
        check_integer_outputs(p, bufs, full_reach=False)
        t = W.tensors(p.T_pad, wl.Hq, wl.Hkv, wl.d, seed=ti, device=DEV)
        o, lse, dq, dk, dv = run_attention(bufs, t["q"], t["k"], t["v"], t["do"])
        q, k, v, do = (_f64(t[n]) for n in ("q", "k", "v", "do"))
        rows = _sampled_rows(p, n_rows, rng)
        heads = range(wl.Hq)
        ro, rl, rdq, _, _ = OA.rows_forward_backward(q, k, v, do, p, rows, heads,
                                                      key_grads=False)
        o_np, dq_np, lse_np = _f64(o), _f64(dq), lse.cpu().numpy()
        errs_o, errs_dq = [], []
        for i in rows:
            for h in heads:
                errs_o.append(np.abs(o_np[i, h] - ro[(i, h)]) - max_bound(ro[(i, h)]))
                errs_dq.append(np.abs(dq_np[i, h] - rdq[(i, h)]) - max_bound(rdq[(i, h)]))
                assert abs(lse_np[h, i] - rl[(i, h)]) <= LSE_ERR
        for name, e in (("O", np.concatenate(errs_o)), ("dQ", np.concatenate(errs_dq))):
            assert e.max() <= 0, (name, e.max())
        # dK/dV of keys in the deepest nodes (few rows see them)
        leaf_nodes = [n for n in range(p.n_nodes) if p.node_exit[n] == n]
        leaf_nodes.sort(key=lambda n: p.node_end[n] - p.node_start[n])
        # a key near the end of a short leaf: only the last few rows see it
        keys = [int(p.node_end[n] - min(7, p.node_end[n] - p.node_start[n]))
                for n in leaf_nodes[:n_keys]]
        kdk, kdv = OA.key_grads(q, k, v, do, p, keys, range(wl.Hkv))
        dk_np, dv_np = _f64(dk), _f64(dv)
        for j in keys:
            for kv in range(wl.Hkv):
                assert (np.abs(dk_np[j, kv] - kdk[(j, kv)]) <= max_bound(kdk[(j, kv)])).all()
                assert (np.abs(dv_np[j, kv] - kdv[(j, kv)]) <= max_bound(kdv[(j, kv)])).all()
        # properties at full size: sum_j dV[j,kv] = sum over heads/real rows of dO;
        # sum_j dK[j,kv] = 0 (rows of dS sum to zero)
        real = torch.from_numpy(p.token_node >= 0).to(DEV)
        g = wl.Hq // wl.Hkv
        want_dv = t["do"].float()[real].view(-1, wl.Hkv, g, wl.d).sum(dim=(0, 2))
        got_dv = dv.float().sum(dim=0)
        scale_ref = t["do"].float()[real].abs().sum(dim=0).view(wl.Hkv, g, wl.d).sum(1)
        assert ((got_dv - want_dv).abs() <= 1e-2 * scale_ref + 1.0).all()
        assert (dk.float().sum(dim=0).abs() <= 1e-2 * dk.float().abs().sum(dim=0) + 1.0).all()
        assert not torch.isnan(dq).any() and not torch.isnan(dk).any()


def test_full_fanout():
    check_full_size("fanout", [0])


def test_full_grpo_sampled_tries():
    check_full_size("grpo", [25])


def test_full_agent_sampled_tries():
    check_full_size("agent", [0])


def test_full_long_sampled_tries():
    check_full_size("long", [0])
