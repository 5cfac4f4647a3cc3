"""C-ABI checks that need no GPU: the library loads and exports every symbol
declared in include/tree_attn.h, host-side argument errors come back
synchronously, and the host packer matches the oracle's packer bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W
from oracle import mask as OM
from oracle import trie as OT

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tree_attn.h")

ptg = pytest.importorskip("prefix_tree_attention_gb300")
lib = ctypes.CDLL(ptg.LIB_PATH)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    return sorted({n for n in names if n.startswith("tree_") and n not in ("tree_status_t",)})


def test_every_declared_symbol_is_exported():
    names = _declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert set(ptg.EXPORTED_SYMBOLS) == set(names)



def test_debug_build_exports_the_same_symbols():
    dbg = os.path.join(os.path.dirname(ptg.LIB_PATH), "libtreeattn_debug.so")
    if not os.path.exists(dbg):
        pytest.skip("the TREE_DEBUG library is not built")
    d = ctypes.CDLL(dbg)
    for n in _declared_functions():
        assert hasattr(d, n), f"{n} declared but not exported by the debug build"
    d.tree_debug_build.restype = ctypes.c_int32
    lib.tree_debug_build.restype = ctypes.c_int32
    assert d.tree_debug_build() == 1 and lib.tree_debug_build() == 0
    d.tree_status_string.restype = ctypes.c_char_p
    assert d.tree_status_string(9) == b"TREE_ERR_BOUNDS"

def test_status_strings_and_version():
    assert ptg.status_string(0) == "TREE_OK"
    assert ptg.status_string(4) == "TREE_ERR_MALFORMED_TREE"
    assert ptg.status_string(7) == "TREE_ERR_TIMEOUT"
    assert ptg.status_string(9) == "TREE_ERR_BOUNDS"
    assert ptg.status_string(99) == "TREE_ERR_UNKNOWN"
    assert re.fullmatch(r"\d+\.\d+\.\d+", ptg.version())


def test_workspace_sizes():
    assert ptg.blockmap_bytes(128) == 4 * (5 + 7 + 1)
    nb = 512
    assert ptg.blockmap_bytes(nb * 128) == 4 * (5 + 7 * nb + nb * (nb + 1) // 2)
    assert ptg.attn_bwd_workspace_bytes(1024, 32, 128) == 1024 * 32 * (128 + 2) * 4
    assert ptg.pack_positions_workspace_bytes(4096, 100) > 4 * (4096 + 6 * 100)


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced


def test_host_side_errors_return_before_launch():
    f = lib.tree_attn_fwd
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    f.argtypes = [P, P, P, P, P, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_float, P, P, P, P]
    args = lambda T, Hq, Hkv, d, q=FAKE, bm_bytes=1 << 20: (
        q, FAKE, FAKE, FAKE, FAKE, bm_bytes, T, Hq, Hkv, d, 0.1, FAKE, FAKE, FAKE, None)
    assert f(*args(256, 4, 4, 64, bm_bytes=16)) == 8   # blockmap buffer too small
    assert f(*args(200, 4, 4, 64)) == 2          # T_pad not a multiple of 128
    assert f(*args(256, 4, 3, 64)) == 1          # Hq % Hkv
    assert f(*args(256, 4, 4, 96)) == 5          # head_dim unsupported
    assert f(*args(256, 4, 4, 64, q=None)) == 1  # null pointer
    assert f(*args(256, 4, 4, 64, q=FAKE + 4)) == 2  # unaligned pointer
    assert f(*args(0, 4, 4, 64)) == 0            # empty input is a no-op
    for bad in (0.0, -0.1, float("nan"), float("inf")):   # scale not positive and finite
        a = list(args(256, 4, 4, 64))
        a[10] = bad
        assert f(*a) == 1, bad
    b = lib.tree_blockmap_build
    b.restype = ctypes.c_int
    b.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_size_t, P, P]
    assert b(FAKE, 256, 64, FAKE, 1 << 20, FAKE, None) == 5      # block != 128
    assert b(FAKE, 250, 128, FAKE, 1 << 20, FAKE, None) == 2
    assert b(FAKE, 256, 128, FAKE, 8, FAKE, None) == 8           # buffer too small
    pp = lib.tree_pack_positions
    pp.restype = ctypes.c_int
    pp.argtypes = [P, ctypes.c_int32, P, P, ctypes.c_int32, P, P, P, ctypes.c_size_t, P, P]
    assert pp(FAKE, 256, FAKE, FAKE, 4, FAKE, FAKE, FAKE, 16, FAKE, None) == 8
    assert pp(FAKE, 256, FAKE, FAKE, 300, FAKE, FAKE, FAKE, 1 << 20, FAKE, None) == 1
    assert pp(FAKE, 100, FAKE, FAKE, 4, FAKE, FAKE, FAKE, 1 << 20, FAKE, None) == 2
    bw = lib.tree_attn_bwd
    bw.restype = ctypes.c_int
    bw.argtypes = [P] * 8 + [ctypes.c_size_t] + [ctypes.c_int32] * 4 + [ctypes.c_float] + \
        [P] * 4 + [ctypes.c_size_t, P, P]
    MB = 1 << 20
    assert bw(*([FAKE] * 8), MB, 256, 8, 2, 128, 0.1, FAKE, FAKE, FAKE, FAKE, 64, FAKE,
              None) == 8                                     # workspace too small
    assert bw(*([FAKE] * 8), 16, 256, 8, 2, 128, 0.1, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE,
              None) == 8                                     # blockmap too small
    assert bw(*([FAKE] * 8), MB, 256, 8, 2, 128, -1.0, FAKE, FAKE, FAKE, FAKE, 1 << 30, FAKE,
              None) == 1



def test_dta_attn_checks_arguments_before_launch():
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    f = lib.tree_dta_attn
    f.restype = ctypes.c_int
    f.argtypes = [P] * 6 + [SZ, I32, I32, I32, I32, ctypes.c_float, P, I64] + [P] * 6 + \
        [SZ, P, P]
    T, Hq, Hkv, d = 256, 4, 2, 64
    ws = ptg.dta_attn_workspace_bytes(T, Hq, Hkv, d)
    assert ws == ptg.attn_bwd_workspace_bytes(T, Hq, d) + 2 * T * Hkv * d * 4

    def call(ops, n=None, T=T, ws_bytes=ws, bm_bytes=1 << 20, d=d):
        arr = np.ascontiguousarray(np.asarray(ops, np.int32).reshape(-1, 3))
        return f(*([FAKE] * 6), bm_bytes, T, Hq, Hkv, d, 0.125,
                 arr.ctypes.data if arr.size else None, arr.shape[0] if n is None else n,
                 *([FAKE] * 6), ws_bytes, FAKE, None)
    assert call([[3, 0, 8]]) == 1                # unknown op kind
    assert call([[0, 8, 8]]) == 1                # empty row range
    assert call([[1, 0, T + 1]]) == 1            # past T_pad
    assert call([[2, -1, 4]]) == 1               # negative start
    assert call([[0, 0, 8]], n=-1) == 1          # negative count
    assert call([[0, 0, 8]], ws_bytes=ws - 16) == 8
    assert call([[0, 0, 8]], bm_bytes=16) == 8
    assert call([[0, 0, 8]], T=200) == 2
    assert call([[0, 0, 8]], d=96) == 5
    assert call([], T=0) == 0                    # empty input is a no-op


def test_logprob_entry_points_check_arguments_before_launch():
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    f = lib.tree_logprobs_entropy
    f.restype = ctypes.c_int
    f.argtypes = [P, I32, I64, I32, I32, P, P, P, SZ, P, P, P, P, P, P, P, P]

    def call(dtype=0, stride=1000, T=256, V=1000, tok=FAKE, bm=FAKE, bm_bytes=1 << 20,
             lse=FAKE, logprob=FAKE, pred=None, logits=FAKE):
        return f(logits, dtype, stride, T, V, tok, FAKE, bm, bm_bytes, lse, None, None, None,
                 logprob, pred, FAKE, None)
    assert call(dtype=2) == 5                    # dtype other than bf16 / fp32
    assert call(V=0) == 1 and call(stride=999) == 1
    assert call(T=200) == 2                      # T_pad not a multiple of 128
    assert call(logits=None) == 1 and call(lse=None) == 1
    assert call(bm=None) == 1                    # labels need the blockmap
    assert call(tok=None) == 1                   # logprob needs token ids
    assert call(bm_bytes=16) == 8                # blockmap buffer too small
    assert call(T=0) == 0 and call(T=0, logits=None) == 0   # empty input is a no-op
    m = lib.tree_merge_per_sequence
    m.restype = ctypes.c_int
    m.argtypes = [P, I64, P, I64, P, I32, I32, I32, I32, ctypes.c_float, P, P, P]
    assert m(FAKE, 10, FAKE, 10, FAKE, 2, 8, 1, 0, 0.0, FAKE, FAKE, None) == 1   # trim < shift
    assert m(FAKE, 10, FAKE, 10, FAKE, 2, 8, -1, 0, 0.0, FAKE, FAKE, None) == 1
    assert m(FAKE, -1, FAKE, 10, FAKE, 2, 8, 1, 1, 0.0, FAKE, FAKE, None) == 1
    assert m(None, 10, FAKE, 10, FAKE, 2, 8, 1, 1, 0.0, FAKE, FAKE, None) == 1
    assert m(FAKE, 10, FAKE, 10, FAKE, 0, 8, 1, 1, 0.0, FAKE, FAKE, None) == 0   # no-op



def test_logprob_gradient_entry_points_check_arguments_before_launch():
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f = lib.tree_logprobs_entropy_bwd
    f.restype = ctypes.c_int
    f.argtypes = [P, I32, I64, I32, I32, P, P, P, P, P, P, P, I64, P, P]

    def call(dtype=0, stride=1000, T=256, V=1000, tok=FAKE, ent=FAKE, g_lp=FAKE, g_ent=FAKE,
             out=FAKE, out_stride=1000, lse=FAKE, logits=FAKE):
        return f(logits, dtype, stride, T, V, tok, FAKE, lse, ent, g_lp, g_ent, out, out_stride,
                 FAKE, None)
    assert call(dtype=2) == 5
    assert call(V=0) == 1 and call(stride=999) == 1 and call(out_stride=999) == 1
    assert call(T=200) == 2
    assert call(logits=None) == 1 and call(lse=None) == 1 and call(out=None) == 1
    assert call(tok=None) == 1                   # logprob gradient needs token ids
    assert call(ent=None) == 1                   # entropy gradient needs the entropy
    assert call(T=0) == 0 and call(T=0, logits=None) == 0   # empty input is a no-op
    m = lib.tree_merge_per_sequence_bwd
    m.restype = ctypes.c_int
    m.argtypes = [P, P, I64, P, I32, I32, I32, I32, P, I64, P, P]
    assert m(FAKE, FAKE, 10, FAKE, 2, 8, 1, 0, FAKE, 10, FAKE, None) == 1   # trim < shift
    assert m(FAKE, FAKE, 10, FAKE, 2, 8, -1, 0, FAKE, 10, FAKE, None) == 1
    assert m(FAKE, FAKE, 10, FAKE, 2, 8, 1, 1, FAKE, -1, FAKE, None) == 1
    assert m(None, FAKE, 10, FAKE, 2, 8, 1, 1, FAKE, 10, FAKE, None) == 1
    assert m(FAKE, FAKE, 10, FAKE, 2, 8, 1, 1, None, 10, FAKE, None) == 1
    assert m(FAKE, FAKE, 10, FAKE, 0, 8, 1, 1, FAKE, 10, FAKE, None) == 0   # no-op

def test_sequence_index_arrays_layout():
    tries = ptg.pack_sequences([[1, 2, 3], [1, 2, 4, 5], [7]], 128)
    pos, offs = ptg.sequence_index_arrays(tries, 3)
    assert offs.tolist() == [0, 3, 7, 8]
    for sid, L in enumerate((3, 4, 1)):
        t = next(t for t in tries if sid in t.seq_index)
        base = sum(u.T_pad for u in tries[:tries.index(t)])
        assert pos[offs[sid]:offs[sid + 1]].tolist() == (t.seq_index[sid] + base).tolist()
        assert offs[sid + 1] - offs[sid] == L


def _same_packing(mine, ref):
    assert len(mine) == len(ref)
    for a, b in zip(mine, ref):
        assert (a.n_tokens, a.T_pad, a.n_nodes) == (b.n_tokens, b.T_pad, b.n_nodes)
        assert np.array_equal(a.token_node, b.token_node)
        assert np.array_equal(a.token_ids, b.token_ids)
        assert np.array_equal(a.node_entry, b.node_entry)
        assert np.array_equal(a.node_exit, b.node_exit)
        assert a.seq_ids == b.seq_ids
        for sid in b.seq_ids:
            assert np.array_equal(a.seq_index[sid], b.seq_index[sid])


def test_packer_worked_example_and_pairs():
    seqs = [[1, 2, 3, 4], [1, 2, 5, 6], [1, 7, 8]]
    mine = ptg.pack_sequences(seqs, 2048)
    ref = OT.pack_sequences(seqs, 2048)
    _same_packing(mine, ref)
    assert mine[0].visible_pairs == 22 == OM.visible_pairs(ref[0])


def test_packer_errors():
    with pytest.raises(ptg.TreeError) as e:
        ptg.pack_sequences([[1, 2]], 0)
    assert e.value.status == 1
    with pytest.raises(ptg.TreeError) as e:
        ptg.pack_sequences([[1, 2]], 100)
    assert e.value.status == 2
    with pytest.raises(ptg.TreeError) as e:
        ptg.pack_sequences([list(range(1, 200))], 128)
    assert e.value.status == 3
    with pytest.raises(ptg.TreeError) as e:
        ptg.pack_sequences([[1], []], 128)
    assert e.value.status == 1


def test_packer_random_small_sets():
    rng = W.SplitMix64(4242)
    for trial in range(300):
        seqs = W.random_sequences(rng, rng.randint(1, 8), 40, rng.randint(1, 3))
        cap = 128 * rng.randint(1, 3)
        mine = ptg.pack_sequences(seqs, cap)
        ref = OT.pack_sequences(seqs, cap)
        _same_packing(mine, ref)
        for a, b in zip(mine, ref):
            assert a.visible_pairs == OM.visible_pairs(b)


def test_packer_wide_nodes():
    # A root and a shared prefix with 20 distinct continuations each, with
    # repeats, so that children are looked up before and after a node gets
    # more than a handful of them (the packer then also indexes them by hash).
    rng = W.SplitMix64(99)
    seqs = []
    for rep in range(3):
        for c in range(20):
            seqs.append([7, 7, 7, 100 + c] + [rng.randint(1, 3) for _ in range(rng.randint(1, 6))])
            seqs.append([500 + c] + [rng.randint(1, 3) for _ in range(rng.randint(1, 6))])
    for cap in (128, 1024):
        mine = ptg.pack_sequences(seqs, cap)
        ref = OT.pack_sequences(seqs, cap)
        _same_packing(mine, ref)
        for a, b in zip(mine, ref):
            assert a.visible_pairs == OM.visible_pairs(b)


def test_packer_pad_to_max():
    seqs = W.sequences("tiny")
    mine = ptg.pack_sequences(seqs, 2048, pad_to_max=True)
    ref = OT.pack_sequences(seqs, 2048, pad_to_max=True)
    _same_packing(mine, ref)
    assert mine[0].T_pad == 2048


@pytest.mark.parametrize("key", ["tiny", "fanout", "long", "agent", "grpo"])
def test_packer_matches_oracle_on_workloads(key):
    seqs = W.sequences(key)
    wl = W.WORKLOADS[key]
    mine = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)
    ref = OT.pack_sequences(seqs, wl.max_tokens_per_mb)
    _same_packing(mine, ref)
    # pairs against the closed form "position = token depth" summed per node
    for a, b in zip(mine, ref):
        depth_base = np.zeros(b.n_nodes, np.int64)
        for r in range(b.n_nodes):
            par = b.node_parent[r]
            if par >= 0:
                depth_base[r] = depth_base[par] + (b.node_end[par] - b.node_start[par] + 1)
        L = (b.node_end - b.node_start + 1).astype(np.int64)
        pairs = int((L * depth_base + L * (L + 1) // 2).sum())
        assert a.visible_pairs == pairs
