"""Cases for the bounds-checked TREE_DEBUG build of the library.

Run as a script with ``PREFIX_TREE_ATTN_DEBUG=1`` (the package then loads
``libtreeattn_debug.so``): it refuses to run unless the loaded library
reports itself as the debug build, runs a clean trie through positions,
blockmap, forward and backward, then the same trie with one index word of
its blockmap or key_reach corrupted per case, then the clean trie again, and
writes the clean outputs (``.npz``) and every case's status (``.json``).

Each corrupted word is one the debug build validates before its first use
(see tree_debug_build in include/tree_attn.h): a row of the row order past
the last query block, a key block past its row in a row's list, a row
offset past the CSR array, a column of the column order below 0, and a
key_reach value past the last token.  The blockmap build itself reads
key_reach only at in-range token indices, so a corrupted value there stays
a wrong value, which the debug build reports.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HQ, HKV, D = 8, 2, 128


def _trie():
    import workloads as W
    from oracle import trie as OT
    rng = W.SplitMix64(2718)
    seqs = W.random_sequences(rng, 10, 300, 3)
    (packed,) = OT.pack_sequences(seqs, 4096)
    return packed


class Case:
    """Device buffers of one trie, its inputs and outputs."""

    def __init__(self, ptg, packed):
        import torch
        import workloads as W
        self.ptg, self.packed = ptg, packed
        dev = "cuda"
        T = packed.T_pad
        self.T, self.nb = T, T // 128
        self.bufs = ptg.TrieBuffers(T, packed.n_nodes, HQ, D, device=dev)
        self.tn = torch.from_numpy(packed.token_node).to(dev)
        self.en = torch.from_numpy(packed.node_entry).to(dev)
        self.ex = torch.from_numpy(packed.node_exit).to(dev)
        self.t = W.tensors(T, HQ, HKV, D, seed=5, device=dev)
        self.o = torch.empty_like(self.t["q"])
        self.lse = torch.empty((HQ, T), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.t["q"])
        self.dk = torch.empty_like(self.t["k"])
        self.dv = torch.empty_like(self.t["v"])

    def positions_blockmap(self):
        b = self.bufs
        b.status.zero_()
        self.ptg.tree_pack_positions(self.tn, self.en, self.ex, b.position_ids, b.key_reach,
                                     b.pos_ws, b.status)
        self.ptg.tree_blockmap_build(b.key_reach, b.blockmap, b.status)

    def forward(self):
        b, t = self.bufs, self.t
        self.ptg.tree_attn_fwd(t["q"], t["k"], t["v"], b.key_reach, b.blockmap, self.o, self.lse,
                               b.status)

    def backward(self):
        b, t = self.bufs, self.t
        self.ptg.tree_attn_bwd(t["q"], t["k"], t["v"], self.o, t["do"], self.lse, b.key_reach,
                               b.blockmap, self.dq, self.dk, self.dv, b.bwd_ws, b.status)

    def status(self) -> int:
        import torch
        torch.cuda.synchronize()
        return int(self.bufs.status.item())

    def outputs(self) -> dict:
        b = self.bufs
        f = lambda x: x.view(torch_int16()).cpu().numpy()  # noqa: E731  (bf16 bits)
        bm = b.blockmap.cpu().numpy()
        # the words the build defines: the header and the row lists it filled
        # (the tail of the worst-case row-list area stays as allocated)
        used = _row_idx(self.nb) + int(bm[_row_ptr(self.nb) + self.nb])
        return {"position_ids": b.position_ids.cpu().numpy(),
                "key_reach": b.key_reach.cpu().numpy(), "blockmap": bm[:used],
                "o": f(self.o), "lse": self.lse.cpu().numpy(), "dq": f(self.dq),
                "dk": f(self.dk), "dv": f(self.dv)}


def torch_int16():
    import torch
    return torch.int16


def run_clean(case: Case) -> dict:
    case.positions_blockmap()
    case.forward()
    case.backward()
    st = case.status()
    assert st == 0, case.ptg.status_string(st)
    return case.outputs()


# blockmap word offsets (tree_blockmap_build's layout)
def _row_cnt(nb):
    return 4 + 2 * nb


def _row_ptr(nb):
    return 4 + 4 * nb


def _row_order(nb):
    return 5 + 5 * nb


def _col_order(nb):
    return 5 + 6 * nb


def _row_idx(nb):
    return 5 + 7 * nb


def run_corrupted(case: Case) -> dict:
    """Status of each corrupted case (fresh positions and blockmap each time)."""
    nb = case.nb
    out = {}

    def fresh():
        case.positions_blockmap()
        assert case.status() == 0
        return case.bufs.blockmap

    bm = fresh()
    bm[_row_order(nb)] = nb + 5                      # a query block past the last
    case.forward()
    out["row_order_past_end"] = case.status()

    bm = fresh()
    qa = int(bm[_row_order(nb)].item())              # the heaviest row: >= 1 tile
    assert int(bm[_row_cnt(nb) + qa].item()) >= 1
    off = int(bm[_row_ptr(nb) + qa].item())
    bm[_row_idx(nb) + off] = nb + 3                  # a key block past the row
    case.forward()
    out["row_list_key_block_past_row"] = case.status()

    bm = fresh()
    bm[_row_ptr(nb) + qa] = 100_000_000              # a row offset past the CSR array
    case.forward()
    out["row_offset_past_array"] = case.status()

    bm = fresh()
    bm[_col_order(nb)] = -1                          # a key block below 0
    case.backward()
    out["col_order_negative"] = case.status()

    case.bufs.status.zero_()
    b = case.bufs
    case.ptg.tree_pack_positions(case.tn, case.en, case.ex, b.position_ids, b.key_reach,
                                 b.pos_ws, b.status)
    assert case.status() == 0
    b.key_reach[5] = case.T + 100                    # a reach past the last token
    case.ptg.tree_blockmap_build(b.key_reach, b.blockmap, b.status)
    out["key_reach_past_end"] = case.status()
    case.forward()                                   # everything after the error skips
    case.backward()
    out["after_error_status"] = case.status()
    return out


def main(out_prefix: str) -> int:
    import prefix_tree_attention_gb300 as ptg
    if not ptg.debug_build():
        print("refusing: the loaded library is not the TREE_DEBUG build", file=sys.stderr)
        return 3
    case = Case(ptg, _trie())
    first = run_clean(case)
    statuses = run_corrupted(case)
    again = run_clean(case)
    np.savez(out_prefix + ".npz", **first)
    same = all(np.array_equal(first[k], again[k]) for k in first)
    with open(out_prefix + ".json", "w") as f:
        json.dump({"statuses": statuses, "clean_rerun_identical": same}, f)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
