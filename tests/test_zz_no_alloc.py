"""GPU test of tree_pack_positions_noalloc, the entry point for callers that
cannot allocate device memory (for example an operator inside a framework
that owns all device allocations and hands over only input and output
buffers).  It must give exactly what tree_pack_positions gives with a caller
workspace — position ids and key reach are integers, so bit for bit — on two
calls in a row, the second on a different trie so that anything left over in
the shared scratch array from the first call would show.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process (the first call does the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefix_tree_attention_gb300 as ptg  # noqa: E402


def _call_noalloc(tn, en, ex, pos, reach, status):
    # straight through the C ABI symbol
    rc = ptg._lib.tree_pack_positions_noalloc(
        ctypes.c_void_p(tn.data_ptr()), tn.numel(), ctypes.c_void_p(en.data_ptr()),
        ctypes.c_void_p(ex.data_ptr()), en.numel(), ctypes.c_void_p(pos.data_ptr()),
        ctypes.c_void_p(reach.data_ptr()), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def _case(tr):
    dev = "cuda"
    tn = torch.from_numpy(tr.token_node).to(dev)
    en = torch.from_numpy(tr.node_entry).to(dev)
    ex = torch.from_numpy(tr.node_exit).to(dev)
    return tn, en, ex


def _with_workspace(tn, en, ex):
    bufs = ptg.TrieBuffers(tn.numel(), en.numel(), 1, 64)
    ptg.tree_pack_positions(tn, en, ex, bufs.position_ids, bufs.key_reach, bufs.pos_ws,
                            bufs.status)
    torch.cuda.synchronize()
    assert bufs.status.item() == 0
    return bufs.position_ids.cpu().numpy(), bufs.key_reach.cpu().numpy()


def test_noalloc_matches_workspace_version_twice_in_a_row():
    fan = ptg.pack_sequences(W.sequences("fanout"), W.WORKLOADS["fanout"].max_tokens_per_mb)[0]
    tiny = ptg.pack_sequences(W.sequences("tiny"), W.WORKLOADS["tiny"].max_tokens_per_mb)[0]
    for tr in (fan, tiny):        # large first, then small: stale scratch would show
        tn, en, ex = _case(tr)
        want_pos, want_reach = _with_workspace(tn, en, ex)
        pos = torch.full_like(tn, -7)
        reach = torch.full_like(tn, -7)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _call_noalloc(tn, en, ex, pos, reach, status) == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        assert np.array_equal(pos.cpu().numpy(), want_pos)
        assert np.array_equal(reach.cpu().numpy(), want_reach)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    tn = torch.full((65536 + 128,), -1, dtype=torch.int32, device="cuda")
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    pos = torch.empty_like(tn)
    reach = torch.empty_like(tn)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(tn, empty, empty, pos, reach, status) == 8   # TREE_ERR_WORKSPACE
