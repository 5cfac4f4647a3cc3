"""The bounds-checked TREE_DEBUG build on the GPU.

The debug library (``libtreeattn_debug.so``, built by ``build()`` beside the
release library) runs in a child process (``PREFIX_TREE_ATTN_DEBUG=1``;
see tests/debug_build_cases.py).  On a clean trie its positions, blockmap,
O, LSE, dQ, dK and dV must equal the release library's bit for bit (the
checks sit outside the arithmetic).  With one index word of the blockmap or
key_reach corrupted, it must report TREE_ERR_BOUNDS through the status word
and leave the context usable: the clean trie run again afterwards gives the
same results.  The corrupted cases never run on the release build, which
trusts those buffers.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import prefix_tree_attention_gb300 as ptg  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
TREE_ERR_BOUNDS = 9


def test_debug_build_matches_release_and_reports_bad_indices(tmp_path):
    dbg_lib = os.path.join(os.path.dirname(ptg.LIB_PATH), "libtreeattn_debug.so")
    assert os.path.exists(dbg_lib), "build() builds the debug library"
    assert not ptg.debug_build()
    prefix = str(tmp_path / "debug_case")
    env = dict(os.environ, PREFIX_TREE_ATTN_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py"), prefix],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    with open(prefix + ".json") as f:
        rec = json.load(f)
    assert rec["clean_rerun_identical"]
    for name, st in rec["statuses"].items():
        assert st == TREE_ERR_BOUNDS, (name, ptg.status_string(st))
    import debug_build_cases as C
    case = C.Case(ptg, C._trie())
    release = C.run_clean(case)
    debug = np.load(prefix + ".npz")
    for k, v in release.items():
        assert np.array_equal(v, debug[k]), k
