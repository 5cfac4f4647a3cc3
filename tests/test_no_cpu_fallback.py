"""The product path has no CPU fallback: every device entry point of the
binding refuses host tensors loudly instead of computing anything (CPU only;
no kernel is launched)."""
import pytest
import torch

import prefix_tree_attention_gb300 as ptg


def _i32(n):
    return torch.zeros(n, dtype=torch.int32)


def test_device_entry_points_refuse_host_tensors():
    T = 128
    f32 = torch.zeros(T, dtype=torch.float32)
    bf = torch.zeros((T, 2, 64), dtype=torch.bfloat16)
    calls = [
        lambda: ptg.tree_pack_positions(_i32(T), _i32(1), _i32(1), _i32(T), _i32(T), _i32(64),
                                        _i32(1)),
        lambda: ptg.tree_pack_positions_noalloc(_i32(T), _i32(1), _i32(1), _i32(T), _i32(T),
                                                _i32(1)),
        lambda: ptg.tree_blockmap_build(_i32(T), _i32(4096), _i32(1)),
        lambda: ptg.tree_attn_fwd(bf, bf, bf, _i32(T), _i32(4096), bf.clone(),
                                  torch.zeros((2, T)), _i32(1)),
        lambda: ptg.tree_attn_bwd(bf, bf, bf, bf, bf, torch.zeros((2, T)), _i32(T), _i32(4096),
                                  bf.clone(), bf.clone(), bf.clone(), torch.zeros(16), _i32(1)),
        lambda: ptg.tree_logprobs_entropy(torch.zeros((T, 64), dtype=torch.bfloat16), _i32(T),
                                          f32, _i32(1)),
        lambda: ptg.tree_merge_per_sequence(f32, _i32(4), torch.zeros(3, dtype=torch.int64),
                                            torch.zeros((2, 4)), _i32(1), 1, 1),
    ]
    calls += [
        lambda: ptg.tree_attn_bwd_prepare(bf, bf, torch.zeros((2, T)), torch.zeros(16), _i32(1)),
        lambda: ptg.tree_attn_bwd_main(bf, bf, bf, bf, _i32(T), _i32(4096), bf.clone(),
                                       bf.clone(), torch.zeros(16), _i32(1)),
        lambda: ptg.tree_attn_bwd_finish(torch.zeros(16), bf.clone(), _i32(1)),
        lambda: ptg.tree_debug_wait_timeout(_i32(1), 1_000_000),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


class _FakeDev:
    def __init__(self, kind):
        self.type = kind


class _Fake:
    """Only what the device check reads."""

    def __init__(self, kind):
        self.device = _FakeDev(kind)


def test_device_check_accepts_device_tensors_and_names_the_host_one():
    ptg._on_device(a=_Fake("cuda"), b=None, c=_Fake("cuda"))
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        ptg._on_device(q=_Fake("cuda"), workspace=_Fake("cpu"))
