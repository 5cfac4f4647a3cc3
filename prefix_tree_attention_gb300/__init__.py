"""Python binding of ``libtreeattn`` — packed prefix-trie attention for GB300.

Argument marshalling only: every step of the hot path runs in the library's
sm_103a kernels (``include/tree_attn.h``).  PyTorch provides device memory
and streams.  There is no fallback: if the compiled library is missing the
import fails loudly; build it with ``python prefix_tree_attention_gb300/build.py``.

Entry points mirror the C ABI names: ``tree_pack_positions``,
``tree_blockmap_build``, ``tree_attn_fwd``, ``tree_attn_bwd`` (each takes
tensors, checks their dtype/shape/device, passes raw pointers and the current
CUDA stream, and raises ``TreeError`` on a non-OK status), the log-probability
gather ``tree_logprobs_entropy`` with its merge ``tree_merge_per_sequence``
and their gradients ``tree_logprobs_entropy_bwd`` / ``tree_merge_per_sequence_bwd``,
the LM head fused with the gather ``tree_lm_head_logprobs_entropy`` and its
chunked logits gradient ``tree_lm_head_logits_grad``,
plus the host packer ``pack_sequences``, partitioner ``partition_sequences``
and the DFS traversal schedule ``dta_schedule``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# PREFIX_TREE_ATTN_DEBUG=1 selects the bounds-checked TREE_DEBUG build of the
# same sources (``build.py --debug``); the entry points are the same.
_DEBUG = os.environ.get("PREFIX_TREE_ATTN_DEBUG", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "lib", "libtreeattn_debug.so" if _DEBUG else "libtreeattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python prefix_tree_attention_gb300/build.py"
        + (" --debug`" if _DEBUG else "`"))

_lib = ctypes.CDLL(LIB_PATH)

_P, _I32, _I64, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
_sig = {
    "tree_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tree_version": (ctypes.c_char_p, []),
    "tree_debug_build": (_I32, []),
    "tree_pack_positions_workspace_bytes": (_SZ, [_I32, _I32]),
    "tree_pack_positions": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _P, _P, _P, _SZ, _P, _P]),
    "tree_blockmap_bytes": (_SZ, [_I32]),
    "tree_blockmap_build": (ctypes.c_int, [_P, _I32, _I32, _P, _SZ, _P, _P]),
    "tree_attn_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _SZ, _I32, _I32, _I32, _I32, _F32, _P,
                                     _P, _P, _P]),
    "tree_attn_bwd_workspace_bytes": (_SZ, [_I32, _I32, _I32]),
    "tree_attn_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I32, _I32, _I32,
                                     _I32, _F32, _P, _P, _P, _P, _SZ, _P, _P]),
    "tree_packing_build": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _I32, _P]),
    "tree_packing_free": (None, [_P]),
    "tree_packing_num_tries": (_I32, [_P]),
    "tree_packing_trie_info": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P]),
    "tree_packing_trie_arrays": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P]),
    "tree_packing_seq_indices": (ctypes.c_int, [_P, _I32, _I32, _P, _I32]),
    "tree_debug_wait_timeout": (ctypes.c_int, [_P, _I64, _P]),
    "tree_attn_bwd_prepare": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, _P, _SZ, _P, _P]),
    "tree_attn_bwd_main": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _SZ, _I32, _I32, _I32, _I32,
                                          _F32, _P, _P, _P, _SZ, _P, _P]),
    "tree_attn_bwd_finish": (ctypes.c_int, [_I32, _I32, _I32, _F32, _P, _SZ, _P, _P, _P]),
    "tree_launch_count": (ctypes.c_uint64, []),
    "tree_pack_positions_noalloc": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _P, _P, _P, _P]),
    "tree_partition_sequences": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _P, _P]),
    "tree_logprobs_entropy": (ctypes.c_int, [_P, _I32, _I64, _I32, _I32, _P, _P, _P, _SZ, _P,
                                             _P, _P, _P, _P, _P, _P, _P]),
    "tree_merge_per_sequence": (ctypes.c_int, [_P, _I64, _P, _I64, _P, _I32, _I32, _I32, _I32,
                                               _F32, _P, _P, _P]),
    "tree_merge_per_sequence_bwd": (ctypes.c_int, [_P, _P, _I64, _P, _I32, _I32, _I32, _I32, _P,
                                                   _I64, _P, _P]),
    "tree_logprobs_entropy_bwd": (ctypes.c_int, [_P, _I32, _I64, _I32, _I32, _P, _P, _P, _P, _P,
                                                 _P, _P, _I64, _P, _P]),
    "tree_lm_head_workspace_bytes": (_SZ, [_I32, _I32]),
    "tree_lm_head_logprobs_entropy": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P, _SZ,
                                                     _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tree_lm_head_grad_workspace_bytes": (_SZ, [_I32]),
    "tree_lm_head_logits_grad": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P,
                                                _P, _P, _P, _P, _P, _I64, _P, _SZ, _P, _P]),
    "tree_dta_schedule": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _I32, _P, _I64, _P, _P]),
    "tree_dta_attn_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32]),
    "tree_dta_attn": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _SZ, _I32, _I32, _I32, _I32, _F32,
                                     _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
}
for _name, (_res, _args) in _sig.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED_SYMBOLS = tuple(_sig)

TREE_OK = 0
BLOCK = 128


class TreeError(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} ({status})")


def status_string(status: int) -> str:
    return _lib.tree_status_string(int(status)).decode()


def version() -> str:
    return _lib.tree_version().decode()


def debug_build() -> bool:
    """True when the loaded library is the bounds-checked TREE_DEBUG build."""
    return bool(_lib.tree_debug_build())


def _check(fn: str, status: int) -> None:
    if status != TREE_OK:
        raise TreeError(fn, status)


def _stream_ptr(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _need(t, dtype, name):
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    del torch


def _on_device(**tensors):
    """Every tensor handed to a device entry point must live on a CUDA device:
    a host pointer reaching a kernel would fault, and there is no CPU path."""
    for name, t in tensors.items():
        if t is not None and t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")


def _check_reach_blockmap(key_reach, blockmap, T):
    """key_reach must hold T_pad int32 values; the blockmap buffer's size is
    passed to the library, which refuses one that is too small."""
    import torch
    _need(key_reach, torch.int32, "key_reach")
    if key_reach.numel() != T:
        raise ValueError(f"key_reach must hold T_pad = {T} values, got {key_reach.numel()}")
    if not blockmap.is_contiguous():
        raise ValueError("blockmap must be contiguous")


# --------------------------------------------------------------- workspaces
def pack_positions_workspace_bytes(T_pad: int, n_nodes: int) -> int:
    return int(_lib.tree_pack_positions_workspace_bytes(T_pad, n_nodes))


def blockmap_bytes(T_pad: int) -> int:
    return int(_lib.tree_blockmap_bytes(T_pad))


def attn_bwd_workspace_bytes(T_pad: int, Hq: int, d: int) -> int:
    return int(_lib.tree_attn_bwd_workspace_bytes(T_pad, Hq, d))


# --------------------------------------------------------------- hot path
def tree_pack_positions(token_node, node_entry, node_exit, position_ids, key_reach, workspace,
                        dev_status, stream=None):
    import torch
    _on_device(token_node=token_node, node_entry=node_entry, node_exit=node_exit,
               position_ids=position_ids, key_reach=key_reach, workspace=workspace,
               dev_status=dev_status)
    _need(token_node, torch.int32, "token_node")
    for t, n in ((position_ids, "position_ids"), (key_reach, "key_reach")):
        _need(t, torch.int32, n)
    T_pad = token_node.numel()
    N = node_entry.numel()
    _check("tree_pack_positions", _lib.tree_pack_positions(
        _ptr(token_node), T_pad, _ptr(node_entry) if N else 0, _ptr(node_exit) if N else 0, N,
        _ptr(position_ids), _ptr(key_reach), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream_ptr(stream)))


def tree_pack_positions_noalloc(token_node, node_entry, node_exit, position_ids, key_reach,
                                dev_status, stream=None):
    """tree_pack_positions with the library's fixed device scratch array
    (no workspace argument; T_pad and n_nodes up to 65536)."""
    import torch
    _on_device(token_node=token_node, node_entry=node_entry, node_exit=node_exit,
               position_ids=position_ids, key_reach=key_reach, dev_status=dev_status)
    _need(token_node, torch.int32, "token_node")
    for t, n in ((position_ids, "position_ids"), (key_reach, "key_reach")):
        _need(t, torch.int32, n)
    N = node_entry.numel()
    _check("tree_pack_positions_noalloc", _lib.tree_pack_positions_noalloc(
        _ptr(token_node), token_node.numel(), _ptr(node_entry) if N else 0,
        _ptr(node_exit) if N else 0, N, _ptr(position_ids), _ptr(key_reach), _ptr(dev_status),
        _stream_ptr(stream)))


def tree_blockmap_build(key_reach, blockmap, dev_status, stream=None, block: int = BLOCK):
    import torch
    _on_device(key_reach=key_reach, blockmap=blockmap, dev_status=dev_status)
    _need(key_reach, torch.int32, "key_reach")
    _check("tree_blockmap_build", _lib.tree_blockmap_build(
        _ptr(key_reach), key_reach.numel(), block, _ptr(blockmap),
        blockmap.numel() * blockmap.element_size(), _ptr(dev_status), _stream_ptr(stream)))


def tree_attn_fwd(q, k, v, key_reach, blockmap, o, lse, dev_status, scale=None, stream=None):
    import torch
    _on_device(q=q, k=k, v=v, key_reach=key_reach, blockmap=blockmap, o=o, lse=lse,
               dev_status=dev_status)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    if k.shape != (T, Hkv, d) or v.shape != k.shape or o.shape != q.shape or lse.shape != (Hq, T):
        raise ValueError("shape mismatch")
    _check_reach_blockmap(key_reach, blockmap, T)
    scale = d ** -0.5 if scale is None else float(scale)
    _check("tree_attn_fwd", _lib.tree_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(key_reach), _ptr(blockmap), _nbytes(blockmap), T, Hq,
        Hkv, d, scale, _ptr(o), _ptr(lse), _ptr(dev_status), _stream_ptr(stream)))


def tree_attn_bwd(q, k, v, o, d_o, lse, key_reach, blockmap, dq, dk, dv, workspace, dev_status,
                  scale=None, stream=None):
    import torch
    _on_device(q=q, k=k, v=v, o=o, d_o=d_o, lse=lse, key_reach=key_reach, blockmap=blockmap,
               dq=dq, dk=dk, dv=dv, workspace=workspace, dev_status=dev_status)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (d_o, "d_o"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _need(t, torch.bfloat16, n)
    if dk.shape != k.shape or dv.shape != v.shape or dq.shape != q.shape or d_o.shape != q.shape:
        raise ValueError("shape mismatch")
    if o.shape != q.shape or lse.shape != (Hq, T):
        raise ValueError("shape mismatch")
    _need(lse, torch.float32, "lse")
    _check_reach_blockmap(key_reach, blockmap, T)
    scale = d ** -0.5 if scale is None else float(scale)
    _check("tree_attn_bwd", _lib.tree_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o), _ptr(lse), _ptr(key_reach),
        _ptr(blockmap), _nbytes(blockmap), T, Hq, Hkv, d, scale, _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), _nbytes(workspace), _ptr(dev_status), _stream_ptr(stream)))


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


DTYPE_BF16, DTYPE_F32 = 0, 1


def tree_logprobs_entropy(logits, key_reach, lse, dev_status, token_ids=None, blockmap=None,
                          entropy=None, vocab_min=None, vocab_max=None, logprob=None,
                          token_pred=None, stream=None):
    """Per-row log-sum-exp (and optionally entropy, vocab min/max) of packed
    logits ``[T_pad, V]`` (bf16 or fp32, unit stride along V), and per token
    the log-probability of its id under its predicting row and that row."""
    import torch
    _on_device(logits=logits, key_reach=key_reach, lse=lse, dev_status=dev_status,
               token_ids=token_ids, blockmap=blockmap, entropy=entropy, vocab_min=vocab_min,
               vocab_max=vocab_max, logprob=logprob, token_pred=token_pred)
    if logits.dim() != 2 or logits.stride(1) != 1 or logits.device.type != "cuda":
        raise ValueError("logits must be a 2-D CUDA tensor with unit stride along the vocabulary")
    code = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}.get(logits.dtype)
    if code is None:
        raise TypeError(f"logits must be bf16 or float32, got {logits.dtype}")
    T_pad, V = logits.shape
    _need(key_reach, torch.int32, "key_reach")
    if key_reach.numel() != T_pad:
        raise ValueError(f"key_reach must hold T_pad = {T_pad} values")
    if blockmap is not None:
        _need(blockmap, torch.int32, "blockmap")
    for t, n in ((lse, "lse"), (entropy, "entropy"), (vocab_min, "vocab_min"),
                 (vocab_max, "vocab_max"), (logprob, "logprob")):
        if t is not None:
            _need(t, torch.float32, n)
            if t.numel() != T_pad:
                raise ValueError(f"{n} must hold T_pad = {T_pad} values")
    for t, n in ((token_ids, "token_ids"), (token_pred, "token_pred")):
        if t is not None:
            _need(t, torch.int32, n)
            if t.numel() != T_pad:
                raise ValueError(f"{n} must hold T_pad = {T_pad} values")
    _check("tree_logprobs_entropy", _lib.tree_logprobs_entropy(
        _ptr(logits), code, logits.stride(0), T_pad, V, _ptr(token_ids), _ptr(key_reach),
        _ptr(blockmap), 0 if blockmap is None else _nbytes(blockmap), _ptr(lse), _ptr(entropy),
        _ptr(vocab_min), _ptr(vocab_max), _ptr(logprob), _ptr(token_pred), _ptr(dev_status),
        _stream_ptr(stream)))


def tree_merge_per_sequence(src, seq_pos, seq_offsets, out, dev_status, shift: int, trim: int,
                            padding_value: float = 0.0, stream=None):
    """``out[s, t] = src[seq_pos[seq_offsets[s] + t + shift]]`` for
    ``t < len(s) - trim``, else ``padding_value``; ``out`` is [n_seqs, max_len]."""
    import torch
    _on_device(src=src, seq_pos=seq_pos, seq_offsets=seq_offsets, out=out, dev_status=dev_status)
    _need(src, torch.float32, "src")
    _need(seq_pos, torch.int32, "seq_pos")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(out, torch.float32, "out")
    n_seqs, max_len = out.shape
    if seq_offsets.numel() != n_seqs + 1:
        raise ValueError("seq_offsets must hold n_seqs + 1 values")
    _check("tree_merge_per_sequence", _lib.tree_merge_per_sequence(
        _ptr(src), src.numel(), _ptr(seq_pos), seq_pos.numel(), _ptr(seq_offsets), n_seqs,
        max_len, int(shift), int(trim), float(padding_value), _ptr(out), _ptr(dev_status),
        _stream_ptr(stream)))


def tree_merge_per_sequence_bwd(out_grad, seq_pos, seq_offsets, src_grad, dev_status,
                                shift: int, trim: int, stream=None):
    """Adjoint of ``tree_merge_per_sequence`` with the same ``seq_pos``,
    ``seq_offsets``, ``shift`` and ``trim``: ``src_grad[seq_pos[seq_offsets[s]
    + t + shift]] += out_grad[s, t]``.  Accumulates: zero ``src_grad`` first."""
    import torch
    _on_device(out_grad=out_grad, seq_pos=seq_pos, seq_offsets=seq_offsets, src_grad=src_grad,
               dev_status=dev_status)
    _need(out_grad, torch.float32, "out_grad")
    _need(seq_pos, torch.int32, "seq_pos")
    _need(seq_offsets, torch.int64, "seq_offsets")
    _need(src_grad, torch.float32, "src_grad")
    if out_grad.dim() != 2:
        raise ValueError("out_grad must be [n_seqs, max_len]")
    n_seqs, max_len = out_grad.shape
    if seq_offsets.numel() != n_seqs + 1:
        raise ValueError("seq_offsets must hold n_seqs + 1 values")
    _check("tree_merge_per_sequence_bwd", _lib.tree_merge_per_sequence_bwd(
        _ptr(out_grad), _ptr(seq_pos), seq_pos.numel(), _ptr(seq_offsets), n_seqs, max_len,
        int(shift), int(trim), _ptr(src_grad), src_grad.numel(), _ptr(dev_status),
        _stream_ptr(stream)))


def tree_logprobs_entropy_bwd(logits, key_reach, lse, grad_logits, dev_status, token_ids=None,
                              entropy=None, grad_logprob=None, grad_entropy=None, stream=None):
    """Gradient of the log-probability / entropy gather with respect to the
    packed logits: ``grad_logits`` (same dtype and shape as ``logits``) from
    the per-token ``grad_logprob`` and per-row ``grad_entropy`` (either may
    be None), using the ``lse`` and ``entropy`` of the forward call."""
    import torch
    _on_device(logits=logits, key_reach=key_reach, lse=lse, grad_logits=grad_logits,
               dev_status=dev_status, token_ids=token_ids, entropy=entropy,
               grad_logprob=grad_logprob, grad_entropy=grad_entropy)
    for t, n in ((logits, "logits"), (grad_logits, "grad_logits")):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{n} must be 2-D with unit stride along the vocabulary")
    code = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}.get(logits.dtype)
    if code is None:
        raise TypeError(f"logits must be bf16 or float32, got {logits.dtype}")
    if grad_logits.dtype != logits.dtype or grad_logits.shape != logits.shape:
        raise ValueError("grad_logits must match the logits' dtype and shape")
    T_pad, V = logits.shape
    _need(key_reach, torch.int32, "key_reach")
    for t, n in ((key_reach, "key_reach"), (lse, "lse"), (entropy, "entropy"),
                 (grad_logprob, "grad_logprob"), (grad_entropy, "grad_entropy"),
                 (token_ids, "token_ids")):
        if t is not None:
            _need(t, torch.int32 if n in ("key_reach", "token_ids") else torch.float32, n)
            if t.numel() != T_pad:
                raise ValueError(f"{n} must hold T_pad = {T_pad} values")
    _check("tree_logprobs_entropy_bwd", _lib.tree_logprobs_entropy_bwd(
        _ptr(logits), code, logits.stride(0), T_pad, V, _ptr(token_ids), _ptr(key_reach),
        _ptr(lse), _ptr(entropy), _ptr(grad_logprob), _ptr(grad_entropy), _ptr(grad_logits),
        grad_logits.stride(0), _ptr(dev_status), _stream_ptr(stream)))


def lm_head_workspace_bytes(T_pad: int, V: int) -> int:
    return int(_lib.tree_lm_head_workspace_bytes(int(T_pad), int(V)))


def tree_lm_head_logprobs_entropy(hidden, weight, key_reach, lse, workspace, dev_status,
                                  token_ids=None, blockmap=None, entropy=None, vocab_min=None,
                                  vocab_max=None, logprob=None, token_pred=None, stream=None):
    """The LM head (``hidden [T_pad, H] @ weight [V, H]^T``, bf16) fused with
    the gather: the outputs of ``tree_logprobs_entropy`` without the logits
    ever being written."""
    import torch
    _on_device(hidden=hidden, weight=weight, key_reach=key_reach, lse=lse, workspace=workspace,
               dev_status=dev_status, token_ids=token_ids, blockmap=blockmap, entropy=entropy,
               vocab_min=vocab_min, vocab_max=vocab_max, logprob=logprob, token_pred=token_pred)
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden must be [T_pad, H] and weight [V, H]")
    T_pad, H = hidden.shape
    V = weight.shape[0]
    _need(key_reach, torch.int32, "key_reach")
    if blockmap is not None:
        _need(blockmap, torch.int32, "blockmap")
    for t, n in ((key_reach, "key_reach"), (token_ids, "token_ids"), (token_pred, "token_pred"),
                 (lse, "lse"), (entropy, "entropy"), (vocab_min, "vocab_min"),
                 (vocab_max, "vocab_max"), (logprob, "logprob")):
        if t is not None:
            _need(t, torch.int32 if n in ("key_reach", "token_ids", "token_pred")
                  else torch.float32, n)
            if t.numel() != T_pad:
                raise ValueError(f"{n} must hold T_pad = {T_pad} values")
    _check("tree_lm_head_logprobs_entropy", _lib.tree_lm_head_logprobs_entropy(
        _ptr(hidden), _ptr(weight), T_pad, H, V, _ptr(token_ids), _ptr(key_reach),
        _ptr(blockmap), 0 if blockmap is None else _nbytes(blockmap), _ptr(lse), _ptr(entropy),
        _ptr(vocab_min), _ptr(vocab_max), _ptr(logprob), _ptr(token_pred), _ptr(workspace),
        _nbytes(workspace), _ptr(dev_status), _stream_ptr(stream)))


def lm_head_grad_workspace_bytes(rows: int) -> int:
    return int(_lib.tree_lm_head_grad_workspace_bytes(int(rows)))


def tree_lm_head_logits_grad(hidden, weight, key_reach, lse, grad_logits, workspace, dev_status,
                             row_lo: int = 0, row_hi: int | None = None, token_ids=None,
                             entropy=None, grad_logprob=None, grad_entropy=None, stream=None):
    """Gradient of the fused gather with respect to the logits of rows
    ``[row_lo, row_hi)`` into ``grad_logits`` (bf16 ``[rows, V]``, unit stride
    along V), recomputing the logits tile by tile."""
    import torch
    _on_device(hidden=hidden, weight=weight, key_reach=key_reach, lse=lse,
               grad_logits=grad_logits, workspace=workspace, dev_status=dev_status,
               token_ids=token_ids, entropy=entropy, grad_logprob=grad_logprob,
               grad_entropy=grad_entropy)
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight")
    T_pad, H = hidden.shape
    V = weight.shape[0]
    row_hi = T_pad if row_hi is None else int(row_hi)
    if (grad_logits.dtype != torch.bfloat16 or grad_logits.dim() != 2
            or grad_logits.stride(1) != 1 or grad_logits.shape[1] != V
            or grad_logits.shape[0] != row_hi - int(row_lo)):
        raise ValueError("grad_logits must be bf16 [row_hi - row_lo, V] with unit stride along V")
    for t, n in ((key_reach, "key_reach"), (token_ids, "token_ids"), (lse, "lse"),
                 (entropy, "entropy"), (grad_logprob, "grad_logprob"),
                 (grad_entropy, "grad_entropy")):
        if t is not None:
            _need(t, torch.int32 if n in ("key_reach", "token_ids") else torch.float32, n)
            if t.numel() != T_pad:
                raise ValueError(f"{n} must hold T_pad = {T_pad} values")
    _check("tree_lm_head_logits_grad", _lib.tree_lm_head_logits_grad(
        _ptr(hidden), _ptr(weight), T_pad, H, V, int(row_lo), row_hi, _ptr(token_ids),
        _ptr(key_reach), _ptr(lse), _ptr(entropy), _ptr(grad_logprob), _ptr(grad_entropy),
        _ptr(grad_logits), grad_logits.stride(0), _ptr(workspace), _nbytes(workspace),
        _ptr(dev_status), _stream_ptr(stream)))


DTA_FWD_PUSH, DTA_FWD_BWD, DTA_BWD_POP = 0, 1, 2


def dta_schedule(token_node, node_entry, node_exit, chunk: int = 2048):
    """The depth-first traversal of dynamic tree attention for one packed
    trie (host arrays): returns ``(ops, peak_stack_tokens)`` with ``ops`` an
    int32 array ``[n_ops, 3]`` of ``(kind, t0, t1)``."""
    tn = np.ascontiguousarray(token_node, dtype=np.int32)
    en = np.ascontiguousarray(node_entry, dtype=np.int32)
    ex = np.ascontiguousarray(node_exit, dtype=np.int32)
    n_ops, peak = ctypes.c_int64(), ctypes.c_int64()
    args = (tn.ctypes.data if tn.size else None, tn.size, en.ctypes.data if en.size else None,
            ex.ctypes.data if ex.size else None, en.size, int(chunk))
    _check("tree_dta_schedule", _lib.tree_dta_schedule(*args, None, 0, ctypes.byref(n_ops),
                                                       ctypes.byref(peak)))
    ops = np.zeros((max(1, n_ops.value), 3), np.int32)
    _check("tree_dta_schedule", _lib.tree_dta_schedule(*args, ops.ctypes.data, n_ops.value,
                                                       ctypes.byref(n_ops), ctypes.byref(peak)))
    return ops[:n_ops.value], int(peak.value)


def dta_attn_workspace_bytes(T_pad: int, Hq: int, Hkv: int, d: int) -> int:
    return int(_lib.tree_dta_attn_workspace_bytes(T_pad, Hq, Hkv, d))


def tree_dta_attn(q, k, v, d_o, key_reach, blockmap, ops, o, lse, dq, dk, dv, workspace,
                  dev_status, scale=None, stream=None):
    """Attention forward + backward executed op by op through a depth-first
    traversal schedule ``ops`` (host int32 ``[n_ops, 3]`` of (kind, t0, t1),
    e.g. from :func:`dta_schedule`)."""
    import torch
    _on_device(q=q, k=k, v=v, d_o=d_o, key_reach=key_reach, blockmap=blockmap, o=o, lse=lse,
               dq=dq, dk=dk, dv=dv, workspace=workspace, dev_status=dev_status)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_o, "d_o"), (o, "o"), (dq, "dq"), (dk, "dk"),
                 (dv, "dv")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    if (k.shape != (T, Hkv, d) or v.shape != k.shape or d_o.shape != q.shape or
            o.shape != q.shape or dq.shape != q.shape or dk.shape != k.shape or
            dv.shape != k.shape or lse.shape != (Hq, T)):
        raise ValueError("shape mismatch")
    _check_reach_blockmap(key_reach, blockmap, T)
    host_ops = np.ascontiguousarray(ops, dtype=np.int32).reshape(-1, 3)
    scale = d ** -0.5 if scale is None else float(scale)
    _check("tree_dta_attn", _lib.tree_dta_attn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(d_o), _ptr(key_reach), _ptr(blockmap),
        _nbytes(blockmap), T, Hq, Hkv, d, scale,
        host_ops.ctypes.data if host_ops.size else None, host_ops.shape[0], _ptr(o), _ptr(lse),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), _nbytes(workspace), _ptr(dev_status),
        _stream_ptr(stream)))


def sequence_index_arrays(tries, n_seqs: int, trie_offsets=None):
    """Host bookkeeping for ``tree_merge_per_sequence``: the packed indices
    of every input sequence's tokens (plus its trie's offset in a buffer that
    holds several tries), flattened in sequence-id order, and the int64
    offsets of each sequence in that list."""
    if trie_offsets is None:
        trie_offsets = np.cumsum([0] + [t.T_pad for t in tries[:-1]]).tolist()
    per = [None] * n_seqs
    for t, base in zip(tries, trie_offsets):
        for sid, idx in t.seq_index.items():
            per[sid] = np.asarray(idx, np.int64) + int(base)
    lens = np.array([0 if p is None else p.size for p in per], np.int64)
    offs = np.zeros(n_seqs + 1, np.int64)
    np.cumsum(lens, out=offs[1:])
    flat = np.concatenate([p for p in per if p is not None]) if offs[-1] else np.zeros(0)
    return flat.astype(np.int32), offs


def tree_attn_bwd_prepare(o, d_o, lse, workspace, dev_status, stream=None):
    _on_device(o=o, d_o=d_o, lse=lse, workspace=workspace, dev_status=dev_status)
    T, Hq, d = o.shape
    _check("tree_attn_bwd_prepare", _lib.tree_attn_bwd_prepare(
        _ptr(o), _ptr(d_o), _ptr(lse), T, Hq, d, _ptr(workspace), _nbytes(workspace),
        _ptr(dev_status), _stream_ptr(stream)))


def tree_attn_bwd_main(q, k, v, d_o, key_reach, blockmap, dk, dv, workspace, dev_status,
                       scale=None, stream=None):
    _on_device(q=q, k=k, v=v, d_o=d_o, key_reach=key_reach, blockmap=blockmap, dk=dk, dv=dv,
               workspace=workspace, dev_status=dev_status)
    T, Hq, d = q.shape
    _check_reach_blockmap(key_reach, blockmap, T)
    scale = d ** -0.5 if scale is None else float(scale)
    _check("tree_attn_bwd_main", _lib.tree_attn_bwd_main(
        _ptr(q), _ptr(k), _ptr(v), _ptr(d_o), _ptr(key_reach), _ptr(blockmap),
        _nbytes(blockmap), T, Hq, k.shape[1], d, scale, _ptr(dk), _ptr(dv), _ptr(workspace),
        _nbytes(workspace), _ptr(dev_status), _stream_ptr(stream)))


def tree_attn_bwd_finish(workspace, dq, dev_status, scale=None, stream=None):
    _on_device(workspace=workspace, dq=dq, dev_status=dev_status)
    T, Hq, d = dq.shape
    scale = d ** -0.5 if scale is None else float(scale)
    _check("tree_attn_bwd_finish", _lib.tree_attn_bwd_finish(
        T, Hq, d, scale, _ptr(workspace), _nbytes(workspace), _ptr(dq), _ptr(dev_status),
        _stream_ptr(stream)))


def launch_count() -> int:
    """Kernels the library has queued so far in this process."""
    return int(_lib.tree_launch_count())


def tree_debug_wait_timeout(dev_status, limit_ns: int, stream=None):
    """Run the bounded-wait probe; TREE_ERR_TIMEOUT lands in dev_status."""
    _on_device(dev_status=dev_status)
    _check("tree_debug_wait_timeout", _lib.tree_debug_wait_timeout(
        _ptr(dev_status), int(limit_ns), _stream_ptr(stream)))


# --------------------------------------------------------------- host packer
@dataclass
class Trie:
    """One packed trie from the host packer (numpy int32 arrays)."""

    n_tokens: int
    T_pad: int
    n_nodes: int
    visible_pairs: int
    token_node: np.ndarray
    token_ids: np.ndarray
    node_entry: np.ndarray
    node_exit: np.ndarray
    seq_ids: list
    seq_index: dict      # input sequence index -> packed token indices


def pack_sequences(seqs, max_tokens_per_mb: int, block: int = BLOCK, pad_to_max: bool = False):
    """Pack token sequences into tries with the library's host packer."""
    lens = np.array([len(s) for s in seqs], dtype=np.int64)
    offs = np.zeros(len(seqs) + 1, dtype=np.int64)
    np.cumsum(lens, out=offs[1:])
    flat = np.zeros(max(1, int(offs[-1])), dtype=np.int32)
    for i, s in enumerate(seqs):
        flat[offs[i]:offs[i + 1]] = s
    handle = ctypes.c_void_p()
    _check("tree_packing_build", _lib.tree_packing_build(
        flat.ctypes.data, offs.ctypes.data, len(seqs), int(max_tokens_per_mb), int(block),
        1 if pad_to_max else 0, ctypes.byref(handle)))
    try:
        out = []
        for t in range(_lib.tree_packing_num_tries(handle)):
            nt, tp, nn, ns = (ctypes.c_int32() for _ in range(4))
            pairs = ctypes.c_int64()
            _check("tree_packing_trie_info", _lib.tree_packing_trie_info(
                handle, t, ctypes.byref(nt), ctypes.byref(tp), ctypes.byref(nn),
                ctypes.byref(ns), ctypes.byref(pairs)))
            token_node = np.empty(tp.value, np.int32)
            token_ids = np.empty(tp.value, np.int32)
            entry = np.empty(nn.value, np.int32)
            exit_ = np.empty(nn.value, np.int32)
            sids = np.empty(ns.value, np.int32)
            _check("tree_packing_trie_arrays", _lib.tree_packing_trie_arrays(
                handle, t, token_node.ctypes.data, token_ids.ctypes.data, entry.ctypes.data,
                exit_.ctypes.data, sids.ctypes.data))
            seq_index = {}
            for k_, sid in enumerate(sids.tolist()):
                idx = np.empty(len(seqs[sid]), np.int32)
                _check("tree_packing_seq_indices", _lib.tree_packing_seq_indices(
                    handle, t, k_, idx.ctypes.data, idx.size))
                seq_index[sid] = idx
            out.append(Trie(nt.value, tp.value, nn.value, pairs.value, token_node, token_ids,
                            entry, exit_, sids.tolist(), seq_index))
        return out
    finally:
        _lib.tree_packing_free(handle)


def _flatten(seqs):
    lens = np.array([len(s) for s in seqs], dtype=np.int64)
    offs = np.zeros(len(seqs) + 1, dtype=np.int64)
    np.cumsum(lens, out=offs[1:])
    flat = np.zeros(max(1, int(offs[-1])), dtype=np.int32)
    for i, s in enumerate(seqs):
        flat[offs[i]:offs[i + 1]] = s
    return flat, offs


def partition_sequences(seqs, n_groups: int):
    """Split token sequences over ``n_groups`` workers with the library's
    load-balanced partitioner (contiguous segments of the sequences' DFS
    order, largest per-group prefix-tree token count minimised).  Returns
    ``(group_of_seq int32[n], group_cost int64[n_groups], max_cost)``."""
    flat, offs = _flatten(seqs)
    groups = np.empty(len(seqs), np.int32)
    cost = np.empty(max(1, int(n_groups)), np.int64)
    mx = ctypes.c_int64()
    _check("tree_partition_sequences", _lib.tree_partition_sequences(
        flat.ctypes.data, offs.ctypes.data, len(seqs), int(n_groups), groups.ctypes.data,
        cost.ctypes.data, ctypes.byref(mx)))
    return groups, cost[:int(n_groups)], int(mx.value)


# --------------------------------------------------------------- convenience
class TrieBuffers:
    """Device buffers for one trie: positions, reach, blockmap, workspaces.

    Allocates with torch once; every call after that only launches kernels.
    """

    def __init__(self, T_pad: int, n_nodes: int, Hq: int, d: int, device="cuda"):
        import torch
        self.T_pad, self.n_nodes, self.Hq, self.d = T_pad, n_nodes, Hq, d
        i32 = dict(dtype=torch.int32, device=device)
        self.position_ids = torch.empty(T_pad, **i32)
        self.key_reach = torch.empty(T_pad, **i32)
        self.pos_ws = torch.empty((pack_positions_workspace_bytes(T_pad, n_nodes) + 3) // 4, **i32)
        self.blockmap = torch.empty((blockmap_bytes(T_pad) + 3) // 4, **i32)
        self.bwd_ws = torch.empty((attn_bwd_workspace_bytes(T_pad, Hq, d) + 3) // 4,
                                  dtype=torch.float32, device=device)
        self.status = torch.zeros(1, **i32)


def blockmap_view(blockmap_words: np.ndarray) -> dict:
    """Decode a blockmap buffer (host copy, int32 words) into its fields."""
    nb = int(blockmap_words[0])
    w = blockmap_words
    nnz = int(w[1])
    col_full_hi = w[4:4 + nb]
    col_hi = w[4 + nb:4 + 2 * nb]
    row_cnt = w[4 + 2 * nb:4 + 3 * nb]
    row_nfull = w[4 + 3 * nb:4 + 4 * nb]
    row_ptr = w[4 + 4 * nb:5 + 5 * nb]
    row_order = w[5 + 5 * nb:5 + 6 * nb]
    col_order = w[5 + 6 * nb:5 + 7 * nb]
    row_idx = w[5 + 7 * nb:5 + 7 * nb + nnz]
    return dict(nb=nb, nnz=nnz, col_full_hi=col_full_hi, col_hi=col_hi, row_cnt=row_cnt,
                row_nfull=row_nfull, row_ptr=row_ptr, row_order=row_order, col_order=col_order,
                row_idx=row_idx)


def tile_classes_from_blockmap(view: dict) -> np.ndarray:
    """Dense uint8[nb, nb] tile classes (0 EMPTY, 1 FULL, 2 PARTIAL) expanded
    from the blockmap's per-column runs."""
    nb = view["nb"]
    cls = np.zeros((nb, nb), np.uint8)
    for kb in range(nb):
        hi, fh = int(view["col_hi"][kb]), int(view["col_full_hi"][kb])
        for qa in range(kb, hi + 1):
            cls[qa, kb] = 2 if (qa == kb or qa > fh) else 1
    return cls
