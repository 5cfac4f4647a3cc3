"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers: token sequences with the structure of
each workload, and N(0, 1) bf16 tensors.  It holds none of the method's
arithmetic (no trie, no packing, no mask, no attention), so both the CUDA
path and the oracle can consume what it produces.

Workloads (structure follows the tree-training pages' shared-prefix RL
batches: n_samples responses per prompt, shared system prompts, multi-turn
histories; the pages' own agent benchmark data is not used — these seeded
stand-ins have its shapes and length mix):

1. ``tiny``     1 trie, 8 responses to one 256-token prompt, response length
                U[32,256]; responses (0,1), (2,3), ... also share U[0,64]
                further tokens (capped so the pair still diverges);
                max_tokens_per_mb 2048; 4 q / 4 kv heads, head_dim 64.
2. ``grpo``     64 prompts x 8 samples, prompt U[512,2048], response
                U[256,4096], no shared response tokens; max_tokens_per_mb
                32768; 32 q / 8 kv heads, head_dim 128.
3. ``agent``    32 tasks x 8 rollouts under one 1024-token system prompt;
                4..10 turns of U[128,1024] tokens; rollout r > 0 copies the
                first b ~ U{0..min(n_r, n_parent) - 1} turns of a uniformly
                chosen earlier rollout of its task; max_tokens_per_mb 32768.
4. ``long``     16 prompts x 8 samples, prompt U[1024,2048], response
                lognormal(ln 4096, 0.5) clipped to [2048, 8192];
                max_tokens_per_mb 65536.
5. ``fanout``   one 16384-token prefix with 512 leaves of U[16,64] tokens;
                max_tokens_per_mb 49152.

Every fresh segment gets token ids never used before, so siblings always
diverge and the only sharing is the one the recipe builds.

Random numbers: structure comes from SplitMix64 (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014), uniform
integers by scaling a 53-bit uniform, normals by Box-Muller.  Tensor values
come from ``torch.randn`` under a seeded ``torch.Generator`` on the device
that will hold them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

_MASK = (1 << 64) - 1


class SplitMix64:
    """Counter-based 64-bit generator (published constants of SplitMix64)."""

    def __init__(self, seed: int):
        self.state = seed & _MASK

    def next_u64(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & _MASK
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
        return z ^ (z >> 31)

    def uniform(self) -> float:
        return (self.next_u64() >> 11) * (1.0 / (1 << 53))

    def randint(self, lo: int, hi: int) -> int:
        """Uniform integer in [lo, hi] (both inclusive)."""
        return lo + min(hi - lo, int(self.uniform() * (hi - lo + 1)))

    def normal(self) -> float:
        u1 = max(self.uniform(), 1e-300)
        u2 = self.uniform()
        return math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)


@dataclass(frozen=True)
class Workload:
    key: str
    index: int          # 1-based position in the workload list
    Hq: int
    Hkv: int
    d: int
    max_tokens_per_mb: int
    description: str


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 4, 64, 2048,
                     "1 trie: 8 responses U[32,256] to a 256-token prompt, pairs share U[0,64]"),
    "grpo": Workload("grpo", 2, 32, 8, 128, 32768,
                     "64 prompts U[512,2048] x 8 responses U[256,4096], FFD at 32768"),
    "agent": Workload("agent", 3, 32, 8, 128, 32768,
                      "32 tasks x 8 rollouts, 1024-token system prompt, 4-10 turns U[128,1024]"),
    "long": Workload("long", 4, 32, 8, 128, 65536,
                     "16 prompts U[1024,2048] x 8 responses lognormal(ln4096,0.5) in [2048,8192]"),
    "fanout": Workload("fanout", 5, 32, 8, 128, 49152,
                       "16384-token prefix + 512 leaves U[16,64]"),
}


class _Ids:
    def __init__(self):
        self.next = 1

    def fresh(self, n: int) -> list[int]:
        out = list(range(self.next, self.next + n))
        self.next += n
        return out


def _tiny(rng: SplitMix64, ids: _Ids):
    prompt = ids.fresh(256)
    seqs = []
    for _pair in range(4):
        la, lb = rng.randint(32, 256), rng.randint(32, 256)
        s = min(rng.randint(0, 64), min(la, lb) - 1)
        shared = ids.fresh(s)
        for L in (la, lb):
            seqs.append(prompt + shared + ids.fresh(L - s))
    return seqs


def _grpo(rng: SplitMix64, ids: _Ids):
    seqs = []
    for _p in range(64):
        prompt = ids.fresh(rng.randint(512, 2048))
        for _s in range(8):
            seqs.append(prompt + ids.fresh(rng.randint(256, 4096)))
    return seqs


def _agent(rng: SplitMix64, ids: _Ids):
    system = ids.fresh(1024)
    seqs = []
    for _task in range(32):
        rollouts: list[list[list[int]]] = []
        for r in range(8):
            n = rng.randint(4, 10)
            if r == 0:
                turns = [ids.fresh(rng.randint(128, 1024)) for _ in range(n)]
            else:
                parent = rollouts[rng.randint(0, r - 1)]
                b = rng.randint(0, min(n, len(parent)) - 1)
                turns = parent[:b] + [ids.fresh(rng.randint(128, 1024))
                                      for _ in range(n - b)]
            rollouts.append(turns)
            seqs.append(system + [t for turn in turns for t in turn])
    return seqs


def _long(rng: SplitMix64, ids: _Ids):
    seqs = []
    for _p in range(16):
        prompt = ids.fresh(rng.randint(1024, 2048))
        for _s in range(8):
            L = int(round(math.exp(math.log(4096.0) + 0.5 * rng.normal())))
            seqs.append(prompt + ids.fresh(min(8192, max(2048, L))))
    return seqs


def _fanout(rng: SplitMix64, ids: _Ids):
    prefix = ids.fresh(16384)
    return [prefix + ids.fresh(rng.randint(16, 64)) for _ in range(512)]


_BUILDERS = {"tiny": _tiny, "grpo": _grpo, "agent": _agent, "long": _long,
             "fanout": _fanout}


def sequences(key: str, seed: int = 0) -> list[list[int]]:
    """Token sequences of workload ``key`` (each a list of positive ids)."""
    return _BUILDERS[key](SplitMix64(0x5EED0000 + 7919 * seed + WORKLOADS[key].index), _Ids())


def random_sequences(rng: SplitMix64, n_seqs: int, max_len: int, alphabet: int):
    """Small random sequences over ``alphabet`` letters (ids 1..alphabet)."""
    return [[rng.randint(1, alphabet) for _ in range(rng.randint(1, max_len))]
            for _ in range(n_seqs)]


def tensors(T: int, Hq: int, Hkv: int, d: int, seed: int, stream: int = 0,
            device="cpu"):
    """bf16 N(0, 1) tensors q, k, v, do of shapes [T, H, d] for one trie."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((0x7A11 + 1000003 * seed + 8191 * stream) & ((1 << 63) - 1))
    shape_q, shape_kv = (T, Hq, d), (T, Hkv, d)
    out = {}
    for name, shape in (("q", shape_q), ("k", shape_kv), ("v", shape_kv), ("do", shape_q)):
        out[name] = torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
    return out


def logits(T: int, V: int, seed: int, device="cpu", dtype=None, sigma: float = 2.0,
           row_stride: int | None = None):
    """Packed next-token logits [T, V] drawn as sigma * N(0, 1), rounded to
    ``dtype`` (bf16 by default).  With ``row_stride`` > V the rows sit in a
    wider buffer and the view [:, :V] is returned."""
    import torch
    dtype = torch.bfloat16 if dtype is None else dtype
    g = torch.Generator(device=device)
    g.manual_seed((0x10C1 + 1000033 * seed) & ((1 << 63) - 1))
    width = V if row_stride is None else row_stride
    buf = torch.randn((T, width), generator=g, device=device, dtype=torch.float32)
    buf = (buf * sigma).to(dtype)
    return buf[:, :V]


def lm_head(T: int, H: int, V: int, seed: int, device="cpu"):
    """Hidden states [T, H] ~ N(0, 1) and LM-head weights [V, H] ~
    N(0, (2 / sqrt(H))^2), both rounded to bf16, so the logits
    hidden @ weight^T have standard deviation about 2 (the sigma of
    ``logits``)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((0x1A4E + 7919 * seed) & ((1 << 63) - 1))
    hidden = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
    weight = torch.randn((V, H), generator=g, device=device, dtype=torch.float32)
    weight *= 2.0 / float(H) ** 0.5
    return hidden.to(torch.bfloat16), weight.to(torch.bfloat16)
