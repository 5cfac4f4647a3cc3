"""Benchmark of the packed-trie attention hot path on GB300.

One step = the whole hot path over one batch of the workload: for every trie
of the batch, position ids + key reach (a1), blockmap (a2), attention forward
(a3), backward prepare / main / finish (a4-a6).  The tries of a batch are
independent, so consecutive tries alternate over two CUDA streams (each with
its own backward workspace): one trie's kernels fill the SMs that another
trie's kernel tails and small kernels leave idle.  The per-kernel roofline
figures come from a separate pass that runs the tries on one stream.  Default workload: GRPO-style
groups (64 prompts x 8 responses, first-fit-decreasing into 32768-token tries,
Qwen3-8B attention heads 32 q / 8 kv, head_dim 128), seeded synthetic data.

Metric: effective TFLOP/s = 14 * d * Hq * (visible pairs) / step time, where
visible pairs count only unmasked (i, j) over real tokens (4 d Hq per pair
for the forward, 10 d Hq for the backward).  Packed tokens/s is reported too.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--split replicas|balanced] [--path attention|logprob|dta|lmhead]
--path logprob times the tree-aware log-probability / entropy gather over the
same batch instead (bf16 logits over the Qwen3 vocabulary; its own JSON line);
--path dta runs the attention through the depth-first traversal schedule of
dynamic tree attention (--chunk tokens per op) beside the packed step;
--path lmhead times Qwen3-8B's LM head fused with the gather (no logits).
Under torchrun each rank runs its own batch (seed = rank, --split replicas,
the default): weak scaling, no collective on the data path.  With --split
balanced every rank takes the same global batch and keeps one group of the
library's load-balanced partition (contiguous segments of the batch's DFS
order, largest per-rank prefix-tree token count minimised): strong scaling.
Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "tree-attn fwd+bwd effective TFLOP/s and packed tokens/s vs bf16 TC peak"
UNIT = "TFLOP/s"
FWD_FLOPS_PER_PAIR = 4      # times d * Hq
BWD_FLOPS_PER_PAIR = 10
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "bwd_main_traffic.json")
CSRC = os.path.join(ROOT, "prefix_tree_attention_gb300", "csrc")
# A kernel's source: its translation unit and the headers it includes.
KERNEL_SOURCE = [os.path.join(CSRC, f) for f in ("attn_bwd.cu", "common.cuh", "ptx.cuh")]
LOGPROB_TRAFFIC = os.path.join(ROOT, "profiles", "logprob_row_stats_traffic.json")
LOGPROB_BWD_TRAFFIC = os.path.join(ROOT, "profiles", "logprob_row_bwd_traffic.json")
LOGPROB_SOURCE = [os.path.join(CSRC, f)
                  for f in ("logprob.cu", "rowstats.cuh", "common.cuh", "ptx.cuh")]


# ------------------------------------------------------------------ helpers
def rank_batch(ptg, key: str, seed: int, rank: int, world: int, split: str):
    """Sequences this rank trains on, and the seed of its tensor data.

    replicas: an independent batch per rank (seed + rank).
    balanced: the global batch (seed) split over the ranks by the library's
    load-balanced partitioner; rank r keeps group r."""
    if split == "replicas" or world == 1:
        return W.sequences(key, seed + rank), seed + rank
    seqs = W.sequences(key, seed)
    groups, _cost, _mx = ptg.partition_sequences(seqs, world)
    return [sq for sq, g in zip(seqs, groups.tolist()) if g == rank], seed + rank


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(bf16=p["bf16_tflops"], bf16_sustained=p["bf16_tflops_sustained"],
                    hbm=p["hbm_gbs"], source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


def source_hash(paths) -> str:
    """sha256/16 of a kernel's source files, concatenated in the order given."""
    h = hashlib.sha256()
    for path in ([paths] if isinstance(paths, str) else paths):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_logprob_traffic_per_row(path=LOGPROB_TRAFFIC):
    """DRAM bytes per real packed row of a log-prob row kernel (the forward
    row pass, or with ``LOGPROB_BWD_TRAFFIC`` the gradient's), from a
    committed ncu summary of a smaller case; None when absent or taken on a
    different kernel source."""
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256_16") != source_hash(LOGPROB_SOURCE):
        return None
    return rec["dram_bytes_captured_launch"] / rec["real_rows_captured_launch"]


def recorded_traffic():
    """DRAM bytes of the bwd main kernel over one step of the default
    workload (all its launches), from a committed ncu summary; None when
    absent or taken on a different kernel source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256_16") != source_hash(KERNEL_SOURCE):
        return None
    return rec.get("dram_bytes_per_step")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        self.index = ids[local_index] if local_index < len(ids) else str(local_index)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if s[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ oracle leg
def oracle_sample(key: str, seed: int, budget_s: float, tensors_fn=None):
    """Time the oracle (as it stands) on a bounded sample of the workload: the
    per-row forward + backward of evenly spaced rows of the first trie, for
    the query heads of key/value head 0.  Returns (TFLOP/s, description,
    seconds, threads)."""
    from oracle import attention as OA
    from oracle import trie as OT
    import torch

    wl = W.WORKLOADS[key]
    seqs = W.sequences(key, seed)
    (ref, *_rest) = OT.pack_sequences(seqs, wl.max_tokens_per_mb)
    g = wl.Hq // wl.Hkv
    if tensors_fn is None:
        t = W.tensors(ref.T_pad, wl.Hq, wl.Hkv, wl.d, seed=seed * 1000, device="cpu")
    else:
        t = tensors_fn(ref)
    q = t["q"][:, :g].double().numpy()
    k = t["k"][:, :1].double().numpy()
    v = t["v"][:, :1].double().numpy()
    do = t["do"][:, :g].double().numpy()
    real = np.nonzero(ref.token_node >= 0)[0]
    order = real[np.argsort((real * 0.6180339887) % 1.0)]   # spread-out row order
    from oracle import mask as OM
    done = []
    t0 = time.perf_counter()
    c0 = time.process_time()
    for i in order:
        _o, _l, _dq, _dk, _dv = OA.rows_forward_backward(q, k, v, do, ref, [int(i)], range(g))
        done.append(int(i))
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    # threads the sample actually kept busy: process CPU time over wall time
    # (numpy's BLAS may thread the per-row products; the Python loop is serial)
    cores_used = round((time.process_time() - c0) / dt, 2) if dt > 0 else 1.0
    rows_done = len(done)
    pairs = sum(int(OM.mask_rows(ref, i, i + 1).sum()) for i in done)
    flops = (FWD_FLOPS_PER_PAIR + BWD_FLOPS_PER_PAIR) * wl.d * g * pairs
    desc = (f"oracle per-row fwd+bwd (fp64 numpy), {rows_done} rows of trie 0 of '{key}' "
            f"({pairs} visible pairs), query heads 0-{g - 1} of kv head 0; one Python "
            f"process, {cores_used} cores busy on average (CPU time / wall time), "
            f"{os.cpu_count()} host cores present")
    del torch
    return flops / dt / 1e12, desc, dt, cores_used


def logprob_oracle_rate(budget_s: float, seed: int, rows: int = 64, V: int = 151936):
    """Time the log-prob oracle (as it stands) on host rows of bf16 logits over
    the Qwen3 vocabulary: per row its statistics (log-sum-exp, entropy, vocab
    min/max) and its log-softmax, which is what every packed token costs.
    Returns (rows per second, description)."""
    from oracle import logprob as OL
    host = W.logits(rows, V, seed=seed).float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    done = 0
    while True:
        OL.row_stats(host[done % rows])
        OL.log_softmax(host[done % rows])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, f"{done} rows of V={V} (row stats + log-softmax, fp64 numpy, one core)"


def run_reference_logprob(args):
    budget = min(args.cpu_budget, 10.0)
    vals, desc = [], None
    for step in range(args.warmup + args.steps):
        v, desc = logprob_oracle_rate(budget, args.seed)
        if step >= args.warmup:
            vals.append(v)
    value = round(float(np.median(vals)), 2)
    line = {
        "impl": "reference", "metric": LOGPROB_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "path": "logprob", "vocab": 151936},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_lmhead(args):
    budget = min(args.cpu_budget, 15.0)
    vals, desc = [], None
    for step in range(args.warmup + args.steps):
        v, desc = lmhead_oracle_rate(budget / max(1, args.warmup + args.steps) * 4, args.seed)
        if step >= args.warmup:
            vals.append(v)
    value = round(float(np.median(vals)), 3)
    line = {
        "impl": "reference", "metric": LMHEAD_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "path": "lmhead", "hidden": QWEN3_HIDDEN,
                   "vocab": QWEN3_VOCAB},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, rank, ws):
    if rank != 0:
        return
    if args.path == "logprob":
        run_reference_logprob(args)
        return
    if args.path == "lmhead":
        run_reference_lmhead(args)
        return
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    vals = []
    desc = cores = None
    for step in range(args.warmup + args.steps):
        v, desc, _dt, cores = oracle_sample(args.workload, args.seed, budget)
        if step >= args.warmup:
            vals.append(v)
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": W.WORKLOADS[args.workload].description},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
class TrieCase:
    """Device-resident inputs, outputs and buffers of one trie."""

    def __init__(self, ptg, tr, wl, seed, idx, device):
        import torch
        self.tr = tr
        T = tr.T_pad
        self.T, self.Hq, self.Hkv, self.d = T, wl.Hq, wl.Hkv, wl.d
        self.token_node = torch.from_numpy(tr.token_node).to(device)
        self.entry = torch.from_numpy(tr.node_entry).to(device)
        self.exit = torch.from_numpy(tr.node_exit).to(device)
        t = W.tensors(T, wl.Hq, wl.Hkv, wl.d, seed=seed * 1000 + idx, device=device)
        self.q, self.k, self.v, self.do = t["q"], t["k"], t["v"], t["do"]
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((wl.Hq, T), dtype=torch.float32, device=device)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.bufs = ptg.TrieBuffers(T, tr.n_nodes, wl.Hq, wl.d, device=device)
        self.pairs = tr.visible_pairs
        self.n_tokens = tr.n_tokens

    def input_tensors(self):
        return [self.token_node, self.entry, self.exit, self.q, self.k, self.v, self.do]

    def output_tensors(self):
        return [self.o, self.dq, self.dk, self.dv]


def run_path(ptg, c, ws_bwd, stream, ev=None):
    """Queue the whole hot path for one trie on `stream`."""
    b = c.bufs
    ptg.tree_pack_positions(c.token_node, c.entry, c.exit, b.position_ids, b.key_reach, b.pos_ws,
                            b.status, stream=stream)
    ptg.tree_blockmap_build(b.key_reach, b.blockmap, b.status, stream=stream)
    if ev is not None:
        ev[0].record(stream)
    ptg.tree_attn_fwd(c.q, c.k, c.v, b.key_reach, b.blockmap, c.o, c.lse, b.status, stream=stream)
    if ev is not None:
        ev[1].record(stream)
    ptg.tree_attn_bwd_prepare(c.o, c.do, c.lse, ws_bwd, b.status, stream=stream)
    if ev is not None:
        ev[2].record(stream)
    ptg.tree_attn_bwd_main(c.q, c.k, c.v, c.do, b.key_reach, b.blockmap, c.dk, c.dv, ws_bwd,
                           b.status, stream=stream)
    if ev is not None:
        ev[3].record(stream)
    ptg.tree_attn_bwd_finish(ws_bwd, c.dq, b.status, stream=stream)


def build_cases(ptg, key, seed, rank, ws, split, n_tries, device):
    """Packed tries of one workload with their device-resident inputs."""
    wl = W.WORKLOADS[key]
    seqs, seed = rank_batch(ptg, key, seed, rank, ws, split)
    tries = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)
    if n_tries:
        tries = tries[:n_tries]
        used = {s for tr in tries for s in tr.seq_ids}
        seqs = [s for i, s in enumerate(seqs) if i in used]
    cases = [TrieCase(ptg, tr, wl, seed, i, device) for i, tr in enumerate(tries)]
    return wl, seqs, cases


class Stepper:
    """One step = the whole hot path over every trie of the batch; trie i on
    stream i % n_streams (each stream with its own backward workspace)."""

    def __init__(self, ptg, cases, wl, n_streams, device):
        import torch
        self.ptg, self.cases = ptg, cases
        ws_bytes = max(ptg.attn_bwd_workspace_bytes(c.T, wl.Hq, wl.d) for c in cases)
        self.n_streams = max(1, min(n_streams, len(cases)))
        self.ws_bwds = [torch.empty((ws_bytes + 3) // 4, dtype=torch.float32, device=device)
                        for _ in range(self.n_streams)]
        self.streams = [torch.cuda.Stream(device=device) for _ in range(self.n_streams)]
        self.stream = self.streams[0]

    def step(self):
        import torch
        start = torch.cuda.Event()
        start.record(self.stream)
        for st in self.streams[1:]:
            st.wait_event(start)
        for i, c in enumerate(self.cases):
            st = self.streams[i % self.n_streams]
            with torch.cuda.stream(st):
                run_path(self.ptg, c, self.ws_bwds[i % self.n_streams], st)
        for st in self.streams[1:]:
            done = torch.cuda.Event()
            done.record(st)
            self.stream.wait_event(done)

    def serial_step(self, ev_list):
        """The whole batch on one stream, with per-kernel events."""
        import torch
        with torch.cuda.stream(self.stream):
            for i, c in enumerate(self.cases):
                run_path(self.ptg, c, self.ws_bwds[0], self.stream, ev_list[i])

    def check_status(self, when):
        bad = [int(c.bufs.status.item()) for c in self.cases]
        if any(bad):
            raise RuntimeError(f"device status {self.ptg.status_string(max(bad))} {when}")

    def timed(self, steps, clk_index=None):
        """Per-step device times (ms) of `steps` steps, CUDA events on the
        stream that starts and joins every step."""
        import torch
        mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        torch.cuda.synchronize()
        per_step = []
        for _ in range(steps):
            s0, s1 = mk(), mk()
            s0.record(self.stream)
            self.step()
            s1.record(self.stream)
            per_step.append((s0, s1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in per_step]


def workload_stats(wl, seqs, cases):
    pairs = sum(c.pairs for c in cases)
    tokens = sum(c.n_tokens for c in cases)
    original = sum(len(s) for s in seqs)
    causal_pairs = sum(len(s) * (len(s) + 1) // 2 for s in seqs)
    return dict(pairs=pairs, tokens=tokens, original=original, causal_pairs=causal_pairs,
                flops=(FWD_FLOPS_PER_PAIR + BWD_FLOPS_PER_PAIR) * wl.d * wl.Hq * pairs)


def run_extra_workload(ptg, key, args, rank, ws, device, peaks):
    """A bounded timing of another workload of the metric (same step, same
    streams), reported under config.per_workload."""
    import torch
    wl, seqs, cases = build_cases(ptg, key, args.seed, rank, ws, args.split, 0, device)
    st = Stepper(ptg, cases, wl, args.streams, device)
    stats = workload_stats(wl, seqs, cases)
    steps = max(1, min(args.steps, 10))
    for _ in range(3):
        st.step()
    torch.cuda.synchronize()
    st.check_status("during warm-up of " + key)
    ms = st.timed(steps)
    st.check_status("in the timed steps of " + key)
    ms_mean = max_over_ranks(float(np.mean(ms)), ws)
    flops_all = sum_over_ranks(stats["flops"], ws)
    eff = flops_all / (ms_mean * 1e-3) / 1e12
    out = {
        "description": wl.description, "tries": len(cases), "steps": steps, "warmup": 3,
        "ms_per_step": round(ms_mean, 3), "visible_pairs": stats["pairs"],
        "packed_tokens": stats["tokens"],
        "tree_token_ratio": round(stats["tokens"] / stats["original"], 4),
        "flops_saved_vs_unpacked_causal": round(1 - stats["pairs"] / stats["causal_pairs"], 4),
        "effective_tflops": round(eff, 2),
        "frac_of_bf16_peak": round(eff / peaks["bf16"], 4),
        "packed_tokens_per_s": round(sum_over_ranks(stats["tokens"], ws) / (ms_mean * 1e-3), 1),
    }
    del st, cases
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, ws):
    import torch
    import prefix_tree_attention_gb300 as ptg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl, seqs, cases = build_cases(ptg, args.workload, args.seed, rank, ws, args.split,
                                  args.tries, device)
    st = Stepper(ptg, cases, wl, args.streams, device)
    stats = workload_stats(wl, seqs, cases)
    pairs, tokens, flops = stats["pairs"], stats["tokens"], stats["flops"]
    bwd_flops = BWD_FLOPS_PER_PAIR * wl.d * wl.Hq * pairs
    fwd_flops = FWD_FLOPS_PER_PAIR * wl.d * wl.Hq * pairs

    # ---- warm-up (also checks that nothing failed)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    st.check_status("during warm-up")
    # non-empty 128x128 tiles of every trie (blockmap word 1), read once here:
    # bwd main adds one 128 x d fp32 dQ tile per (non-empty tile, query head)
    nnz_tiles = sum(int(c.bufs.blockmap[1].item()) for c in cases)

    # ---- device-resident timed region
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches0 = ptg.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_ms = st.timed(args.steps)
    barrier(ws)
    launches = ptg.launch_count() - launches0
    st.check_status("in the timed steps")
    # per-kernel times: the same batch on one stream, every launch bracketed
    # by events on the stream it runs on
    roof_steps = max(1, min(args.steps, 2))
    serial = []
    for _ in range(roof_steps):
        evs = [[mk() for _ in range(4)] for _ in cases]
        st.serial_step(evs)
        serial.append(evs)
    torch.cuda.synchronize()
    fwd_ms = sum(ev[0].elapsed_time(ev[1]) for evs in serial for ev in evs) * args.steps / roof_steps
    bwd_main_ms = sum(ev[2].elapsed_time(ev[3]) for evs in serial for ev in evs) * args.steps / roof_steps
    ms_per_step = float(np.mean(step_ms))
    ms_max = max_over_ranks(ms_per_step, ws)
    flops_all = sum_over_ranks(flops, ws)
    value = flops_all / (ms_max * 1e-3) / 1e12
    tokens_all = sum_over_ranks(tokens, ws)

    # ---- roofline of the dominant kernel (bwd main) from the live events.
    # The one-stream pass takes well under a second, so the denominator is
    # the burst peak (a kernel timed on its own); the sustained figure is
    # reported beside it.
    peaks = measured_peaks()
    n_launch = len(cases) * args.steps
    bwd_achieved = bwd_flops * args.steps / (bwd_main_ms * 1e-3) / 1e12
    dq_bytes = float(nnz_tiles) * wl.Hq * 128 * wl.d * 4
    fwd_achieved = fwd_flops * args.steps / (fwd_ms * 1e-3) / 1e12
    traffic = recorded_traffic()
    roofline = {
        "kernel": "tree_attn_bwd_kernel (a5, bwd main)",
        "bound": "tensor", "achieved": round(bwd_achieved, 1),
        "peak": peaks["bf16"], "unit": "TFLOP/s",
        "frac": round(bwd_achieved / peaks["bf16"], 4),
        "peak_kind": f"bf16 dense, burst ({peaks['source']})",
        "frac_of_sustained": round(bwd_achieved / peaks["bf16_sustained"], 4),
        "traffic": None if traffic is None else traffic / len(cases),
        "avg_launch_ms": round(bwd_main_ms / n_launch, 4),
        "flops_per_launch": bwd_flops / len(cases),
        "fwd_achieved": round(fwd_achieved, 1),
        "fwd_frac": round(fwd_achieved / peaks["bf16"], 4),
        # the dQ accumulation: fp32 reduce-adds at L2, the step's other limit
        "dq_reduce": {
            "bytes_per_launch": dq_bytes / len(cases),
            "achieved_GBps": round(dq_bytes * args.steps / (bwd_main_ms * 1e-3) / 1e9, 1),
            "note": "bulk tensor reduce-adds of 32x32 fp32 boxes; a stand-alone "
                    "measurement on GB300 tops out at 4000-4400 GB/s",
        },
    }

    # ---- end to end through the API with host buffers
    e2e = None
    if not args.no_e2e:
        # one compute stream here: with the host copies in flight, a second
        # compute stream measured slower end to end
        e2e = run_e2e(ptg, cases, st.ws_bwds[:1], st.streams[:1], args, ws, flops_all)

    config = {
        "workload": args.workload + (f" (first {args.tries} tries)" if args.tries else ""),
        "description": wl.description,
        "tries": len(cases), "packed_tokens": tokens, "original_tokens": stats["original"],
        "tree_token_ratio": round(tokens / stats["original"], 4),
        "visible_pairs": pairs,
        "flops_saved_vs_unpacked_causal": round(1 - pairs / stats["causal_pairs"], 4),
        "heads": f"{wl.Hq}q/{wl.Hkv}kv", "head_dim": wl.d,
        "packed_tokens_per_s": round(tokens_all / (ms_max * 1e-3), 1),
        "frac_of_bf16_peak": round(value / peaks["bf16"], 4),
        "streams": st.n_streams,
        "fwd_ms_per_step_one_stream": round(fwd_ms / args.steps, 3),
        "bwd_main_ms_per_step_one_stream": round(bwd_main_ms / args.steps, 3),
        "l2": "inputs larger than L2 (no flush needed)",
        "parallelism": (f"balanced split of one batch x{ws}" if args.split == "balanced"
                        else f"replicas x{ws}"),
    }
    del st, cases
    torch.cuda.empty_cache()

    # ---- the metric's other Qwen3-8B-head workloads, timed the same way
    if not args.tries and not args.no_extra:
        per = {}
        for key in ("agent", "long", "fanout"):
            if key != args.workload:
                per[key] = run_extra_workload(ptg, key, args, rank, ws, device, peaks)
        config["per_workload"] = per

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 3),
        "higher_is_better": True,
        "scaling": "strong" if (args.split == "balanced" and ws > 1) else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, _dt, cores = oracle_sample(args.workload, args.seed, args.cpu_budget,
                                            tensors_fn=None)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_dta(args, rank, ws):
    """``--path dta``: attention forward + backward executed through the
    depth-first traversal of dynamic tree attention (AREAL-DTA 3.1-3.2), one
    ``tree_dta_attn`` call per trie with its schedule at ``--chunk`` tokens,
    against the packed step on the same batch in the same run.  One step =
    for every trie: positions, blockmap, then the schedule's ops.  Same
    metric as the packed path (effective TFLOP/s over visible pairs)."""
    import torch
    import prefix_tree_attention_gb300 as ptg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl, seqs, cases = build_cases(ptg, args.workload, args.seed, rank, ws, args.split,
                                  args.tries, device)
    stats = workload_stats(wl, seqs, cases)
    t_sched = time.perf_counter()
    scheds = [ptg.dta_schedule(c.tr.token_node, c.tr.node_entry, c.tr.node_exit, args.chunk)
              for c in cases]
    sched_s = time.perf_counter() - t_sched
    n_ops = sum(len(o) for o, _ in scheds)
    peak = max(pk for _, pk in scheds)
    ws_bytes = max(ptg.dta_attn_workspace_bytes(c.T, wl.Hq, wl.Hkv, wl.d) for c in cases)
    wsp = torch.empty((ws_bytes + 3) // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    def step():
        for c, (ops, _pk) in zip(cases, scheds):
            b = c.bufs
            ptg.tree_pack_positions(c.token_node, c.entry, c.exit, b.position_ids, b.key_reach,
                                    b.pos_ws, b.status)
            ptg.tree_blockmap_build(b.key_reach, b.blockmap, b.status)
            ptg.tree_dta_attn(c.q, c.k, c.v, c.do, b.key_reach, b.blockmap, ops, c.o, c.lse,
                              c.dq, c.dk, c.dv, wsp, b.status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bad = [int(c.bufs.status.item()) for c in cases]
    if any(bad):
        raise RuntimeError("device status " + ptg.status_string(max(bad)))
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches0 = ptg.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    per_step = []
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            s0, s1 = mk(), mk()
            s0.record(stream)
            step()
            s1.record(stream)
            per_step.append((s0, s1))
        torch.cuda.synchronize()
    barrier(ws)
    launches = ptg.launch_count() - launches0
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in per_step])), ws)
    # the packed step on the same tries, same run (one stream, as the DTA step)
    st = Stepper(ptg, cases, wl, 1, device)
    for _ in range(3):
        st.step()
    packed_ms = max_over_ranks(float(np.mean(st.timed(args.steps))), ws)
    st.check_status("in the packed comparison")
    flops_all = sum_over_ranks(stats["flops"], ws)
    peaks = measured_peaks()
    value = flops_all / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "strong" if (args.split == "balanced" and ws > 1) else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": args.workload + (f" (first {args.tries} tries)" if args.tries else ""),
            "path": "dta", "chunk": args.chunk, "tries": len(cases),
            "visible_pairs": stats["pairs"], "packed_tokens": stats["tokens"],
            "ops_per_step": n_ops, "peak_stack_tokens": peak,
            "largest_trie_tokens": max(c.T for c in cases),
            "schedule_host_ms": round(sched_s * 1e3, 2),
            "packed_ms_per_step_same_run": round(packed_ms, 3),
            "packed_tflops_same_run": round(flops_all / (packed_ms * 1e-3) / 1e12, 2),
            "dta_over_packed_time": round(ms / packed_ms, 4),
            "frac_of_bf16_peak": round(value / peaks["bf16"], 4),
            "l2": "inputs larger than L2 (no flush needed)",
        },
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


LOGPROB_METRIC = "tree log-prob/entropy gather of packed logits, packed tokens/s"
QWEN3_VOCAB = 151936


def run_logprob(args, rank, ws):
    """``--path logprob``: the tree-aware log-probability gather over one batch.

    One step = for every trie of the batch, tree_logprobs_entropy over that
    trie's rows of a bf16 logits buffer [T_pad, 151936] (row log-sum-exp and
    entropy, then each token's label log-probability), followed by the merge
    of log-probabilities and entropies into [n_seqs, max_len].  Positions and
    blockmap (a1, a2) are inputs here.  One 10 GB logits buffer, larger than
    L2, serves every trie (an LM head would write each micro-batch's logits
    into such a buffer).  The roofline is the row kernel against HBM: it must
    read the T_real x V logits once.
    """
    import torch
    import prefix_tree_attention_gb300 as ptg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl = W.WORKLOADS[args.workload]
    seqs, seed = rank_batch(ptg, args.workload, args.seed, rank, ws, args.split)
    tries = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)
    if args.tries:
        tries = tries[:args.tries]
    used = sorted({s for tr in tries for s in tr.seq_ids})
    remap = {s: i for i, s in enumerate(used)}
    for tr in tries:
        tr.seq_index = {remap[s]: v for s, v in tr.seq_index.items()}
    V = QWEN3_VOCAB
    t_max = max(tr.T_pad for tr in tries)
    logits = W.logits(t_max, V, seed=seed, device=device)
    offs = np.cumsum([0] + [tr.T_pad for tr in tries]).tolist()
    total = offs[-1]
    f32 = dict(dtype=torch.float32, device=device)
    lse_all, ent_all, lp_all = (torch.empty(total, **f32) for _ in range(3))
    cases = []
    for tr in tries:
        bufs = ptg.TrieBuffers(tr.T_pad, tr.n_nodes, 1, 64, device=device)
        tn = torch.from_numpy(tr.token_node).to(device)
        ptg.tree_pack_positions(tn, torch.from_numpy(tr.node_entry).to(device),
                                torch.from_numpy(tr.node_exit).to(device), bufs.position_ids,
                                bufs.key_reach, bufs.pos_ws, bufs.status)
        ptg.tree_blockmap_build(bufs.key_reach, bufs.blockmap, bufs.status)
        # the workload's fresh token ids run past the vocabulary: fold them in
        tok = np.where(tr.token_ids >= 0, tr.token_ids % V, -1).astype(np.int32)
        cases.append((tr, bufs, torch.from_numpy(tok).to(device)))
    pos, soffs = ptg.sequence_index_arrays(tries, len(used), offs[:-1])
    pos_d = torch.from_numpy(pos).to(device)
    soffs_d = torch.from_numpy(soffs).to(device)
    max_len = max(int(soffs[i + 1] - soffs[i]) for i in range(len(used))) - 1
    out_lp = torch.empty((len(used), max_len), **f32)
    out_ent = torch.empty_like(out_lp)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    tokens = sum(tr.n_tokens for tr in tries)

    def step():
        for i, (tr, bufs, tok) in enumerate(cases):
            sl = slice(offs[i], offs[i + 1])
            ptg.tree_logprobs_entropy(logits[:tr.T_pad], bufs.key_reach, lse_all[sl],
                                      bufs.status, token_ids=tok, blockmap=bufs.blockmap,
                                      entropy=ent_all[sl], logprob=lp_all[sl])
        ptg.tree_merge_per_sequence(lp_all, pos_d, soffs_d, out_lp, status, 1, 1, 0.0)
        ptg.tree_merge_per_sequence(ent_all, pos_d, soffs_d, out_ent, status, 0, 1, 0.0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bad = [int(b.status.item()) for _, b, _ in cases] + [int(status.item())]
    if any(bad):
        raise RuntimeError("device status " + ptg.status_string(max(bad)))
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches0 = ptg.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    per_step = []
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            s0, s1 = mk(), mk()
            s0.record(stream)
            step()
            s1.record(stream)
            per_step.append((s0, s1))
        torch.cuda.synchronize()
    barrier(ws)
    launches = ptg.launch_count() - launches0
    ms_per_step = float(np.mean([a.elapsed_time(b) for a, b in per_step]))
    ms_max = max_over_ranks(ms_per_step, ws)
    tokens_all = sum_over_ranks(tokens, ws)
    # the row kernel alone (no label pass): each launch bracketed by events
    row_ms = 0.0
    for tr, bufs, tok in cases:
        e0, e1 = mk(), mk()
        e0.record(stream)
        ptg.tree_logprobs_entropy(logits[:tr.T_pad], bufs.key_reach, lse_all[:tr.T_pad],
                                  bufs.status, entropy=ent_all[:tr.T_pad])
        e1.record(stream)
        torch.cuda.synchronize()
        row_ms += e0.elapsed_time(e1)
    row_bytes = sum(tr.n_tokens * (V * 2 + 8) + tr.T_pad * 4 for tr in tries)
    peaks = measured_peaks()
    backward = None if args.no_extra else logprob_backward(
        ptg, cases, offs, logits, lse_all, ent_all, pos_d, soffs_d, (len(used), max_len), V,
        tokens, seed, args, ws, peaks)
    per_row = recorded_logprob_traffic_per_row()
    achieved = row_bytes / (row_ms * 1e-3) / 1e9
    line = {
        "metric": LOGPROB_METRIC, "value": round(tokens_all / (ms_max * 1e-3), 1),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 3), "higher_is_better": True,
        "scaling": "strong" if (args.split == "balanced" and ws > 1) else "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": args.workload + (f" (first {args.tries} tries)" if args.tries else ""),
            "path": "logprob", "tries": len(tries), "packed_tokens": tokens,
            "sequences": len(used), "vocab": V, "logits": "bf16 sigma*N(0,1), sigma 2",
            "logits_gb_read_per_step": round(row_bytes / 1e9, 2),
            "l2": "logits larger than L2 (no flush needed)",
            "parallelism": (f"balanced split of one batch x{ws}" if args.split == "balanced"
                            else f"replicas x{ws}"),
        },
        "roofline": {
            "kernel": "k_row_stats (row log-sum-exp / entropy)", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peaks["hbm"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm"], 4),
            "peak_kind": f"HBM copy ({peaks['source']})",
            "traffic": (None if per_row is None
                        else round(per_row * tokens / len(cases), 1)),
            "traffic_note": "ncu DRAM bytes of a tiny-workload launch scaled by real rows",
            "avg_launch_ms": round(row_ms / len(cases), 4),
            "bytes_per_launch": row_bytes / len(cases),
        },
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None,
        "backward": backward,
    }
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc = logprob_oracle_rate(min(args.cpu_budget, 10.0), seed)
        line["cpu_baseline"] = {"value": round(rate, 2), "unit": "tokens/s", "cores": 1,
                                "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)


def logprob_backward(ptg, cases, offs, logits, lse_all, ent_all, pos_d, soffs_d, merged_shape,
                     V, tokens, seed, args, ws, peaks):
    """The gather's gradient over the same batch, timed apart from the
    forward: per-sequence gradients of log-probabilities and entropies
    ([n_seqs, max_len], fp32 N(0, 1)) go back through the two merge adjoints
    (tree_merge_per_sequence_bwd) to packed per-token / per-row gradients,
    then tree_logprobs_entropy_bwd writes the bf16 logits gradient of every
    trie, reading its logits once more.  Returns the ``backward`` object of
    the log-prob line: its own rate and the row kernel's HBM roofline."""
    import torch
    device = logits.device
    g = torch.Generator(device=device)
    g.manual_seed(1000 + seed)
    g_lp = torch.randn(merged_shape, generator=g, device=device, dtype=torch.float32)
    g_ent = torch.randn(merged_shape, generator=g, device=device, dtype=torch.float32)
    total = offs[-1]
    tok_g = torch.empty(total, dtype=torch.float32, device=device)
    row_g = torch.empty_like(tok_g)
    grad = torch.empty_like(logits)            # one gradient buffer, like the logits
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()

    def rows(i, tr, bufs, tok):
        sl = slice(offs[i], offs[i + 1])
        ptg.tree_logprobs_entropy_bwd(logits[:tr.T_pad], bufs.key_reach, lse_all[sl],
                                      grad[:tr.T_pad], bufs.status, token_ids=tok,
                                      entropy=ent_all[sl], grad_logprob=tok_g[sl],
                                      grad_entropy=row_g[sl])

    def step():
        tok_g.zero_()
        row_g.zero_()
        ptg.tree_merge_per_sequence_bwd(g_lp, pos_d, soffs_d, tok_g, status, 1, 1)
        ptg.tree_merge_per_sequence_bwd(g_ent, pos_d, soffs_d, row_g, status, 0, 1)
        for i, (tr, bufs, tok) in enumerate(cases):
            rows(i, tr, bufs, tok)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bad = [int(b.status.item()) for _, b, _ in cases] + [int(status.item())]
    if any(bad):
        raise RuntimeError("device status " + ptg.status_string(max(bad)))
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches0 = ptg.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    per_step = []
    for _ in range(args.steps):
        s0, s1 = mk(), mk()
        s0.record(stream)
        step()
        s1.record(stream)
        per_step.append((s0, s1))
    torch.cuda.synchronize()
    barrier(ws)
    launches = ptg.launch_count() - launches0
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in per_step])), ws)
    # the row kernel alone, each launch bracketed by events
    row_ms = 0.0
    for i, (tr, bufs, tok) in enumerate(cases):
        e0, e1 = mk(), mk()
        e0.record(stream)
        rows(i, tr, bufs, tok)
        e1.record(stream)
        torch.cuda.synchronize()
        row_ms += e0.elapsed_time(e1)
    # per real row: V logits read, V gradients written (bf16), lse, entropy,
    # reach, the row's entropy gradient, its children's gradients; a pad row
    # writes its V zeros
    bwd_bytes = sum(tr.n_tokens * (V * 4 + 24) + (tr.T_pad - tr.n_tokens) * (V * 2 + 4)
                    for tr, _, _ in cases)
    achieved = bwd_bytes / (row_ms * 1e-3) / 1e9
    per_row = recorded_logprob_traffic_per_row(LOGPROB_BWD_TRAFFIC)
    real_rows = sum(tr.n_tokens for tr, _, _ in cases)
    return {
        "what": "merge adjoints (log-prob, entropy) + logits gradient of every trie",
        "ms_per_step": round(ms, 3),
        "tokens_per_s": round(sum_over_ranks(tokens, ws) / (ms * 1e-3), 1),
        "gpu_launches": launches,
        "roofline": {
            "kernel": "k_row_bwd (logits gradient)", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peaks["hbm"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm"], 4),
            "peak_kind": f"HBM copy ({peaks['source']})",
            "traffic": (None if per_row is None
                        else round(per_row * real_rows / len(cases), 1)),
            "traffic_note": "ncu DRAM bytes of a tiny-workload launch scaled by real rows",
            "avg_launch_ms": round(row_ms / len(cases), 4),
            "bytes_per_launch": bwd_bytes / len(cases),
        },
    }


LMHEAD_METRIC = "LM head fused with the tree log-prob gather, packed tokens/s"
QWEN3_HIDDEN = 4096


def lmhead_oracle_child(budget_s: float, seed: int, rows: int, H: int, V: int, v_slice: int):
    """Body of the oracle timing for ``--path lmhead`` (run in a child process
    whose BLAS is limited to one thread): per pass, the LM-head logits of
    ``rows`` token rows against a ``v_slice``-row slice of the weights in
    fp64 (``oracle.logprob.lm_head_logits``), then each row's statistics and
    log-softmax over the slice; rows per second are scaled by v_slice / V to
    the whole vocabulary.  Prints one JSON object."""
    from oracle import logprob as OL
    hidden, weight = W.lm_head(rows, H, v_slice, seed=seed)
    h = hidden.float().numpy().astype(np.float64)
    w = weight.float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    passes = 0
    while True:
        x = OL.lm_head_logits(h, w)
        for r in range(rows):
            OL.row_stats(x[r])
            OL.log_softmax(x[r])
        passes += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    rate = passes * rows / dt * v_slice / V
    print(json.dumps({"rate": rate, "sample": (
        f"{passes} passes of {rows} rows x H={H} against a {v_slice}-row vocabulary slice "
        f"(fp64 numpy LM-head logits + row stats + log-softmax, one BLAS thread), "
        f"scaled to V={V}")}))


def lmhead_oracle_rate(budget_s: float, seed: int, rows: int = 16, H: int = QWEN3_HIDDEN,
                       V: int = QWEN3_VOCAB, v_slice: int = 16384):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import bench; bench.lmhead_oracle_child(%r, %d, %d, %d, %d, %d)"
            % (budget_s, seed, rows, H, V, v_slice))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed: " + r.stderr[-2000:])
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    return rec["rate"], rec["sample"]


def lmhead_backward(ptg, cases, offs, hidden, weight, lse_all, ent_all, pos_d, soffs_d,
                    merged_shape, tokens, flops, seed, args, ws, peaks):
    """The fused gather's gradient with respect to the logits over the same
    batch: per-sequence gradients of log-probabilities and entropies
    ([n_seqs, max_len], fp32 N(0, 1)) through the two merge adjoints, then
    tree_lm_head_logits_grad over every trie's rows as one chunk into one bf16
    [T_pad, V] buffer (the logits tiles recomputed in TMEM).  The LM head's own
    gradients (two plain GEMMs of that buffer) are the model's and not timed."""
    import torch
    device = hidden.device
    g = torch.Generator(device=device)
    g.manual_seed(2000 + seed)
    g_lp = torch.randn(merged_shape, generator=g, device=device, dtype=torch.float32)
    g_ent = torch.randn(merged_shape, generator=g, device=device, dtype=torch.float32)
    tok_g = torch.empty(offs[-1], dtype=torch.float32, device=device)
    row_g = torch.empty_like(tok_g)
    t_max = hidden.shape[0]
    V = weight.shape[0]
    grad = torch.empty((t_max, (V + 7) // 8 * 8), dtype=torch.bfloat16, device=device)[:, :V]
    gws = torch.empty(ptg.lm_head_grad_workspace_bytes(t_max) // 4, dtype=torch.float32,
                      device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()

    def rows(i, tr, bufs, tok):
        sl = slice(offs[i], offs[i + 1])
        ptg.tree_lm_head_logits_grad(hidden[:tr.T_pad], weight, bufs.key_reach, lse_all[sl],
                                     grad[:tr.T_pad], gws, bufs.status, 0, tr.T_pad,
                                     token_ids=tok, entropy=ent_all[sl], grad_logprob=tok_g[sl],
                                     grad_entropy=row_g[sl])

    def step():
        tok_g.zero_()
        row_g.zero_()
        ptg.tree_merge_per_sequence_bwd(g_lp, pos_d, soffs_d, tok_g, status, 1, 1)
        ptg.tree_merge_per_sequence_bwd(g_ent, pos_d, soffs_d, row_g, status, 0, 1)
        for i, (tr, bufs, tok) in enumerate(cases):
            rows(i, tr, bufs, tok)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bad = [int(b.status.item()) for _, b, _ in cases] + [int(status.item())]
    if any(bad):
        raise RuntimeError("device status " + ptg.status_string(max(bad)))
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches0 = ptg.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    per_step = []
    for _ in range(args.steps):
        s0, s1 = mk(), mk()
        s0.record(stream)
        step()
        s1.record(stream)
        per_step.append((s0, s1))
    torch.cuda.synchronize()
    barrier(ws)
    launches = ptg.launch_count() - launches0
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in per_step])), ws)
    call_ms = 0.0
    for i, (tr, bufs, tok) in enumerate(cases):
        e0, e1 = mk(), mk()
        e0.record(stream)
        rows(i, tr, bufs, tok)
        e1.record(stream)
        torch.cuda.synchronize()
        call_ms += e0.elapsed_time(e1)
    achieved = flops / (call_ms * 1e-3) / 1e12
    return {
        "what": "merge adjoints + logits gradient of every trie (logits recomputed in TMEM)",
        "ms_per_step": round(ms, 3),
        "tokens_per_s": round(sum_over_ranks(tokens, ws) / (ms * 1e-3), 1),
        "gpu_launches": launches,
        "grad_gb_written_per_step": round(sum(tr.T_pad for tr, _, _ in cases) * V * 2 / 1e9, 2),
        "roofline": {
            "kernel": "k_lmh_gemm<true> (LM-head GEMM + logits-gradient epilogue) with its "
                      "coefficient and one-hot passes",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16"], 4),
            "peak_kind": f"bf16 dense, burst ({peaks['source']})",
            "frac_of_sustained": round(achieved / peaks["bf16_sustained"], 4),
            "traffic": None, "avg_launch_ms": round(call_ms / len(cases), 4),
            "flops_per_launch": flops / len(cases),
        },
    }


def run_lmhead(args, rank, ws):
    """``--path lmhead``: the LM head fused with the log-prob gather.

    One step = for every trie of the batch, tree_lm_head_logprobs_entropy
    over that trie's rows: Qwen3-8B's LM head (hidden size 4096, vocabulary
    151,936, bf16 hidden states [T_pad, 4096] and weights [151936, 4096],
    synthetic N(0, 1) and N(0, (2/64)^2)) with the row log-sum-exp and
    entropy in the GEMM's epilogue and each token's label log-probability;
    then the merge of log-probabilities and entropies into [n_seqs, max_len].
    Positions and blockmap (a1, a2) are inputs here.  No logits buffer
    exists.  The roofline is the call's GEMM against the bf16 tensor peak:
    2 * real rows * V * H flops per trie."""
    import torch
    import prefix_tree_attention_gb300 as ptg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl = W.WORKLOADS[args.workload]
    seqs, seed = rank_batch(ptg, args.workload, args.seed, rank, ws, args.split)
    tries = ptg.pack_sequences(seqs, wl.max_tokens_per_mb)
    if args.tries:
        tries = tries[:args.tries]
    used = sorted({s for tr in tries for s in tr.seq_ids})
    remap = {s: i for i, s in enumerate(used)}
    for tr in tries:
        tr.seq_index = {remap[s]: v for s, v in tr.seq_index.items()}
    V, H = QWEN3_VOCAB, QWEN3_HIDDEN
    t_max = max(tr.T_pad for tr in tries)
    hidden, weight = W.lm_head(t_max, H, V, seed=seed, device=device)
    offs = np.cumsum([0] + [tr.T_pad for tr in tries]).tolist()
    total = offs[-1]
    f32 = dict(dtype=torch.float32, device=device)
    lse_all, ent_all, lp_all = (torch.empty(total, **f32) for _ in range(3))
    ws_buf = torch.empty(ptg.lm_head_workspace_bytes(t_max, V) // 4, **f32)
    cases = []
    for tr in tries:
        bufs = ptg.TrieBuffers(tr.T_pad, tr.n_nodes, 1, 64, device=device)
        ptg.tree_pack_positions(torch.from_numpy(tr.token_node).to(device),
                                torch.from_numpy(tr.node_entry).to(device),
                                torch.from_numpy(tr.node_exit).to(device), bufs.position_ids,
                                bufs.key_reach, bufs.pos_ws, bufs.status)
        ptg.tree_blockmap_build(bufs.key_reach, bufs.blockmap, bufs.status)
        tok = np.where(tr.token_ids >= 0, tr.token_ids % V, -1).astype(np.int32)
        cases.append((tr, bufs, torch.from_numpy(tok).to(device)))
    pos, soffs = ptg.sequence_index_arrays(tries, len(used), offs[:-1])
    pos_d = torch.from_numpy(pos).to(device)
    soffs_d = torch.from_numpy(soffs).to(device)
    max_len = max(int(soffs[i + 1] - soffs[i]) for i in range(len(used))) - 1
    out_lp = torch.empty((len(used), max_len), **f32)
    out_ent = torch.empty_like(out_lp)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    tokens = sum(tr.n_tokens for tr in tries)

    def call(i, tr, bufs, tok, labels=True):
        sl = slice(offs[i], offs[i + 1])
        ptg.tree_lm_head_logprobs_entropy(
            hidden[:tr.T_pad], weight, bufs.key_reach, lse_all[sl], ws_buf, bufs.status,
            token_ids=tok, blockmap=bufs.blockmap, entropy=ent_all[sl],
            logprob=lp_all[sl] if labels else None)

    def step():
        for i, (tr, bufs, tok) in enumerate(cases):
            call(i, tr, bufs, tok)
        ptg.tree_merge_per_sequence(lp_all, pos_d, soffs_d, out_lp, status, 1, 1, 0.0)
        ptg.tree_merge_per_sequence(ent_all, pos_d, soffs_d, out_ent, status, 0, 1, 0.0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bad = [int(b.status.item()) for _, b, _ in cases] + [int(status.item())]
    if any(bad):
        raise RuntimeError("device status " + ptg.status_string(max(bad)))
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    launches0 = ptg.launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    per_step = []
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            s0, s1 = mk(), mk()
            s0.record(stream)
            step()
            s1.record(stream)
            per_step.append((s0, s1))
        torch.cuda.synchronize()
    barrier(ws)
    launches = ptg.launch_count() - launches0
    ms_per_step = float(np.mean([a.elapsed_time(b) for a, b in per_step]))
    ms_max = max_over_ranks(ms_per_step, ws)
    tokens_all = sum_over_ranks(tokens, ws)
    # the GEMM with its statistics epilogue and the partials' combine, each
    # call bracketed by events (the label pass left out)
    gemm_ms = 0.0
    for i, (tr, bufs, tok) in enumerate(cases):
        e0, e1 = mk(), mk()
        e0.record(stream)
        call(i, tr, bufs, tok, labels=False)
        e1.record(stream)
        torch.cuda.synchronize()
        gemm_ms += e0.elapsed_time(e1)
    flops = sum(2.0 * tr.n_tokens * V * H for tr in tries)
    peaks = measured_peaks()
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    step_tflops = sum_over_ranks(flops, ws) / (ms_max * 1e-3) / 1e12
    backward = None if args.no_extra else lmhead_backward(
        ptg, cases, offs, hidden, weight, lse_all, ent_all, pos_d, soffs_d,
        (len(used), max_len), tokens, flops, seed, args, ws, peaks)
    line = {
        "metric": LMHEAD_METRIC, "value": round(tokens_all / (ms_max * 1e-3), 1),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 3), "higher_is_better": True,
        "scaling": "strong" if (args.split == "balanced" and ws > 1) else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": args.workload + (f" (first {args.tries} tries)" if args.tries else ""),
            "path": "lmhead", "tries": len(tries), "packed_tokens": tokens,
            "sequences": len(used), "hidden": H, "vocab": V,
            "inputs": "bf16 hidden N(0,1) [T_pad, 4096], weight N(0,(2/64)^2) [151936, 4096]",
            "step_tflops": round(step_tflops, 1),
            "l2": "weights (1.24 GB) larger than L2 (no flush needed)",
            "parallelism": (f"balanced split of one batch x{ws}" if args.split == "balanced"
                            else f"replicas x{ws}"),
        },
        "roofline": {
            "kernel": "k_lmh_gemm<false> (LM-head GEMM + row statistics) with k_lmh_combine",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16"],
            "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16"], 4),
            "peak_kind": f"bf16 dense, burst ({peaks['source']})",
            "frac_of_sustained": round(achieved / peaks["bf16_sustained"], 4),
            "traffic": None, "avg_launch_ms": round(gemm_ms / len(cases), 4),
            "flops_per_launch": flops / len(cases),
        },
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None,
        "backward": backward,
    }
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc = lmhead_oracle_rate(min(args.cpu_budget, 15.0), seed)
        line["cpu_baseline"] = {"value": round(rate, 3), "unit": "tokens/s", "cores": 1,
                                "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(ptg, cases, ws_bwds, streams, args, ws, flops_all):
    """Same metric, each step copying its inputs host->device from pinned
    memory and its outputs (O, dQ, dK, dV) device->host, through the same
    API calls; copies overlap compute on their own streams.  The tries
    alternate over the given compute streams."""
    import torch
    # Pinned host copies of every input and output.  Keep them well inside the
    # host's available memory: if the whole batch does not fit in 40% of it,
    # run the e2e leg on the leading tries that do and report that.
    need = [sum(t.numel() * t.element_size() for t in c.input_tensors() + c.output_tensors())
            for c in cases]
    avail = _mem_available_bytes()
    budget = 0.4 * avail if avail else float(sum(need))
    n_fit, acc = 0, 0
    for b in need:
        if acc + b > budget:
            break
        acc += b
        n_fit += 1
    if n_fit == 0:
        return {"value": None, "unit": UNIT, "skipped": "host memory too small for pinned buffers"}
    subset = n_fit < len(cases)
    cases = cases[:n_fit]
    if subset:
        flops_all = sum_over_ranks(
            (FWD_FLOPS_PER_PAIR + BWD_FLOPS_PER_PAIR) * cases[0].d * cases[0].Hq *
            sum(c.pairs for c in cases), ws)
    slab_in = _PinnedSlab(sum(_padded(t) for c in cases for t in c.input_tensors()))
    slab_out = _PinnedSlab(sum(_padded(t) for c in cases for t in c.output_tensors()))
    host_in = [[slab_in.take(t) for t in c.input_tensors()] for c in cases]
    for c, hs in zip(cases, host_in):
        for dst, src in zip(hs, c.input_tensors()):
            dst.copy_(src)
    host_out = [[slab_out.take(t) for t in c.output_tensors()] for c in cases]
    h2d = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
    d2h = sum(t.numel() * t.element_size() for hs in host_out for t in hs)
    copy_in = torch.cuda.Stream()
    copy_out = torch.cuda.Stream()

    n_streams = len(streams)
    # Per-trie events of the previous step: trie i's uploads may start once
    # its previous compute has consumed the inputs, and its compute once its
    # previous outputs are downloaded, so consecutive steps pipeline on the
    # host link instead of draining at every step boundary.
    prev_compute = [None] * len(cases)
    prev_download = [None] * len(cases)

    def e2e_step():
        ready = []
        for i, c in enumerate(cases):
            if prev_compute[i] is not None:
                copy_in.wait_event(prev_compute[i])
            with torch.cuda.stream(copy_in):
                for dst, src in zip(c.input_tensors(), host_in[i]):
                    dst.copy_(src, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_in)
            ready.append(ev)
        for i, c in enumerate(cases):
            st = streams[i % n_streams]
            st.wait_event(ready[i])
            if prev_download[i] is not None:
                st.wait_event(prev_download[i])
            with torch.cuda.stream(st):
                run_path(ptg, c, ws_bwds[i % n_streams], st)
                ev = torch.cuda.Event()
                ev.record(st)
            prev_compute[i] = ev
            copy_out.wait_event(ev)
            with torch.cuda.stream(copy_out):
                for dst, src in zip(host_out[i], c.output_tensors()):
                    dst.copy_(src, non_blocking=True)
                dev = torch.cuda.Event()
                dev.record(copy_out)
            prev_download[i] = dev

    for _ in range(max(1, min(args.warmup, 2))):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / args.steps
    dt = max_over_ranks(dt, ws)

    # The host link on its own, in the same run: the same pinned copies (both
    # directions at once, on the same copy streams) with no compute.
    def copies_only():
        with torch.cuda.stream(copy_in):
            for i, c in enumerate(cases):
                for dst, src in zip(c.input_tensors(), host_in[i]):
                    dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(copy_out):
            for i, c in enumerate(cases):
                for dst, src in zip(host_out[i], c.output_tensors()):
                    dst.copy_(src, non_blocking=True)

    def one_way(h2d_dir):
        stream = copy_in if h2d_dir else copy_out
        with torch.cuda.stream(stream):
            for i, c in enumerate(cases):
                pairs_ = (zip(c.input_tensors(), host_in[i]) if h2d_dir
                          else zip(host_out[i], c.output_tensors()))
                for dst, src in pairs_:
                    dst.copy_(src, non_blocking=True)

    def wall(fn, n):
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t) / n

    n_copy = max(1, min(args.steps, 3))
    both_s = wall(copies_only, n_copy)
    h2d_s = wall(lambda: one_way(True), n_copy)
    d2h_s = wall(lambda: one_way(False), n_copy)
    rec = {"value": round(flops_all / dt / 1e12, 2), "unit": UNIT,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "ms_per_step": round(dt * 1e3, 3),
           "e2e_gbs_per_direction": {"h2d": round(h2d / dt / 1e9, 2),
                                     "d2h": round(d2h / dt / 1e9, 2)},
           "host_link_gbs": {"h2d_alone": round(h2d / h2d_s / 1e9, 2),
                             "d2h_alone": round(d2h / d2h_s / 1e9, 2),
                             "both_at_once_ms": round(both_s * 1e3, 3)},
           # share of the e2e step that the same copies need with no compute:
           # near 1 means the end-to-end number is set by the host link
           "copy_frac": round(both_s / dt, 4),
           "timing": "host wall clock around the steps, synchronised at both ends",
           "copies": "pinned host -> device inputs (token_node, entry, exit, q, k, v, do); "
                     "device -> pinned host outputs (o, dq, dk, dv); copy streams overlap compute, "
                     "consecutive steps chained per trie",
           "route": "the Python binding's ctypes calls of the C ABI, torch doing the copies"}
    rec["host_buffers"] = ("one exact-size page-locked slab per direction "
                           f"({slab_in.kind}; {round(slab_in.nbytes / 1e9, 2)} GB in, "
                           f"{round(slab_out.nbytes / 1e9, 2)} GB out)")
    if subset:
        rec["tries"] = f"first {len(cases)} tries (pinned buffers limited to 40% of host memory)"
    del host_in, host_out
    slab_in.close()
    slab_out.close()
    return rec


def _padded(t) -> int:
    return (t.numel() * t.element_size() + 255) // 256 * 256


class _PinnedSlab:
    """One exact-size page-locked host buffer, handed out as tensors.

    An anonymous mapping registered with cudaHostRegister: the pinned
    footprint is the bytes the step moves (torch's pinned-memory allocator
    rounds every allocation up to a power of two, which nearly doubles the
    footprint of this leg, and a large pinned footprint slows the host link
    on these machines).  Falls back to one torch pinned tensor if
    registration is refused."""

    def __init__(self, nbytes: int):
        import mmap
        import torch
        self.nbytes = max(int(nbytes), 256)
        self.off = 0
        self._mm = mmap.mmap(-1, self.nbytes)
        self._np = np.frombuffer(self._mm, dtype=np.uint8)
        self.base = torch.from_numpy(self._np)
        self._ptr = self.base.data_ptr()
        rt = torch.cuda.cudart()
        self.registered = rt.cudaHostRegister(self._ptr, self.nbytes, 0) == rt.cudaError.success
        self.kind = "anonymous mapping + cudaHostRegister"
        if not self.registered:
            self.base = torch.empty(self.nbytes, dtype=torch.uint8, pin_memory=True)
            self.kind = "torch pinned tensor"

    def take(self, like):
        import torch
        n = like.numel() * like.element_size()
        view = self.base[self.off:self.off + n]
        self.off += _padded(like)
        return view.view(like.dtype).view(like.shape) if n else torch.empty(
            like.shape, dtype=like.dtype)

    def close(self):
        import torch
        if self.registered:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaHostUnregister(self._ptr)
            self.registered = False


def _mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="grpo", choices=sorted(W.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tries", type=int, default=0,
                    help="use only the first N tries of the batch (small profiling cases)")
    ap.add_argument("--split", choices=["replicas", "balanced"], default="replicas",
                    help="N > 1: independent batch per rank, or one batch split by the "
                         "load-balanced partitioner")
    ap.add_argument("--streams", type=int, default=2,
                    help="CUDA streams the independent tries of a batch alternate over")
    ap.add_argument("--path", choices=["attention", "logprob", "dta", "lmhead"],
                    default="attention",
                    help="attention: the fwd+bwd step (default); logprob: the tree-aware "
                         "log-prob / entropy gather over packed logits; dta: the same "
                         "attention executed through the depth-first traversal schedule; "
                         "lmhead: the LM head fused with the gather (no logits buffer)")
    ap.add_argument("--chunk", type=int, default=2048,
                    help="--path dta: chunk length of the traversal schedule")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the timed agent / long / fanout entries of config.per_workload "
                         "and the backward objects of the log-prob and lmhead lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, ws = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, ws)
    elif args.path == "logprob":
        run_logprob(args, rank, ws)
    elif args.path == "dta":
        run_dta(args, rank, ws)
    elif args.path == "lmhead":
        run_lmhead(args, rank, ws)
    else:
        run_ours(args, rank, ws)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
