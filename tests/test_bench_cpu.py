"""Host-side logic of bench.py (CPU only): the reference arm's JSON line, the
rank reductions of the N > 1 path over gloo (world size 2), and the
clock-sample summary."""
import contextlib
import io
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "tiny"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] == bench.METRIC and rec["unit"] == "TFLOP/s"
    assert rec["higher_is_better"] is True
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    assert rec["config"]["workload"] == "tiny"


def test_reference_arm_logprob_path():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--path", "logprob", "--steps", "1", "--warmup", "0",
                    "--cpu-budget", "0.5"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["metric"] == bench.LOGPROB_METRIC
    assert rec["unit"] == "tokens/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["config"]["path"] == "logprob"


def test_reference_arm_lmhead_path():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--path", "lmhead", "--steps", "1", "--warmup", "0",
                    "--cpu-budget", "0.5"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["metric"] == bench.LMHEAD_METRIC
    assert rec["value"] > 0 and rec["cpu_baseline"]["cores"] == 1
    assert rec["config"]["path"] == "lmhead" and rec["config"]["hidden"] == 4096


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    mx = bench.max_over_ranks(10.0 + rank, 2)
    sm = bench.sum_over_ranks(1.5 * (rank + 1), 2)
    bench.barrier(2)
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_rank_reductions_world_size_two():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == (11.0, 4.5) and out[1] == (11.0, 4.5)


def test_clock_summary_parses_samples():
    c = bench.ClockSampler(0)
    c.samples = [["0", "1900", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active",
                  "Active"],
                 ["0", "1950", "2070", "950", "0x0", "Not Active", "Not Active", "Not Active",
                  "Not Active"]]
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1925.0)
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_recorded_traffic_is_null_when_source_changed(tmp_path, monkeypatch):
    rec = {"kernel_source_sha256_16": "0" * 16, "dram_bytes_per_step": 123}
    p = tmp_path / "t.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(p))
    assert bench.recorded_traffic() is None
    rec["kernel_source_sha256_16"] = bench.source_hash(bench.KERNEL_SOURCE)
    p.write_text(json.dumps(rec))
    assert bench.recorded_traffic() == 123


def _split_worker(rank, port, out):
    import prefix_tree_attention_gb300 as ptg
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    seqs, _seed = bench.rank_batch(ptg, "agent", 0, rank, 2, "balanced")
    mine = [tuple(x) for x in seqs]
    gathered = [None, None]
    dist.all_gather_object(gathered, mine)
    out[rank] = gathered
    dist.destroy_process_group()


def test_balanced_split_world_size_two_covers_the_batch_once():
    import workloads as W
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_split_worker, args=(port, out), nprocs=2, start_method="spawn",
                       join=True)
    a, b = out[0]
    assert out[1] == [a, b]
    batch = [tuple(x) for x in W.sequences("agent", 0)]
    assert sorted(a + b) == sorted(batch) and a and b
    # contiguous halves of the DFS (lexicographic) order
    assert max(a) < min(b)


def test_replicas_split_gives_each_rank_its_own_batch():
    import prefix_tree_attention_gb300 as ptg
    import workloads as W
    s0, seed0 = bench.rank_batch(ptg, "tiny", 0, 0, 2, "replicas")
    s1, seed1 = bench.rank_batch(ptg, "tiny", 0, 1, 2, "replicas")
    assert s0 == W.sequences("tiny", 0) and s1 == W.sequences("tiny", 1) and seed1 == seed0 + 1
