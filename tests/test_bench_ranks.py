"""Host side of bench.py on CPU (no GPU): multi-rank runs with two gloo ranks, and
the FLOP accounting.

The path shards with no exchange (every (batch, head) slice is independent), so a
run on N GPUs is N replicas: bench.py times each rank, takes the slowest rank's
time and counts all ranks' work.  These tests run that reduction across two real
processes, and the reference arm under torchrun (rank 0 alone prints its line)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 7.5 * rank  # rank 1 is the slower one
        worst = bench.max_over_ranks(ms, "cpu")
        value = bench.whole_job_tflops(1.0e12, 4, world, worst)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"worst": worst, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [g["worst"] for g in got] == [17.5, 17.5]
    # 2 ranks x 4 steps x 1e12 FLOP in 17.5 ms
    assert all(g["value"] == pytest.approx(8.0e12 / 17.5e-3 / 1e12) for g in got)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_tflops(2.0e12, 10, 1, 20.0) == pytest.approx(1000.0)


def test_reference_arm_prints_once_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--reference-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_executed_flops_exceed_the_algorithmic_count_by_the_diagonal_blocks():
    from exact_causal_attention_gb300 import inputs

    w = inputs.WORKLOADS["causal_b1_h32_n8192_d128_fp16"]
    assert bench.executed_flops(w) == pytest.approx(w.flops * 65 / 64)  # (n + 1) / n with n = 64 tiles
    nc = w.with_causal(False)
    assert bench.executed_flops(nc) == pytest.approx(nc.flops)  # no diagonal: every block is full work


def test_clock_normalised_rate():
    import bench

    # 152 SMs at 2070 MHz retire 8192 * 152 * 2.07e9 FLOP/s = 2577.4 TFLOP/s of dense fp16 MMA work.
    r = bench.clock_normalised(1700.0, {"sm_mhz": 2070.0}, 152)
    assert r["clock_rate_tensor_peak_tflops"] == pytest.approx(2577.4, rel=1e-4)
    assert r["frac_of_clock_rate_peak"] == pytest.approx(1700.0 / 2577.4, rel=1e-4)
    assert r["tflops_per_ghz"] == pytest.approx(1700.0 / 2.07)
    assert bench.clock_normalised(1700.0, {"sm_mhz": None}, 152) is None
    assert bench.clock_normalised(1700.0, None, 152) is None


def test_traffic_record_matches_the_kernel_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu record only while the attention
    kernel's sources hash to the value the record was captured with; a record of other
    sources or another workload reads as null."""
    rec = open(os.path.join(bench.PROFILES, "attn_fwd_n8192_traffic.txt")).read()
    recorded = int(rec.split("dram_bytes_per_launch:")[1].split()[0])
    if f"kernel_source_sha256_16: {bench.kernel_source_hash()}" in rec:
        assert bench.recorded_traffic() == recorded
    else:  # the kernel changed since the capture: no traffic until it is re-captured
        assert bench.recorded_traffic() is None
    stale = tmp_path / "profiles"
    stale.mkdir()
    (stale / "attn_fwd_n8192_traffic.txt").write_text(rec.replace(bench.kernel_source_hash(), "0" * 16))
    monkeypatch.setattr(bench, "PROFILES", str(stale))
    assert bench.recorded_traffic() is None
    (stale / "attn_fwd_n8192_traffic.txt").write_text(rec.replace(bench.WORKLOAD, "another_workload"))
    assert bench.recorded_traffic() is None
