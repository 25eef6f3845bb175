"""Benchmark: causal attention forward TFLOP/s (2BHN^2D) on one GB300 per rank.

Workload: causal fp16, B=1, H=32, N=8192, D=128 (the long end of the N = 512..8192
sweep of "CUDA FlashAttention：从在线 Softmax 到长序列 IO 极限", section 8), inputs
synthetic N(0, 1) from seed 3.  One step = one attn_fwd call over the whole batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  `value` is device time (CUDA events on the
launching stream, L2 flushed between steps); `e2e` is the same metric through the
C ABI with pinned host buffers, copies in and out included.  The reference arm
(--impl reference) is the FP64 CPU oracle on the host cores, timed on a bounded
sample of query rows of the same workload.
Multi-GPU runs are independent replicas (every (batch, head) slice is
independent; there is no exchange step): value = all ranks' FLOPs / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal attn fwd TFLOP/s (2BHN^2D) at N=512..8192, % of GB300 dense FP16 peak"
WORKLOAD = "causal_b1_h32_n8192_d128_fp16"
# The page's own number for this workload (PyTorch SDPA FLASH backend, RTX 3060 Laptop, SM86):
# 25.854 ms at B=1, H=32, N=8192, D=128 causal fp16 -> 2BHN^2D / t.
PAGE_MS_N8192 = 25.854
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2
# NVIDIA's published dense FP16/BF16 tensor rate for this part: the HGX B300 specification
# gives 36 PFLOPS FP16/BF16 per 8 GPUs with 2:4 sparsity, i.e. 2.25 PFLOP/s dense per GPU.
DATASHEET_DENSE_FP16_TFLOPS = 2250.0
DATASHEET_SOURCE = "NVIDIA HGX B300 specification: FP16/BF16 tensor 36 PFLOPS per 8 GPUs with sparsity -> 2.25 dense per GPU"
# Dense fp16 MMA work one SM retires per clock (a 128x128x16 tcgen05.mma every 64 cycles),
# consistent with the ncu capture of the attention kernel (tensor pipe 77.1% active at
# 1.781 GHz while executing 1.71 PFLOP/s over 152 SMs).
MMA_FLOP_PER_CLK_PER_SM = 8192
PROFILES = os.path.join(ROOT, "profiles")


def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest x over the ranks of the default process group (x itself without one)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Every rank runs the same workload (independent replicas): all ranks' work over the
    slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


def executed_flops(w) -> float:
    """MMA FLOPs the kernel executes: every 128 x 128 (query tile, key tile) block it visits,
    the diagonal and ragged blocks counted in full (Q K^T and P V, 2 * 128 * 128 * D each)."""
    n = -(-w.N // 128)
    blocks = n * (n + 1) // 2 if w.causal else n * n
    return 4.0 * 128 * 128 * w.D * w.B * w.H * blocks


def clock_normalised(achieved_tflops, clocks, sm_count):
    """The achieved rate against the tensor rate at the SM clock the run actually saw (median of
    the samples taken during the timed region), so kernel changes can be told from clock luck."""
    mhz = (clocks or {}).get("sm_mhz")
    if not mhz or not sm_count:
        return None
    peak = MMA_FLOP_PER_CLK_PER_SM * sm_count * mhz * 1e6 / 1e12
    return {"sm_mhz_median": mhz, "sm_count": sm_count, "tflops_per_ghz": achieved_tflops / (mhz / 1000.0),
            "clock_rate_tensor_peak_tflops": peak, "frac_of_clock_rate_peak": achieved_tflops / peak}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Sources that define the attention kernel measured by the roofline line.
KERNEL_SOURCES = ("attn_fwd_kernel.cuh", "ptx.cuh", "tmem_ldst.cuh")


def kernel_source_hash():
    csrc = os.path.join(ROOT, "exact_causal_attention_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel."""
    path = os.path.join(PROFILES, "attn_fwd_n8192_traffic.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                key, val = line.split(":", 1)
                rec[key.strip()] = val.strip()
    if rec.get("kernel_source_sha256_16") != kernel_source_hash() or rec.get("workload") != WORKLOAD:
        return None
    return int(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class OracleSampler:
    """The FP64 oracle timed on random query rows of a workload (inputs decoded once)."""

    def __init__(self, q, k, v, w):
        import oracle
        from exact_causal_attention_gb300 import inputs

        self.w = w
        self.qd, self.kd, self.vd = (oracle.decode(inputs.bits(x), w.dtype) for x in (q, k, v))
        self.rows_per_s = None

    def flops(self, rows):
        w = self.w
        return float(sum(4.0 * w.D * ((i + 1) if w.causal else w.N) for _, i in rows))

    def run(self, count, seed):
        """Returns (TFLOP/s, rows, seconds) for `count` seeded random rows."""
        import numpy as np

        import oracle

        w = self.w
        rng = np.random.default_rng(seed)
        rows = [(int(rng.integers(0, w.B * w.H)), int(rng.integers(0, w.N))) for _ in range(count)]
        t0 = time.perf_counter()
        oracle.attention_rows(self.qd, self.kd, self.vd, w.causal, w.scale, rows)
        dt = time.perf_counter() - t0
        return self.flops(rows) / dt / 1e12, len(rows), dt

    def timed(self, seconds, seed):
        """A sample sized to take about `seconds` on this host."""
        if self.rows_per_s is None:
            _, n, dt = self.run(4 * host_cores(), seed + 99991)
            self.rows_per_s = n / max(dt, 1e-9)
        return self.run(max(host_cores(), int(seconds * self.rows_per_s)), seed)


def bench_reference(args, w):
    rank, world, _ = rank_env()
    if rank != 0:
        return
    from exact_causal_attention_gb300 import inputs

    q, k, v = inputs.workload_qkv(w)
    sampler = OracleSampler(q, k, v, w)
    per_step = max(0.02, args.reference_seconds / max(1, args.steps + args.warmup))
    for s in range(args.warmup):
        sampler.timed(per_step, seed=100 + s)
    flops, secs, nrows = 0.0, 0.0, 0
    for s in range(args.steps):
        tf, n, dt = sampler.timed(per_step, seed=200 + s)
        flops += tf * 1e12 * dt
        secs += dt
        nrows += n
    value = flops / secs / 1e12
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "seed": w.seed},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nrows} random query rows of the workload over {args.steps} steps "
                                   f"(two-pass FP64 oracle, {cores} threads)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_split(eca, inputs, dev, stream, flush):
    """The key split on causal B=1 H=4 N=8192 D=128 fp16 (too few heads to fill the GPU with
    pair units), with the default segment count (at least 2), against the unsplit kernel (which
    runs key-halves units here); L2 flushed before every call."""
    import torch

    sw = inputs.Workload("causal_b1_h4_n8192_d128_fp16", 1, 4, 8192, 128, "fp16", True, 5)
    sq, sk, sv = (x.to(dev) for x in inputs.workload_qkv(sw))
    so = torch.empty_like(sq)
    sl = torch.empty((sw.B, sw.H, sw.N), dtype=torch.float32, device=dev)
    default_splits = eca.splitkv_default_splits(sw.B, sw.H, sw.N, sw.D)
    splits = max(2, default_splits)  # the split path itself, even when the default is not to split
    need = eca.splitkv_workspace_bytes(sw.B, sw.H, sw.N, sw.D, splits)
    ws = torch.empty(need + 256, dtype=torch.uint8, device=dev)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + need]

    def timed(fn):
        times = []
        for i in range(13):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize(dev)
        ms = sorted(a.elapsed_time(b) for a, b in times[3:])
        return ms[len(ms) // 2]

    t_plain = timed(lambda: eca.attn_fwd_into(sq, sk, sv, so, sl, causal=True, scale=sw.scale, stream=stream))
    t_split = timed(lambda: eca.attn_fwd_splitkv(sq, sk, sv, so, sl, kv_splits=splits, workspace=ws,
                                                 causal=True, scale=sw.scale, stream=stream))
    return {"workload": sw.name, "default_kv_splits": default_splits, "kv_splits": splits, "workspace_bytes": need,
            "unsplit_ms": round(t_plain, 4), "unsplit_tflops": round(sw.flops / (t_plain * 1e-3) / 1e12, 1),
            "split_ms": round(t_split, 4), "split_tflops": round(sw.flops / (t_split * 1e-3) / 1e12, 1),
            "launches_per_call": 2}


def bench_sweep_point(eca, inputs, dev, stream, flush, n):
    """One point of the sweep (causal B=1 H=32 D=128 fp16, seed 1): 10 single calls after an L2
    flush each (median), and 20 back-to-back calls eager and replayed from a CUDA graph."""
    import torch

    sw = inputs.sweep_workload(n)
    sq, sk, sv = (x.to(dev) for x in inputs.workload_qkv(sw))
    so = torch.empty_like(sq)
    sl = torch.empty((sw.B, sw.H, sw.N), dtype=torch.float32, device=dev)

    def call(s=stream):
        eca.attn_fwd_into(sq, sk, sv, so, sl, causal=True, scale=sw.scale, stream=s)

    for _ in range(3):
        call()
    single = []
    for i in range(13):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        single.append((a, b))
    torch.cuda.synchronize(dev)
    single_ms = sorted(a.elapsed_time(b) for a, b in single[3:])[5]
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(20):
        call()
    b.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = a.elapsed_time(b) / 20
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(20):
            call(gs)
    graph.replay()
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = a.elapsed_time(b) / 20
    tf = lambda ms: round(sw.flops / (ms * 1e-3) / 1e12, 1)  # noqa: E731
    return {"workload": sw.name, "launch_order": launch_order(), "single_ms": round(single_ms, 4),
            "single_tflops": tf(single_ms), "eager_ms": round(eager_ms, 4), "eager_tflops": tf(eager_ms),
            "graph_ms": round(graph_ms, 4), "graph_tflops": tf(graph_ms)}


def measure_host_link(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, s, dev, h2d, d2h, kernel_ms):
    """The host link's own rates for one step's buffers (the upload alone, the download alone, both at
    once; median of 5 each) and the step time they allow with the kernel overlapped: the floor the
    end-to-end number is measured against."""
    import torch

    s2 = torch.cuda.Stream(dev)

    def timed(up, down):
        ts = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            s2.wait_event(a)
            with torch.cuda.stream(s):
                if up:
                    dq.copy_(hq, non_blocking=True)
                    dk.copy_(hk, non_blocking=True)
                    dv.copy_(hv, non_blocking=True)
            with torch.cuda.stream(s2):
                if down:
                    ho.copy_(do, non_blocking=True)
                    hl.copy_(dl, non_blocking=True)
            s.wait_stream(s2)
            b.record(s)
            ts.append((a, b))
        torch.cuda.synchronize(dev)
        return sorted(a.elapsed_time(b) for a, b in ts)[2]

    up_ms, down_ms, both_ms = timed(True, False), timed(False, True), timed(True, True)
    floor_ms = max(up_ms, down_ms, both_ms, kernel_ms)
    return {"h2d_gbs": round(h2d / (up_ms * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h / (down_ms * 1e-3) / 1e9, 1),
            "both_ms": round(both_ms, 4), "floor_ms_per_step": round(floor_ms, 4),
            "note": "floor = the slowest of the upload alone, the download alone, both at once, and the kernel"}


def launch_order() -> str:
    """How the library launches its kernels in this process: programmatic dependent launch
    (the default), or plain stream order with ECA_PDL=0."""
    return "stream" if os.environ.get("ECA_PDL") == "0" else "programmatic"



ANATOMY_POINTS = ("entry", "setup_done", "first_k_load_issued", "first_qk_issued", "first_s_ready",
                  "first_o_ready_tile0", "first_output_issued_tile0", "first_o_ready_tile1", "exit")


def bench_anatomy(eca, inputs, dev, stream, flush, n):
    """Per-CTA milestones of two back-to-back attention launches (the sweep workload at N,
    after an L2 flush, both queued behind a spinning kernel), from the anatomy build of
    the library: for each milestone the min / mean / max over CTAs in microseconds after
    the first CTA of the first launch started, the units per CTA, and the gap between
    the last CTA of the first launch and the first of the second."""
    import ctypes

    import torch

    lib = eca.load_library(eca.ANATOMY_LIB_PATH)
    sw = inputs.sweep_workload(n)
    sq, sk, sv = (x.to(dev) for x in inputs.workload_qkv(sw))
    so = torch.empty_like(sq)
    sl = torch.empty((sw.B, sw.H, sw.N), dtype=torch.float32, device=dev)

    def call():
        eca.attn_fwd_into(sq, sk, sv, so, sl, causal=True, scale=sw.scale, stream=stream)

    for _ in range(3):
        call()
    words = 2 * 160 * 10
    buf = (ctypes.c_ulonglong * words)()
    if lib.attn_anatomy_read(buf, words, 1) != 0:
        raise RuntimeError("attn_anatomy_read failed: not the anatomy build?")
    flush.zero_()
    # A spinning kernel of about 0.5 ms ahead of the two calls, so both are queued on
    # the GPU before the first starts and the gap between them is the GPU's own.
    torch.cuda._sleep(1_000_000)
    call()
    call()
    torch.cuda.synchronize(dev)
    if lib.attn_anatomy_read(buf, words, 1) != 0:
        raise RuntimeError("attn_anatomy_read failed")
    st = [[[buf[(sl_ * 160 + c) * 10 + i] for i in range(10)] for c in range(160)] for sl_ in range(2)]
    t0 = min(st[0][c][0] for c in range(160) if st[0][c][0])
    out = {"workload": sw.name, "launches": []}
    for slot in range(2):
        ctas = [c for c in range(160) if st[slot][c][0]]
        rec = {"ctas": len(ctas), "units_per_cta": sorted({st[slot][c][9] for c in ctas})}
        for i, name in enumerate(ANATOMY_POINTS):
            v = [(st[slot][c][i] - t0) / 1000.0 for c in ctas if st[slot][c][i]]
            if v:
                rec[name] = {"min": round(min(v), 2), "mean": round(sum(v) / len(v), 2), "max": round(max(v), 2)}
        out["launches"].append(rec)
    a, b = out["launches"]
    if "exit" in a and "entry" in b:
        out["gap_us_last_exit_to_next_first_entry"] = round(b["entry"]["min"] - a["exit"]["max"], 2)
    return out


def bench_workloads(eca, inputs, dev, stream, flush):
    """Every parity workload (the page's configurations, bf16 and D = 64 included) timed as a
    single call after an L2 flush (median of 10 after 3) and as 20 calls back to back;
    TFLOP/s counts 2BHN²D causal and 4BHN²D non-causal, as the headline."""
    import torch

    out = {}
    for name, w in inputs.WORKLOADS.items():
        q, k, v = (x.to(dev) for x in inputs.workload_qkv(w))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

        def call():
            eca.attn_fwd_into(q, k, v, o, lse, causal=w.causal, scale=w.scale, stream=stream)

        for _ in range(3):
            call()
        single = []
        for _ in range(13):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            single.append((a, b))
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(20):
            call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = sorted(x.elapsed_time(y) for x, y in single[3:])[5]
        b2b = a.elapsed_time(b) / 20
        out[name] = {"single_ms": round(ms, 4), "single_tflops": round(w.flops / (ms * 1e-3) / 1e12, 1),
                     "back_to_back_ms": round(b2b, 4), "back_to_back_tflops": round(w.flops / (b2b * 1e-3) / 1e12, 1)}
        del q, k, v, o, lse
    return out


def bench_gqa(eca, inputs, dev, stream, flush):
    """Grouped heads, causal B=1 H=32 Hkv=8 N=8192 D=128 fp16 (4 query heads per key/value head);
    L2 flushed before every call; TFLOP/s counts 2BHN²D."""
    import torch

    gq, _, _ = inputs.make_qkv(1, 32, 8192, 128, "fp16", seed=6)
    _, gk, gv = inputs.make_qkv(1, 8, 8192, 128, "fp16", seed=7)
    gq, gk, gv = gq.to(dev), gk.to(dev), gv.to(dev)
    go = torch.empty_like(gq)
    gl = torch.empty((1, 32, 8192), dtype=torch.float32, device=dev)
    times = []
    for i in range(13):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        eca.attn_fwd_gqa(gq, gk, gv, causal=True, o=go, lse=gl, stream=stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize(dev)
    ms = sorted(a.elapsed_time(b) for a, b in times[3:])
    med = ms[len(ms) // 2]
    flops = 2.0 * 32 * 8192 * 8192 * 128
    return {"workload": "causal_b1_h32_hkv8_n8192_d128_fp16", "ms": round(med, 4),
            "tflops": round(flops / (med * 1e-3) / 1e12, 1)}


def bench_row_softmax(eca, inputs, dev, stream, flush):
    """The fp32 online row softmax on the HBM-sized shape (larger than L2) and on the page's shape
    (L2 flushed before each call); GB/s counts one read and one write per element."""
    import torch

    peaks_rs, kind_rs = measured_peaks()
    row_softmax = {}
    for (M, Ncols, seed), label in ((inputs.SOFTMAX_HBM_SHAPE, "hbm"), (inputs.SOFTMAX_PAGE_SHAPE, "page")):
        xs = inputs.uniform_matrix(M, Ncols, seed).to(dev)
        ys = torch.empty_like(xs)
        times = []
        for i in range(13):
            if label == "page":
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            eca.row_softmax(xs, ys, stream=stream)
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize(dev)
        ms = sorted(a.elapsed_time(b) for a, b in times[3:])
        med = ms[len(ms) // 2]
        gbs = 8.0 * M * Ncols / (med * 1e-3) / 1e9
        row_softmax[label] = {"M": M, "N": Ncols, "us": round(med * 1e3, 2), "GB_s": round(gbs, 1),
                              "frac_of_hbm": round(gbs / float(peaks_rs["hbm_gbs"]), 3)}
        del xs, ys
    row_softmax["hbm_peak_gbs"] = float(peaks_rs["hbm_gbs"])
    row_softmax["peak_kind"] = kind_rs
    return row_softmax


def bench_paged(eca, inputs, dev, stream, flush, contexts):
    """Paged GQA decode over the decode page's geometry (B=8, Hq=32, Hkv=8, D=128,
    page size 16): HBM-bound, it must stream 2 B L Hkv D s bytes of K/V per step.
    Median of 10 calls after 3 per context, L2 flushed before each."""
    import torch

    paged = {}
    peaks_pd, _ = measured_peaks()
    pw = inputs.PAGED_BENCH
    gen = torch.Generator(device=dev).manual_seed(pw.seed)
    for ctx in contexts:
        pages = (ctx + pw.page_size - 1) // pw.page_size
        P = pw.B * pages
        cache = torch.randn(P, 2, pw.page_size, pw.Hkv, pw.D, generator=gen, device=dev, dtype=torch.float16)
        table = torch.randperm(P, generator=gen, device=dev).to(torch.int32).view(pw.B, pages).contiguous()
        lens = torch.full((pw.B,), ctx, dtype=torch.int32, device=dev)
        qd = torch.randn(pw.B, pw.Hq, pw.D, generator=gen, device=dev, dtype=torch.float16)
        outd = torch.empty_like(qd)
        lsed = torch.empty((pw.B, pw.Hq), dtype=torch.float32, device=dev)
        splits = eca.load_library().attn_decode_default_splits(pw.B, pw.Hq, pw.Hkv, pw.page_size, pages)
        need = int(eca.load_library().attn_decode_workspace_bytes(pw.B, pw.Hq, pw.D, splits))
        ws = torch.empty(need + 256, dtype=torch.uint8, device=dev) if need else None
        if ws is not None:
            off = (-ws.data_ptr()) % 256
            ws = ws[off:off + need]
        times = []
        for i in range(13):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            eca.decode_paged(qd, cache, table, lens, kv_splits=splits, out=outd, lse=lsed, workspace=ws,
                             stream=stream)
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize(dev)
        ms = sorted(a.elapsed_time(b) for a, b in times[3:])
        med = ms[len(ms) // 2]
        kv = 2 * pw.B * ctx * pw.Hkv * pw.D * 2
        paged[str(ctx)] = {"us": round(med * 1e3, 2), "GB_s": round(kv / (med * 1e-3) / 1e9, 1),
                           "frac_of_hbm": round(kv / (med * 1e-3) / 1e9 / float(peaks_pd["hbm_gbs"]), 3),
                           "kv_splits": splits}
        if ctx == contexts[-1]:
            newkv = torch.randn(pw.B, 2, pw.Hkv, pw.D, generator=gen, device=dev, dtype=torch.float16)
            # The append's device work is far shorter than the host's call, so calls timed one at a
            # time measure the host.  Each group queues 20 calls behind a ~0.5 ms spin (outside the
            # events), so the device runs them back to back: median of 7 group means per call.
            at = []
            reps = 20
            for i in range(9):
                with torch.cuda.stream(stream):
                    torch.cuda._sleep(1_000_000)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(reps):
                    eca.paged_append(newkv, cache, table, lens, stream=stream)
                b.record(stream)
                at.append((a, b))
            torch.cuda.synchronize(dev)
            ams = sorted(a.elapsed_time(b) / reps for a, b in at[2:])
            paged["append_us"] = round(ams[len(ams) // 2] * 1e3, 2)
            paged["append_timing"] = f"per call, {reps} calls back to back behind a spin, median of 7 groups"
        del cache, table, lens, qd, outd, lsed, ws
    span = f"ctx{contexts[0]}" if len(contexts) == 1 else f"ctx{contexts[0]}..{contexts[-1]}"
    paged["workload"] = pw.name.replace("ctx32768", span)
    return paged


def bench_ours(args, w):
    import torch
    import torch.distributed as dist

    import exact_causal_attention_gb300 as eca
    from exact_causal_attention_gb300 import inputs

    rank, world, local = rank_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    eca.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    q, k, v = inputs.workload_qkv(w)
    dq, dk, dv = (x.to(dev) for x in (q, k, v))
    o = torch.empty_like(dq)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        eca.attn_fwd_into(dq, dk, dv, o, lse, causal=w.causal, scale=w.scale, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if eca.device_status() != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    for i in range(args.steps):
        flush.zero_()  # untimed: evicts q, k, v, o from L2 between steps
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    status = eca.device_status()
    if status != 0:
        raise RuntimeError("a kernel wait timed out in the timed region")
    flops = w.flops
    value = whole_job_tflops(flops, args.steps, world, total_ms)
    kernel_ms = total_ms / args.steps

    # End to end through the C ABI: pinned host q, k, v in, o and lse out, every step.
    # Two device buffer sets and three streams, as a serving loop would run it: the
    # upload of step i + 1 and the download of step i - 1 overlap the kernel of step i.
    hq, hk, hv = (x.pin_memory() for x in (q, k, v))
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    bq = [dq, torch.empty_like(dq)]
    bk = [dk, torch.empty_like(dk)]
    bv = [dv, torch.empty_like(dv)]
    bo = [o, torch.empty_like(o)]
    bl = [lse, torch.empty_like(lse)]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_steps = max(4, min(args.steps, 40))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    done_down = [None, None]   # buffer set free again (its download finished)
    done_kernel = [None, None]  # buffer set's inputs consumed and outputs written

    def e2e_run(n):
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(s_up):
                if done_kernel[j] is not None:
                    s_up.wait_event(done_kernel[j])
                bq[j].copy_(hq, non_blocking=True)
                bk[j].copy_(hk, non_blocking=True)
                bv[j].copy_(hv, non_blocking=True)
                up = ev()
                up.record(s_up)
            stream.wait_event(up)
            if done_down[j] is not None:
                stream.wait_event(done_down[j])
            eca.attn_fwd_into(bq[j], bk[j], bv[j], bo[j], bl[j], causal=w.causal, scale=w.scale, stream=stream)
            done_kernel[j] = ev()
            done_kernel[j].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(done_kernel[j])
                ho[j].copy_(bo[j], non_blocking=True)
                hl[j].copy_(bl[j], non_blocking=True)
                done_down[j] = ev()
                done_down[j].record(s_down)

    e2e_run(2)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    e2e_run(e2e_steps)
    s_up.wait_stream(s_down)
    s_up.wait_stream(stream)
    e1.record(s_up)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    if eca.device_status() != 0:
        raise RuntimeError("a kernel wait timed out in the end-to-end loop")
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    host_link = measure_host_link(hq, hk, hv, ho[0], hl[0], bq[1], bk[1], bv[1], bo[1], bl[1], s_up, dev,
                                  h2d, d2h, kernel_ms)
    host_link["e2e_frac_of_floor"] = round(host_link["floor_ms_per_step"] / e2e_ms, 3)

    sweep = {}
    sweep_graph = {}
    if not args.no_sweep and rank == 0:
        # The page's timing (section 8): warm-up, then 7 groups of back-to-back calls timed
        # with CUDA events (5-30 calls a group, about 2 ms of work), the median of the group
        # means; L2 flushed before each group.
        for n in inputs.SWEEP_N:
            sw = inputs.sweep_workload(n)
            sq, sk, sv = (x.to(dev) for x in inputs.workload_qkv(sw))
            so = torch.empty_like(sq)
            sl = torch.empty((sw.B, sw.H, sw.N), dtype=torch.float32, device=dev)

            def call():
                eca.attn_fwd_into(sq, sk, sv, so, sl, causal=True, scale=sw.scale, stream=stream)

            for _ in range(3):
                call()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize(dev)
            reps = int(min(30, max(5, round(2.0 / max(a.elapsed_time(b), 1e-3)))))
            groups = []
            for g in range(7):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(reps):
                    call()
                b.record(stream)
                groups.append((a, b))
            torch.cuda.synchronize(dev)
            means = sorted(a.elapsed_time(b) / reps for a, b in groups)
            med = means[len(means) // 2]
            sweep[str(n)] = {"ms": round(med, 4), "tflops": round(sw.flops / (med * 1e-3) / 1e12, 1),
                             "calls_per_group": reps}
            # The same groups captured once in a CUDA graph and replayed: the calls are
            # unchanged, only the launch gaps between them go (short N is launch-bound).
            gs = torch.cuda.Stream(dev)
            gs.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(reps):
                    eca.attn_fwd_into(sq, sk, sv, so, sl, causal=True, scale=sw.scale, stream=gs)
            graph.replay()
            torch.cuda.synchronize(dev)
            groups = []
            for g in range(7):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graph.replay()
                b.record(stream)
                groups.append((a, b))
            torch.cuda.synchronize(dev)
            means = sorted(a.elapsed_time(b) / reps for a, b in groups)
            med = means[len(means) // 2]
            sweep_graph[str(n)] = {"ms": round(med, 4), "tflops": round(sw.flops / (med * 1e-3) / 1e12, 1),
                                   "calls_per_group": reps}
            del graph, sq, sk, sv, so, sl

    # Key split on a workload too small in B x H to fill the GPU (causal, B=1, H=4, N=8192, D=128).
    splitkv = bench_split(eca, inputs, dev, stream, flush) if (not args.no_sweep and rank == 0) else {}

    # Grouped key/value heads (GQA, 4 query heads per key/value head), causal B=1 H=32 Hkv=8 N=8192 D=128.
    gqa = bench_gqa(eca, inputs, dev, stream, flush) if (not args.no_sweep and rank == 0) else {}
    workloads = bench_workloads(eca, inputs, dev, stream, flush) if (not args.no_sweep and rank == 0) else {}

    # Online row softmax (fp32): an HBM-bound kernel, one read and one write per element.
    row_softmax = bench_row_softmax(eca, inputs, dev, stream, flush) if (not args.no_sweep and rank == 0) else {}

    paged = bench_paged(eca, inputs, dev, stream, flush, inputs.PAGED_CONTEXTS) if (not args.no_sweep and rank == 0) else {}

    fp16_peak = None
    if not args.no_peak and rank == 0:
        a = torch.randn(8192, 8192, device=dev, dtype=torch.float16)
        b = torch.randn(8192, 8192, device=dev, dtype=torch.float16)
        for _ in range(3):
            a @ b
        best = float("inf")
        for _ in range(10):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            a @ b
            s1.record(stream)
            s1.synchronize()
            best = min(best, s0.elapsed_time(s1))
        fp16_peak = 2 * 8192 ** 3 / (best * 1e-3) / 1e12
        del a, b

    cpu = None
    single = None
    if rank == 0 and not args.no_cpu:
        tf, nrows, secs = OracleSampler(q, k, v, w).timed(args.cpu_seconds, seed=7)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{nrows} random query rows of the workload ({secs:.1f} s, two-pass FP64 oracle, "
                         f"{host_cores()} threads)"}
        # The whole of the two small workloads on one host thread.
        import oracle

        single = {}
        for name in ("causal_b1_h2_n256_d64_fp16", "causal_b1_h32_n512_d128_fp16"):
            sw = inputs.WORKLOADS[name]
            qd, kd, vd = (oracle.decode(inputs.bits(x), sw.dtype) for x in inputs.workload_qkv(sw))
            t0 = time.perf_counter()
            oracle.attention(qd, kd, vd, sw.causal, sw.scale, nthreads=1)
            dt = time.perf_counter() - t0
            single[name] = {"s": round(dt, 4), "tflops": sw.flops / dt / 1e12, "threads": 1}

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks, kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])  # fp16 and bf16 share one nominal dense rate (ratio 1.0)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": kernel_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / world / (flops / (PAGE_MS_N8192 * 1e-3) / 1e12),
        "dtype": "fp16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                   "seed": w.seed, "flops_per_step": flops, "executed_flops_per_step": executed_flops(w),
                   "l2": "flushed between timed steps (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{kind} bf16 burst (fp16/bf16 nominal ratio 1.0)",
                     "traffic": recorded_traffic(),
                     # For runs long enough to hold the part at its power cap (the default 2000 steps):
                     # the same rate against the measured sustained GEMM rate.
                     "sustained_peak": float(peaks["bf16_tflops_sustained"]),
                     "frac_of_sustained_peak": achieved / float(peaks["bf16_tflops_sustained"])},
        "cpu_baseline": cpu,
        "oracle_single_thread": single,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "schedule": "pinned host buffers; two device buffer sets; upload, kernel and download on three "
                            "streams, the upload of step i + 1 and download of step i - 1 overlapping kernel i",
                "host_link": host_link},
        "gpu_launches": args.steps,
        "launch_order": launch_order(),
        "clocks": clocks,
        "sweep": sweep,
        "sweep_graph": sweep_graph,
        "splitkv": splitkv,
        "gqa": gqa,
        "workloads": workloads,
        "row_softmax": row_softmax,
        "paged_decode": paged,
        "fp16_matmul_peak_tflops": fp16_peak,
        "frac_of_measured_fp16_matmul": (achieved / fp16_peak) if fp16_peak else None,
        "frac_of_datasheet_dense_fp16": achieved / DATASHEET_DENSE_FP16_TFLOPS,
        "datasheet_source": DATASHEET_SOURCE,
        "clock_normalised": clock_normalised(achieved, clocks, sm_count),
        "vs_baseline_ref": "page's PyTorch SDPA FLASH on RTX 3060 Laptop (SM86): 25.854 ms",
    }
    print(json.dumps(line), flush=True)


def run_probe(name):
    """Builds (if stale) and runs the measurement probe csrc/<name>.cu; returns its JSON output."""
    from exact_causal_attention_gb300 import build as cuda_build

    src = os.path.join(cuda_build.CSRC, name + ".cu")
    exe = os.path.join(cuda_build.BUILD_DIR, name)
    os.makedirs(cuda_build.BUILD_DIR, exist_ok=True)
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        subprocess.run([cuda_build._nvcc(), *cuda_build.ARCH_FLAGS, "-O2", "-std=c++17", "-o", exe, src], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    return json.loads(out)


def bench_launch_cost():
    """csrc/launch_cost_probe.cu: microseconds per launch of empty one-CTA-per-SM kernels, 200 back to
    back, for the launch boundaries that set the floor of a short call."""
    return run_probe("launch_cost_probe")


def bench_ingress():
    """csrc/ingress_probe.cu: the rate at which bulk copies fill one SM's shared memory, from HBM and
    from L2, with 16, 64 and all SMs streaming, each CTA alone or in multicast pairs: the ceiling on
    the K/V tile fills of the attention kernel."""
    return run_probe("ingress_probe")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-peak", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0,
                    help="--impl reference: oracle time over warm-up and timed steps together")
    ap.add_argument("--paged-only", type=int, nargs="*", metavar="CONTEXT",
                    help="only the paged-decode measurement, at the given contexts (default: all)")
    ap.add_argument("--softmax-only", action="store_true", help="only the row-softmax measurement")
    ap.add_argument("--split-only", action="store_true", help="only the key-split measurement")
    ap.add_argument("--gqa-only", action="store_true", help="only the grouped-head measurement")
    ap.add_argument("--anatomy", type=int, metavar="N",
                    help="per-CTA milestones of two back-to-back launches of the sweep workload at N (anatomy build)")
    ap.add_argument("--sweep-only", type=int, metavar="N",
                    help="only the sweep workload at this N (causal B=1 H=32 D=128 fp16), eager and from a graph")
    ap.add_argument("--launch-cost", action="store_true",
                    help="time per launch of empty kernels (with and without global stores and tensor memory) in "
                         "stream order, with programmatic dependent launch and from a CUDA graph")
    ap.add_argument("--ingress", action="store_true",
                    help="shared-memory fill rate per SM by bulk copies, from HBM and from L2")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.launch_cost:
        print(json.dumps({"launch_cost": bench_launch_cost()}), flush=True)
        return
    if args.ingress:
        print(json.dumps({"ingress": bench_ingress()}), flush=True)
        return
    from exact_causal_attention_gb300 import inputs

    w = inputs.WORKLOADS[WORKLOAD]
    if (args.paged_only is not None or args.softmax_only or args.split_only or args.gqa_only or args.sweep_only
            or args.anatomy):
        # One side measurement alone (for profiling its kernels); one JSON line.
        import torch

        import exact_causal_attention_gb300 as eca

        if not args.anatomy:
            eca.load_library()
        dev = torch.device("cuda", 0)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev)
        if args.paged_only is not None:
            contexts = args.paged_only or list(inputs.PAGED_CONTEXTS)
            out = {"paged_decode": bench_paged(eca, inputs, dev, stream, flush, contexts)}
        elif args.softmax_only:
            out = {"row_softmax": bench_row_softmax(eca, inputs, dev, stream, flush)}
        elif args.anatomy:
            out = {"anatomy": bench_anatomy(eca, inputs, dev, stream, flush, args.anatomy)}
        elif args.sweep_only:
            out = {"sweep": bench_sweep_point(eca, inputs, dev, stream, flush, args.sweep_only)}
        elif args.gqa_only:
            out = {"gqa": bench_gqa(eca, inputs, dev, stream, flush)}
        else:
            out = {"splitkv": bench_split(eca, inputs, dev, stream, flush)}
        print(json.dumps(out), flush=True)
        return
    if args.impl == "reference":
        bench_reference(args, w)
    else:
        bench_ours(args, w)


if __name__ == "__main__":
    main()
