#!/usr/bin/env python
"""Throughput of the fused DiT-block elementwise path on GB300.

One step = one pass of the chained block path over one batch of the
75,600-token workload (73,728 video + 1,872 audio tokens, hidden 5120,
40 heads x 128, ffn 13824): RMSNorm + indexed AdaLN -> Q/K RMSNorm + NeoX
RoPE -> SwiGLU, back to back on one stream through the C ABI, inputs
resident in HBM.  The same run also times the valid-only pipeline (gather ->
RMSNorm+AdaLN and Q/K norm+RoPE on the valid rows -> zero-tail merge) on the
32,768-row padded buffer, reports each kernel against the HBM roofline, the
end-to-end rate with host buffers, and the fp64 CPU oracle timed on this
host's cores.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the reference arm).  Multi-GPU (torchrun): every rank runs its own
batch (weak scaling, no collective on the data path); rank 0 reports the
whole-job rate over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402  (seeded inputs; holds none of the path's arithmetic)

METRIC = "tokens/s and achieved HBM GB/s (% of GB300 peak) for the fused DiT-block path"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}
L2_BYTES = 129 * 1024 * 1024


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["tfk", "reference"], default="tfk")
    ap.add_argument("--workload", default="large", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--rows", type=int, default=0,
                    help="use only the first ROWS tokens of the workload (small cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="time box of the oracle baseline")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="time budget of the whole --impl reference run (oracle steps are sized to it)")
    ap.add_argument("--no-valid-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep-workloads", default="tiny,medium,valid_only,large,per_frame",
                    help="comma-separated workloads of --sweep (--rows cuts the chain workloads to a prefix)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every kernel on every workload (one JSON line per workload) instead of the step")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

class Ranks:
    """RANK / WORLD_SIZE / LOCAL_RANK from torchrun; a process group only when world > 1."""

    def __init__(self, backend: str | None = None):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        if self.world > 1:
            import torch.distributed as dist
            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":  # bind this rank's GPU before NCCL picks one for barriers
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, v: float) -> float:
        """Maximum of a host scalar over ranks."""
        if not self.pg:
            return v
        import torch.distributed as dist
        dev = torch.device("cuda", self.local_rank) if dist.get_backend() == "nccl" else torch.device("cpu")
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return per_rank_units * world / max_seconds


# ---------------------------------------------------------------------------
# peaks, clocks, profiles
# ---------------------------------------------------------------------------

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS)


class ClockSampler:
    """nvidia-smi samples every 200 ms while it runs; summarises the window of the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for r in csv.reader(io.StringIO(open(self.path).read())):
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(r[2]), float(r[3]), r[6].strip(), r[7].strip(), r[8].strip(), r[9].strip()))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        reasons = set()
        for r in inside:
            for name, flag in (("hw_slowdown", r[3]), ("hw_thermal_slowdown", r[4]),
                               ("sw_thermal_slowdown", r[5]), ("sw_power_cap", r[6])):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def profiled_traffic(kernel: str, workload: str, source: str) -> float | None:
    """DRAM bytes per launch of `kernel` from the committed ncu summary (a capture of a
    16,384-token prefix scaled to the full workload, profiles/dram_traffic.txt), if it was
    taken on the kernel source as it is now (sha256 of the .cu file)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, "rope_tfk_rmsnorm_gb300", "csrc", source), "rb").read()).hexdigest()
    for line in open(path):
        kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
        if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("source_sha256") == sha:
            return float(kv["dram_bytes_per_launch"])
    return None


# ---------------------------------------------------------------------------
# algorithmic bytes (the bytes the method must move, nothing else)
# ---------------------------------------------------------------------------

def bytes_adaln(rows: int, hidden: int, n_mod_used: int) -> int:
    """x read + y written (2+2 B/element), 4 B index per row, one pass over the fp32
    norm weight and over the shift/scale rows in use."""
    return rows * (4 * hidden + 4) + 4 * hidden + 8 * hidden * n_mod_used


def bytes_qk(rows: int, n_heads: int, head_dim: int) -> int:
    """q, k read and written (8 B per q/k element pair), 4 B position per row, two fp32 weights."""
    return rows * (8 * n_heads * head_dim + 4) + 8 * head_dim


def bytes_swiglu(rows: int, ffn: int) -> int:
    """gate and up read, out written: 6 B per output element."""
    return rows * 6 * ffn


def bytes_gather(valid_rows: int, hidden: int) -> int:
    return 4 * hidden * valid_rows


def bytes_merge(valid_rows: int, padded_rows: int, hidden: int) -> int:
    return 2 * hidden * (valid_rows + padded_rows)


# ---------------------------------------------------------------------------
# the chained block path
# ---------------------------------------------------------------------------

def _pinned_bf16(shape):
    return torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


class Chain:
    """Inputs (pinned host copies + resident device copies) and outputs of one step."""

    def __init__(self, tfk, wl, device):
        self.tfk, self.wl, self.dev = tfk, wl, device
        T, hd, qk, F = wl.rows, wl.hidden, wl.n_heads * wl.head_dim, wl.ffn
        self.host = {"x": _pinned_bf16((T, hd)), "q": _pinned_bf16((T, qk)), "k": _pinned_bf16((T, qk)),
                     "gate_up": _pinned_bf16((T, 2 * F))}
        for tag, t in self.host.items():
            synth.activation(wl, tag, out=_bits(t))
        idx, pos = synth.mod_index(wl), synth.positions(wl)
        self.n_mod_used = int(len(np.unique(idx)))
        self.host["idx"] = torch.from_numpy(idx).pin_memory()
        self.host["pos"] = torch.from_numpy(pos).pin_memory()
        self.params = {k: torch.from_numpy(v).to(device) for k, v in synth.params(wl).items()}
        self.d = {k: v.to(device) for k, v in self.host.items()}
        self.out = {"y": torch.empty((T, hd), dtype=torch.bfloat16, device=device),
                    "q": torch.empty((T, qk), dtype=torch.bfloat16, device=device),
                    "k": torch.empty((T, qk), dtype=torch.bfloat16, device=device),
                    "o": torch.empty((T, F), dtype=torch.bfloat16, device=device)}
        self.host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in self.out.items()}
        self.kernels = ["rmsnorm_adaln", "qk_rmsnorm_rope", "swiglu"]
        self.bytes = [bytes_adaln(T, hd, self.n_mod_used), bytes_qk(T, wl.n_heads, wl.head_dim),
                      bytes_swiglu(T, F)]

    def launch(self, ev=None):
        t, p, d, o, wl = self.tfk, self.params, self.d, self.out, self.wl
        if ev:
            ev[0].record()
        t.tfk_rmsnorm_adaln_indexed(d["x"], p["w"], p["shift"], p["scale"], d["idx"], wl.eps, out=o["y"])
        if ev:
            ev[1].record()
        t.tfk_qk_rmsnorm_rope_neox(d["q"], d["k"], p["w_q"], p["w_k"], d["pos"], wl.n_heads, wl.head_dim,
                                   wl.theta, wl.eps, q_out=o["q"], k_out=o["k"])
        if ev:
            ev[2].record()
        t.tfk_swiglu(d["gate_up"], out=o["o"])
        if ev:
            ev[3].record()

    def upload(self):
        for k, h in self.host.items():
            self.d[k].copy_(h, non_blocking=True)

    def download(self):
        for k, dv in self.out.items():
            self.host_out[k].copy_(dv, non_blocking=True)

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.out.values())


class ValidOnly:
    """Valid-only pipeline on the padded buffer: gather X, Q, K -> RMSNorm+AdaLN and
    Q/K norm+RoPE on the L valid rows -> zero-tail merge of Y, Q', K'."""

    def __init__(self, tfk, wl, device):
        self.tfk, self.wl = tfk, wl
        N, L, hd = wl.rows, synth.valid_len(wl), wl.hidden
        self.N, self.L = N, L
        self.pad = {}
        for tag in ("x", "q", "k"):
            h = _pinned_bf16((N, hd))
            synth.activation(wl, tag, out=_bits(h))
            self.pad[tag] = h.to(device)
        self.idx = torch.from_numpy(synth.mod_index(wl, np.arange(L))).to(device)
        self.pos = torch.from_numpy(synth.positions(wl, np.arange(L))).to(device)
        self.params = {k: torch.from_numpy(v).to(device) for k, v in synth.params(wl).items()}
        mk = lambda r: torch.empty((r, hd), dtype=torch.bfloat16, device=device)  # noqa: E731
        self.comp = {t: mk(L) for t in ("x", "q", "k")}
        self.res = {t: mk(L) for t in ("y", "q", "k")}
        self.merged = {t: mk(N) for t in ("y", "q", "k")}
        self.kernels = ["valid_gather_x3", "rmsnorm_adaln", "qk_rmsnorm_rope", "zero_tail_merge_x3"]
        self.bytes = [3 * bytes_gather(L, hd), bytes_adaln(L, hd, 2), bytes_qk(L, wl.n_heads, wl.head_dim),
                      3 * bytes_merge(L, N, hd)]

    def launch(self, ev=None):
        t, wl, p = self.tfk, self.wl, self.params
        if ev:
            ev[0].record()
        for tag in ("x", "q", "k"):
            t.tfk_valid_gather(self.pad[tag], self.L, compact=self.comp[tag])
        if ev:
            ev[1].record()
        t.tfk_rmsnorm_adaln_indexed(self.comp["x"], p["w"], p["shift"], p["scale"], self.idx, wl.eps,
                                    out=self.res["y"])
        if ev:
            ev[2].record()
        t.tfk_qk_rmsnorm_rope_neox(self.comp["q"], self.comp["k"], p["w_q"], p["w_k"], self.pos, wl.n_heads,
                                   wl.head_dim, wl.theta, wl.eps, q_out=self.res["q"], k_out=self.res["k"])
        if ev:
            ev[3].record()
        for tag in ("y", "q", "k"):
            t.tfk_zero_tail_merge(self.res[tag], self.merged[tag])
        if ev:
            ev[4].record()


def queue_ahead(steps: int):
    """Hold the stream in a GPU-side wait (about 0.1 ms per step, a torch kernel) so that
    the host queues the launches of the per-kernel pass before the GPU reaches them;
    otherwise, for kernels about as short as the host's submission time of a call
    (~10 us through the Python binding), the GPU idles between the events and the
    interval of a launch includes that wait (8,192 x 3072 RMSNorm+AdaLN: 26.1 us mean
    without, 24.6 us with; medians 24.5 us both)."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(min(steps, 1000) * 200_000))


def time_steps(work, steps: int, warmup: int, ranks: Ranks):
    """W untimed steps, then exactly `steps` timed steps between barriers and syncs,
    with CUDA events only at the two ends: an event recorded between two launches
    would make the second wait for the first's full completion and so remove the
    overlap that programmatic dependent launch gives.  A second pass of the same
    steps, outside the timed region, records an event between every launch for
    the per-kernel breakdown.  Returns (total ms of the timed steps on the device,
    per-kernel mean ms, wall t0, wall t1 of the timed steps, per-kernel {p10, p50,
    p90} ms)."""
    n_ev = len(work.kernels) + 1
    for _ in range(warmup):
        work.launch()
    torch.cuda.synchronize()
    ranks.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record()
    for _ in range(steps):
        work.launch()
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    ranks.barrier()
    total = start.elapsed_time(end)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    queue_ahead(steps)
    for s in range(steps):
        work.launch(evs[s])
    torch.cuda.synchronize()
    samples = [[evs[s][j].elapsed_time(evs[s][j + 1]) for s in range(steps)] for j in range(n_ev - 1)]
    per_kernel = [statistics.fmean(v) for v in samples]
    dist = [{f"p{q}": float(np.percentile(v, q)) for q in (10, 50, 90)} for v in samples]
    return total, per_kernel, t0, t1, dist


# ---------------------------------------------------------------------------
# the fp64 CPU oracle as a baseline (bounded samples of the same workload)
# ---------------------------------------------------------------------------

def _oracle_chain(oracle, wl, rows: np.ndarray, p: dict, threads: int):
    """Generate (untimed) and run (timed) the oracle chain on the given rows; returns seconds."""
    x, q, k = (synth.activation(wl, t, rows=rows) for t in ("x", "q", "k"))
    gu = synth.activation(wl, "gate_up", rows=rows) if wl.ffn > 0 else None   # no FFN on the valid-only workload
    idx, pos = synth.mod_index(wl, rows), synth.positions(wl, rows)
    t0 = time.perf_counter()
    oracle.round_bf16(oracle.rmsnorm_adaln_indexed(x, p["w"], p["shift"], p["scale"], idx, wl.eps, threads=threads))
    qo, ko = oracle.qk_rmsnorm_rope_neox(q, k, p["w_q"], p["w_k"], pos, wl.n_heads, wl.head_dim, wl.theta,
                                         wl.eps, threads=threads)
    oracle.round_bf16(qo)
    oracle.round_bf16(ko)
    if gu is not None:
        oracle.round_bf16(oracle.swiglu(gu, threads=threads))
    return time.perf_counter() - t0


def oracle_rates(wl) -> dict:
    """The oracle beside every sweep workload: a bounded sample of rows on one thread
    and on all host threads (a second or two of CPU work per workload)."""
    import oracle
    threads = os.cpu_count() or 1
    p = synth.params(wl)
    limit = synth.valid_len(wl)
    n1, nall = min(limit, 32), min(limit, 512)
    t1 = _oracle_chain(oracle, wl, np.arange(n1), p, 1)
    tall = _oracle_chain(oracle, wl, np.arange(nall), p, threads)
    return {"tokens_per_s_1thread": n1 / t1, "tokens_per_s_all_threads": nall / tall, "threads": threads,
            "sample": f"first {n1} / {nall} rows, fp64 oracle chain, input generation untimed"}


def cpu_baseline(wl, seconds: float) -> dict:
    """The oracle, as it stands, on this host's cores: chunks of 256 rows spread over the
    workload until `seconds` of timed oracle work have run."""
    import oracle
    threads = os.cpu_count() or 1
    p = synth.params(wl)
    rng_rows = np.arange(wl.rows)
    chunk, done, spent, start = 256, 0, 0.0, 0
    stride = max(chunk, wl.rows // 16)
    while spent < seconds and done < wl.rows:
        rows = rng_rows[start:start + chunk]
        if len(rows) == 0:
            break
        spent += _oracle_chain(oracle, wl, rows, p, threads)
        done += len(rows)
        start = (start + stride) % max(1, wl.rows - chunk)
    one = min(64, wl.rows)  # the same oracle on one thread, on a smaller sample
    one_s = _oracle_chain(oracle, wl, rng_rows[:one], p, 1)
    return {"value": done / spent, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} rows of the {wl.name} workload ({wl.rows} rows) in chunks of {chunk}, "
                      f"{spent:.1f} s of timed fp64 oracle work (RMSNorm+AdaLN, Q/K RMSNorm+RoPE, SwiGLU, "
                      f"bf16 rounding, which the oracle runs on one thread); input generation untimed",
            "value_1thread": one / one_s, "sample_1thread": f"the first {one} rows on 1 thread"}


def run_reference(args, ranks: Ranks) -> dict | None:
    """Reference arm: the fp64 CPU oracle, each step a bounded sample of the workload."""
    if ranks.rank != 0:
        return None
    import oracle
    wl = synth.get(args.workload)
    threads = os.cpu_count() or 1
    p = synth.params(wl)
    oracle.build()
    budget = args.ref_seconds / max(1, args.steps + args.warmup)  # seconds per step: the run ends in minutes
    rows_per_step = 64
    probe = _oracle_chain(oracle, wl, np.arange(rows_per_step), p, threads)
    rows_per_step = int(max(16, min(4096, rows_per_step * budget / max(probe, 1e-6))))
    times = []
    for s in range(args.warmup + args.steps):
        start = (s * 7919 * rows_per_step) % max(1, wl.rows - rows_per_step)
        dt = _oracle_chain(oracle, wl, np.arange(start, start + rows_per_step), p, threads)
        if s >= args.warmup:
            times.append(dt)
    step_s = statistics.fmean(times)
    value = rows_per_step / step_s
    sample = (f"{rows_per_step} consecutive rows of the {wl.name} workload per step, fp64 oracle chain on "
              f"{threads} host threads, input generation untimed")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def prefix(wl, rows: int):
    """The first `rows` tokens of a workload (video rows first), same recipe; 0 = all."""
    import dataclasses
    if rows <= 0 or rows >= wl.rows:
        return wl
    n_video = min(wl.n_video, rows)
    return dataclasses.replace(wl, rows=rows, n_video=n_video, n_audio=rows - n_video,
                               n_outliers=wl.n_outliers * rows // wl.rows)


def workload_config(wl) -> dict:
    return {"workload": f"{wl.name}: {wl.rows} tokens ({wl.n_video} video + {wl.n_audio} audio), hidden "
                        f"{wl.hidden}, {wl.n_heads}x{wl.head_dim} heads, ffn {wl.ffn}, {wl.n_mod} modulation rows",
            "rows": wl.rows, "hidden": wl.hidden, "n_heads": wl.n_heads, "head_dim": wl.head_dim, "ffn": wl.ffn,
            "chain": "rmsnorm_adaln -> qk_rmsnorm_rope_neox -> swiglu",
            "l2": "no flush: every kernel's inputs exceed L2 (129 MB)"}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def _roof(nbytes: int, ms: float, peak_gbs: float) -> dict:
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak_gbs}


def _smi_id(device: torch.device) -> str:
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except (AttributeError, RuntimeError):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[device.index] if device.index < len(ids) else str(device.index)


def run_e2e(chain: Chain, steps: int, ranks: Ranks, chunks: int = 16) -> dict:
    """The same chain through the public API with host buffers.  Every step copies all
    of its inputs from pinned host memory and reads all of its outputs back; the rows
    are cut into `chunks` pieces so that the host-to-device copy of one piece, the
    kernels of the previous one and the device-to-host copy of the one before run
    concurrently on three streams (copy engines in both directions + SMs)."""
    T = chain.wl.rows
    bounds = [T * c // chunks for c in range(chunks + 1)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()
    t, p, wl = chain.tfk, chain.params, chain.wl

    def step():
        go = torch.cuda.Event()
        go.record(main)
        for st in (s_in, s_run, s_out):
            st.wait_event(go)
        last = None
        for c in range(chunks):
            a, b = bounds[c], bounds[c + 1]
            ready, done = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                for k, h in chain.host.items():
                    chain.d[k][a:b].copy_(h[a:b], non_blocking=True)
                ready.record(s_in)
            s_run.wait_event(ready)
            d, o = chain.d, chain.out
            t.tfk_rmsnorm_adaln_indexed(d["x"][a:b], p["w"], p["shift"], p["scale"], d["idx"][a:b], wl.eps,
                                        out=o["y"][a:b], stream=s_run)
            t.tfk_qk_rmsnorm_rope_neox(d["q"][a:b], d["k"][a:b], p["w_q"], p["w_k"], d["pos"][a:b], wl.n_heads,
                                       wl.head_dim, wl.theta, wl.eps, q_out=o["q"][a:b], k_out=o["k"][a:b],
                                       stream=s_run)
            t.tfk_swiglu(d["gate_up"][a:b], out=o["o"][a:b], stream=s_run)
            done.record(s_run)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                for k, dv in o.items():
                    chain.host_out[k][a:b].copy_(dv[a:b], non_blocking=True)
            last = torch.cuda.Event()
            last.record(s_out)
        main.wait_event(last)
        main.wait_stream(s_in)
        main.wait_stream(s_run)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    ranks.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main)
    for _ in range(steps):
        step()
    end.record(main)
    torch.cuda.synchronize()
    ranks.barrier()
    max_s = ranks.max(start.elapsed_time(end) / 1e3)
    return {"value": aggregate(T * steps, ranks.world, max_s), "unit": UNIT,
            "h2d_bytes_per_step": chain.h2d_bytes(), "d2h_bytes_per_step": chain.d2h_bytes(),
            "steps": steps, "ms_per_step": max_s * 1e3 / steps,
            "method": f"pinned host inputs and outputs, {chunks} row chunks pipelined over H2D / kernels / D2H "
                      f"streams, all outputs read back every step"}


def run_tfk(args, ranks: Ranks) -> dict | None:
    import dataclasses

    import rope_tfk_rmsnorm_gb300 as tfk
    tfk.load()  # no library, no run: there is no other implementation to fall back to
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    device = torch.device("cuda", ranks.local_rank)
    torch.cuda.set_device(device)
    wl = prefix(synth.get(args.workload), args.rows)
    if ranks.world > 1:  # weak scaling: each rank its own batch of the same shape
        wl = dataclasses.replace(wl, seed=wl.seed + ranks.rank)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]
    K, W = args.steps, args.warmup

    chain = Chain(tfk, wl, device)
    torch.cuda.synchronize()
    sampler = ClockSampler(_smi_id(device)) if ranks.rank == 0 else None
    total_ms, per_kernel, t0, t1, dist = time_steps(chain, K, W, ranks)
    clocks = sampler.stop(t0, t1) if sampler else None
    max_s = ranks.max(total_ms / 1e3)
    value = aggregate(wl.rows * K, ranks.world, max_s)
    chain_bytes = sum(chain.bytes)
    kernels = {n: dict(_roof(b, ms, peak), tokens_per_s=wl.rows / (ms * 1e-3),
                       ms_p10=d["p10"], ms_median=d["p50"], ms_p90=d["p90"])
               for n, b, ms, d in zip(chain.kernels, chain.bytes, per_kernel, dist)}
    dom = max(range(len(per_kernel)), key=lambda j: per_kernel[j])
    dom_name = chain.kernels[dom]
    src = {"rmsnorm_adaln": "rmsnorm_adaln.cu", "qk_rmsnorm_rope": "qk_rmsnorm_rope.cu", "swiglu": "swiglu.cu"}
    roofline = {"bound": "hbm", "kernel": dom_name, "achieved": kernels[dom_name]["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kernels[dom_name]["frac"],
                "traffic": profiled_traffic(dom_name, wl.name, src[dom_name]) if wl.rows == synth.get(wl.name).rows
                else None,
                "traffic_source": "ncu DRAM bytes of a 16,384-token prefix launch, reads scaled by rows, writes "
                                  "= full algorithmic writes minus the L2-resident remainder "
                                  "(profiles/dram_traffic.txt)",
                "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peaks["source"] == "measured" else "fallback 6.8 TB/s",
                "bytes_per_launch": chain.bytes[dom], "ms_per_launch": per_kernel[dom]}

    e2e = None if args.no_e2e else run_e2e(chain, args.e2e_steps, ranks)
    del chain
    torch.cuda.empty_cache()

    valid = None
    if not args.no_valid_only:
        vo = ValidOnly(tfk, synth.get("valid_only"), device)
        k_vo = max(1, min(K, 200))
        vms, vper, _, _, _ = time_steps(vo, k_vo, W, ranks)
        vmax = ranks.max(vms / 1e3)
        valid = {"workload": f"valid_only: {vo.N} padded rows, {vo.L} valid, hidden {vo.wl.hidden}",
                 "valid_tokens_per_s": aggregate(vo.L * k_vo, ranks.world, vmax), "steps": k_vo,
                 "ms_per_step": vmax * 1e3 / k_vo,
                 "hbm_frac": sum(vo.bytes) / (vmax / k_vo) / 1e9 / peak,
                 "kernels": {n: _roof(b, ms, peak) for n, b, ms in zip(vo.kernels, vo.bytes, vper)}}
        del vo
        torch.cuda.empty_cache()

    cpu = None
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(synth.get(args.workload), args.cpu_seconds)

    if ranks.rank != 0:
        return None
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ranks.world, "steps": K, "warmup": W,
            "ms_per_step": max_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "io_dtype": "bf16", "data": "synthetic (seeded SplitMix64 + Box-Muller inputs)",
            "config": workload_config(wl),
            "hbm": {"achieved_gbs": chain_bytes * K * ranks.world / max_s / 1e9 / ranks.world, "peak_gbs": peak,
                    "frac": chain_bytes * K / max_s / 1e9 / peak, "bytes_per_step": chain_bytes},
            "clocks": clocks, "e2e": e2e, "gpu_launches": 3 * K, "roofline": roofline, "kernels": kernels,
            "valid_only": valid, "cpu_baseline": cpu}


class Rotate:
    """Calls its functions in turn (one per copy of the workload's tensors)."""

    def __init__(self, fns):
        self.fns, self.i = fns, 0

    def __call__(self):
        f = self.fns[self.i]
        self.i = (self.i + 1) % len(self.fns)
        f()


class RotateChain:
    """The chain step over several copies of a workload's tensors in turn."""

    def __init__(self, chains):
        self.chains, self.i = chains, 0
        self.kernels, self.bytes = chains[0].kernels, chains[0].bytes

    def launch(self, ev=None):
        c = self.chains[self.i]
        self.i = (self.i + 1) % len(self.chains)
        c.launch(ev)


class Single:
    """One kernel of a workload as a timed unit (the per-kernel sweep)."""

    def __init__(self, name, nbytes, fn):
        self.kernels, self.bytes, self.fn = [name], [nbytes], fn

    def launch(self, ev=None):
        if ev:
            ev[0].record()
        self.fn()
        if ev:
            ev[1].record()


def graph_ms(unit, reps: int) -> float:
    """Device time per launch of `unit` replayed from one CUDA graph of `reps` launches:
    the same kernels without host submission time (which dominates small workloads)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        unit.launch()                      # warm the library's per-device caches outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    # Captured on the stream of the warm-up call, so that the binding's workspace
    # for that stream (RMSNorm+AdaLN's row counters) exists and the graph uses it.
    with torch.cuda.graph(g, stream=side):
        for _ in range(reps):
            unit.launch()
    g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    g.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / reps


def run_sweep(args, ranks: Ranks):
    """Every kernel on every workload at full size; one JSON line per workload (rank 0)."""
    import rope_tfk_rmsnorm_gb300 as tfk
    tfk.load()
    device = torch.device("cuda", ranks.local_rank)
    torch.cuda.set_device(device)
    peak = measured_peaks()["hbm_gbs"]
    K, W = max(1, min(args.steps, 100)), max(3, args.warmup)
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    import oracle
    oracle.build()
    for name in [w.strip() for w in args.sweep_workloads.split(",") if w.strip()]:
        wl = synth.get(name) if name == "valid_only" else prefix(synth.get(name), args.rows)
        res = {}
        buffer_sets = 1
        if name == "valid_only":
            vo = ValidOnly(tfk, wl, device)
            L, N, hd = vo.L, vo.N, wl.hidden
            fx = lambda: tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(  # noqa: E731
                vo.pad["x"], L, vo.params["w"], vo.params["shift"], vo.params["scale"], vo.idx, wl.eps,
                out=vo.merged["y"])
            fq = lambda: tfk.tfk_qk_rmsnorm_rope_neox_fixed_valid(  # noqa: E731
                vo.pad["q"], vo.pad["k"], L, vo.params["w_q"], vo.params["w_k"], vo.pos, wl.n_heads, wl.head_dim,
                wl.theta, wl.eps, q_out=vo.merged["q"], k_out=vo.merged["k"])
            units = [
                Single("valid_gather", bytes_gather(L, hd), lambda: tfk.tfk_valid_gather(vo.pad["x"], L, compact=vo.comp["x"])),
                Single("zero_tail_merge", bytes_merge(L, N, hd), lambda: tfk.tfk_zero_tail_merge(vo.res["y"], vo.merged["y"])),
                Single("rmsnorm_adaln_fixed_valid", bytes_adaln(L, hd, 2) + 2 * hd * (N - L), fx),
                Single("qk_rmsnorm_rope_fixed_valid", bytes_qk(L, wl.n_heads, wl.head_dim) + 4 * hd * (N - L), fq),
                vo,
            ]
            rows_for = {"valid_gather": L, "zero_tail_merge": L, "rmsnorm_adaln_fixed_valid": L,
                        "qk_rmsnorm_rope_fixed_valid": L}
        else:
            ch = Chain(tfk, wl, device)
            # Small workloads: rotate over enough copies of every tensor that each
            # unit's consecutive launches touch more than twice the L2 (HBM-bound
            # numbers, not L2 hits).
            copies = min(16, max(1, -(-2 * l2_bytes // min(ch.bytes))))
            chs = [ch] + [Chain(tfk, wl, device) for _ in range(copies - 1)]
            makers = [
                lambda c: lambda: tfk.tfk_rmsnorm_adaln_indexed(c.d["x"], c.params["w"], c.params["shift"],
                                                                c.params["scale"], c.d["idx"], wl.eps, out=c.out["y"]),
                lambda c: lambda: tfk.tfk_qk_rmsnorm_rope_neox(c.d["q"], c.d["k"], c.params["w_q"], c.params["w_k"],
                                                               c.d["pos"], wl.n_heads, wl.head_dim, wl.theta, wl.eps,
                                                               q_out=c.out["q"], k_out=c.out["k"]),
                lambda c: lambda: tfk.tfk_swiglu(c.d["gate_up"], out=c.out["o"])]
            units = [Single(n, b, Rotate([mk(c) for c in chs])) for n, b, mk in zip(ch.kernels, ch.bytes, makers)]
            units.append(RotateChain(chs))
            buffer_sets = copies
            rows_for = {}
            if name == "large":  # the Ulysses layouts, 8-way (5 heads per rank)
                P = 8
                qk_bytes = bytes_qk(wl.rows, wl.n_heads, wl.head_dim)
                send_q = torch.empty((P, wl.rows, wl.n_heads // P, wl.head_dim), dtype=torch.bfloat16, device=device)
                send_k = torch.empty_like(send_q)
                units.insert(3, Single("qk_rmsnorm_rope_ulysses_p8", qk_bytes, lambda: tfk.tfk_qk_rmsnorm_rope_neox_ulysses(
                    ch.d["q"], ch.d["k"], ch.params["w_q"], ch.params["w_k"], ch.d["pos"], wl.n_heads, wl.head_dim, P,
                    wl.theta, wl.eps, q_send=send_q, k_send=send_k)))
                units.insert(4, Single("ulysses_pack_p8", 4 * wl.n_heads * wl.head_dim * wl.rows,
                                       lambda: tfk.tfk_ulysses_pack(ch.d["q"], wl.n_heads, wl.head_dim, P, dst=send_q)))
                units.insert(5, Single("ulysses_unpack_p8", 4 * wl.n_heads * wl.head_dim * wl.rows,
                                       lambda: tfk.tfk_ulysses_unpack(send_q, wl.n_heads, wl.head_dim, P, dst=ch.out["q"])))
        for u in units:
            with torch.cuda.nvtx.range(u.kernels[0] if len(u.kernels) == 1 else "chain"):  # ncu --nvtx-include
                total, per, _, _, _ = time_steps(u, K, W, ranks)
                gms = graph_ms(u, K)
            if len(u.kernels) == 1:
                ms = per[0]
                rows = rows_for.get(u.kernels[0], wl.rows)
                res[u.kernels[0]] = dict(_roof(u.bytes[0], ms, peak), tokens_per_s=rows / (ms * 1e-3),
                                         graph_ms=gms, graph_frac=_roof(u.bytes[0], gms, peak)["frac"])
            else:
                ms = total / K
                rows = vo.L if name == "valid_only" else wl.rows
                res["chain" if name != "valid_only" else "valid_only_pipeline"] = dict(
                    _roof(sum(u.bytes), ms, peak), tokens_per_s=rows / (ms * 1e-3),
                    graph_ms=gms, graph_frac=_roof(sum(u.bytes), gms, peak)["frac"], kernels=u.kernels)
        if ranks.rank == 0:
            print(json.dumps({"sweep": name, "workload": workload_config(wl)["workload"], "steps": K,
                              "peak_gbs": peak, "buffer_sets": buffer_sets, "results": res,
                              "oracle": oracle_rates(wl)}), flush=True)
        del units
        if name != "valid_only":
            ch = chs = None
        torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    ranks = Ranks()
    try:
        if args.sweep:
            run_sweep(args, ranks)
            return
        out = run_reference(args, ranks) if args.impl == "reference" else run_tfk(args, ranks)
        if out is not None:
            print(json.dumps(out), flush=True)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
