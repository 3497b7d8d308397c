"""bench.py's output contract, checked without a GPU: the reference arm (the
fp64 oracle on the host cores) prints one JSON line with the keys the driver
reads, and the algorithmic byte counts match their per-token definitions."""
import contextlib
import io
import json

import bench
import synth


def _run(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(argv)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    out = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
                "--ref-seconds", "1"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["impl"] == "reference" and out["metric"] == bench.METRIC and out["unit"] == "tokens/s"
    assert out["value"] > 0 and out["ms_per_step"] > 0 and out["higher_is_better"] is True
    assert out["steps"] == 2 and out["warmup"] == 1 and out["n_gpus"] == 1 and out["vs_baseline"] is None
    assert out["config"]["workload"].startswith("tiny:") and out["config"]["rows"] == 320
    assert "model" not in out["config"]
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"] and cb["sample"]
    assert out["e2e"] == {"value": out["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_per_token():
    """Per-token bytes of the 75,600-token workload: RMSNorm+AdaLN reads and writes
    a bf16 row and a 4-byte index, Q/K reads and writes two rows of 40 x 128
    and a 4-byte position, SwiGLU reads 2 x 13824 and writes 13824 values."""
    wl = synth.get("large")
    T, hd = wl.rows, wl.hidden
    assert bench.bytes_adaln(T, hd, 2) - (4 * hd + 8 * hd * 2) == T * 20484
    assert bench.bytes_qk(T, wl.n_heads, wl.head_dim) - 8 * wl.head_dim == T * 40964
    assert bench.bytes_swiglu(T, wl.ffn) == T * 82944
    assert bench.bytes_gather(100, 3072) == 100 * 12288
    assert bench.bytes_merge(100, 128, 3072) == 2 * 3072 * 228


def test_prefix_keeps_the_recipe():
    wl = synth.get("large")
    p = bench.prefix(wl, 16384)
    assert p.rows == 16384 and p.n_video == 16384 and p.n_audio == 0 and p.hidden == wl.hidden
    assert bench.prefix(wl, 0) is wl and bench.prefix(wl, 10 ** 9) is wl


def test_aggregate_is_whole_job_throughput():
    assert bench.aggregate(1000, 1, 2.0) == 500.0
    assert bench.aggregate(1000, 4, 2.0) == 2000.0


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks launched the way the driver launches N > 1 (gloo on CPU): rank 0
    prints the one line, the other rank exits 0 without output."""
    import os
    import socket
    import subprocess
    import sys

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-seconds", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
