"""Seeded synthetic inputs for the fused DiT-block elementwise path.

This module is the one thing the CUDA path's tests and the oracle share: it
draws the inputs and knows the shape and structure of each workload, and it
holds none of the arithmetic of either side (no normalisation, rotation,
activation or rounding of results).  Values are counter-based (SplitMix64 +
Box-Muller, see ``synth.c``), so any subset of rows can be regenerated alone
and equals the same rows of the full tensor bit for bit.

bf16 tensors are returned as numpy ``uint16`` arrays of raw bf16 bits.

Workloads (packed video+audio token buffers of a joint audio-video DiT, as the
MiniMax H3 integration page describes: "packed joint video/audio denoising",
"independent modality schedules"):

* ``tiny``       320 rows (256 video + 64 audio), hidden 512, 8x64 heads, ffn 1024
* ``medium``     8192 rows (7168 + 1024), hidden 3072, 24x128, ffn 8192,
                 4 modulation rows picked per token (modality x coin flip),
                 positions restart at 0 for the audio rows
* ``valid_only`` 32768 padded rows, valid prefix L uniform in [24000, 32768],
                 hidden 3072, 24x128; padded tail rows hold bf16 NaN
* ``large``      75600 rows (73728 + 1872), hidden 5120, 40x128, ffn 13824,
                 756 outlier rows (1%) scaled by 50 in every activation input
* ``per_frame``  56320 rows (27 frames x 2048 video + 1024 audio), hidden 4096,
                 32x128, ffn 11008, modulation index = frame id, 27 for audio
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

SEED = 0
EPS = 1e-6
THETA = 10000.0
BF16_NAN = 0x7FC0
CANARY = 0xFFFF

TAGS = {"x": 1, "w": 2, "shift": 3, "scale": 4, "q": 5, "k": 6, "w_q": 7, "w_k": 8,
        "gate_up": 9, "idx": 10, "outlier": 11, "valid_len": 12, "sample": 13}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libsynth.so in place (plain C, no GPU)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, u64, dbl, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            lib.synth_u64.restype = u64
            lib.synth_u64.argtypes = [u64, u64, u64]
            for fn in (lib.synth_normal_bf16, lib.synth_normal_f32):
                fn.restype = None
                fn.argtypes = [u64, u64, i64, i64, i64, dbl, dbl, vp, vp, ctypes.c_int]
            lib.synth_uniform_int.restype = None
            lib.synth_uniform_int.argtypes = [u64, u64, i64, i64, i64, vp]
            lib.synth_permutation.restype = None
            lib.synth_permutation.argtypes = [u64, u64, i64, vp]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def u64(tag: str, i: int, seed: int = SEED) -> int:
    return int(_load().synth_u64(seed, TAGS[tag], i))


def normal_bf16(tag: str, row0: int, rows: int, cols: int, mean: float, std: float,
                row_scale: np.ndarray | None = None, seed: int = SEED, out: np.ndarray | None = None):
    """Rows [row0, row0+rows) of a seeded [*, cols] bf16 matrix (raw uint16 bits)."""
    if out is None:
        out = np.empty((rows, cols), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.shape == (rows, cols)
    rs = None
    if row_scale is not None:
        row_scale = np.ascontiguousarray(row_scale, dtype=np.float32)
        assert row_scale.shape == (rows,)
        rs = _ptr(row_scale)
    if rows and cols:
        _load().synth_normal_bf16(seed, TAGS[tag], row0, rows, cols, mean, std, rs, _ptr(out), _threads())
    return out


def normal_f32(tag: str, rows: int, cols: int, mean: float, std: float, seed: int = SEED):
    out = np.empty((rows, cols), dtype=np.float32)
    if rows and cols:
        _load().synth_normal_f32(seed, TAGS[tag], 0, rows, cols, mean, std, None, _ptr(out), 1)
    return out


def uniform_int(tag: str, n: int, lo: int, hi: int, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if n:
        _load().synth_uniform_int(seed, TAGS[tag], n, lo, hi, _ptr(out))
    return out


def permutation(tag: str, n: int, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if n:
        _load().synth_permutation(seed, TAGS[tag], n, _ptr(out))
    return out


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    rows: int            # token rows (padded rows N for valid_only)
    n_video: int
    n_audio: int
    hidden: int
    n_heads: int
    head_dim: int
    ffn: int             # 0: no SwiGLU step in this workload
    n_mod: int
    mod_std: float
    n_outliers: int = 0
    outlier_gain: float = 50.0
    frame_rows: int = 0  # per-frame modulation: video rows per frame
    seed: int = SEED
    eps: float = EPS
    theta: float = THETA


WORKLOADS = {
    "tiny": Workload("tiny", 320, 256, 64, 512, 8, 64, 1024, 2, 0.1),
    "medium": Workload("medium", 8192, 7168, 1024, 3072, 24, 128, 8192, 4, 0.1),
    "valid_only": Workload("valid_only", 32768, 32768, 0, 3072, 24, 128, 0, 2, 0.1),
    "large": Workload("large", 75600, 73728, 1872, 5120, 40, 128, 13824, 2, 0.1, n_outliers=756),
    "per_frame": Workload("per_frame", 56320, 55296, 1024, 4096, 32, 128, 11008, 28, 0.2,
                          frame_rows=2048),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def custom(name: str, rows: int, hidden: int, n_heads: int, head_dim: int, ffn: int,
           n_mod: int = 2, n_audio: int = 0, mod_std: float = 0.1, n_outliers: int = 0,
           seed: int = SEED) -> Workload:
    """An ad-hoc workload (ragged sizes, edge cases) with the same recipe."""
    return Workload(name, rows, rows - n_audio, n_audio, hidden, n_heads, head_dim, ffn, n_mod,
                    mod_std, n_outliers=n_outliers, seed=seed)


def valid_len(wl: Workload) -> int:
    """Valid prefix length L of the padded buffer, uniform in [24000, 32768]."""
    if wl.name != "valid_only":
        return wl.rows
    return int(uniform_int("valid_len", 1, 24000, 32768, seed=wl.seed)[0])


def _rows(wl: Workload, rows) -> np.ndarray:
    if rows is None:
        return np.arange(wl.rows, dtype=np.int64)
    return np.asarray(rows, dtype=np.int64)


def mod_index(wl: Workload, rows=None) -> np.ndarray:
    """Per-token modulation row index (int32)."""
    r = _rows(wl, rows)
    is_audio = r >= wl.n_video
    if wl.name == "medium":
        bits = _coin_bits(wl, r)
        return (2 * is_audio + bits).astype(np.int32)
    if wl.frame_rows:
        return np.where(is_audio, wl.n_mod - 1, r // wl.frame_rows).astype(np.int32)
    if wl.name == "valid_only":
        L = valid_len(wl)
        return (r >= L - L // 8).astype(np.int32)
    if wl.n_mod == 1:
        return np.zeros(len(r), dtype=np.int32)
    return np.where(is_audio, 1, 0).astype(np.int32) % wl.n_mod


def _coin_bits(wl: Workload, r: np.ndarray) -> np.ndarray:
    lib = _load()
    out = np.empty(len(r), dtype=np.int64)
    for j, i in enumerate(r):
        out[j] = lib.synth_u64(wl.seed, TAGS["idx"], int(i)) >> 63
    return out


def positions(wl: Workload, rows=None) -> np.ndarray:
    """Per-token RoPE position (int32); the audio block restarts at 0 in ``medium``."""
    r = _rows(wl, rows)
    if wl.name == "medium":
        return np.where(r >= wl.n_video, r - wl.n_video, r).astype(np.int32)
    return r.astype(np.int32)


def outlier_rows(wl: Workload) -> np.ndarray:
    if not wl.n_outliers:
        return np.zeros(0, dtype=np.int64)
    return np.sort(permutation("outlier", wl.rows, seed=wl.seed)[: wl.n_outliers])


def row_scale(wl: Workload, rows=None) -> np.ndarray | None:
    if not wl.n_outliers:
        return None
    r = _rows(wl, rows)
    s = np.ones(len(r), dtype=np.float32)
    s[np.isin(r, outlier_rows(wl))] = wl.outlier_gain
    return s


def activation(wl: Workload, tag: str, rows=None, out: np.ndarray | None = None) -> np.ndarray:
    """Rows of an activation input: 'x' [*, hidden], 'q'/'k' [*, H*D], 'gate_up' [*, 2*ffn].

    Values ~ N(0, 1) (times the outlier gain on outlier rows), rounded to bf16.
    In ``valid_only`` the padded tail rows (>= L) are bf16 NaN.
    """
    cols = {"x": wl.hidden, "q": wl.n_heads * wl.head_dim, "k": wl.n_heads * wl.head_dim,
            "gate_up": 2 * wl.ffn}[tag]
    r = _rows(wl, rows)
    if out is None:
        out = np.empty((len(r), cols), dtype=np.uint16)
    if len(r) == 0:
        return out
    rs = row_scale(wl, r)
    # generate each run of consecutive rows with one call
    breaks = np.flatnonzero(np.diff(r) != 1) + 1
    starts = np.concatenate([[0], breaks])
    ends = np.concatenate([breaks, [len(r)]])
    for s, e in zip(starts, ends):
        normal_bf16(tag, int(r[s]), int(e - s), cols, 0.0, 1.0,
                    None if rs is None else rs[s:e], seed=wl.seed, out=out[s:e])
    if wl.name == "valid_only":
        out[r >= valid_len(wl)] = BF16_NAN
    return out


def params(wl: Workload) -> dict:
    """fp32 parameters: norm weight w [hidden] ~ 1+0.1N, shift/scale [n_mod, hidden] ~ std*N,
    per-head Q/K norm weights w_q, w_k [head_dim] ~ 1+0.1N."""
    return {
        "w": normal_f32("w", 1, wl.hidden, 1.0, 0.1, wl.seed)[0],
        "shift": normal_f32("shift", wl.n_mod, wl.hidden, 0.0, wl.mod_std, wl.seed),
        "scale": normal_f32("scale", wl.n_mod, wl.hidden, 0.0, wl.mod_std, wl.seed),
        "w_q": normal_f32("w_q", 1, wl.head_dim, 1.0, 0.1, wl.seed)[0],
        "w_k": normal_f32("w_k", 1, wl.head_dim, 1.0, 0.1, wl.seed)[0],
    }


def sample_rows(wl: Workload, n: int, limit: int | None = None, tag: str = "sample") -> np.ndarray:
    """A seeded, sorted sample of row indices in [0, limit) that always contains the first
    and last rows, both modality boundaries and a few outlier rows."""
    limit = wl.rows if limit is None else limit
    if limit <= n:
        return np.arange(limit, dtype=np.int64)
    picks = set(int(i) for i in uniform_int(tag, n, 0, limit - 1, seed=wl.seed))
    picks |= {0, 1, limit - 2, limit - 1}
    for b in (wl.n_video - 1, wl.n_video):
        if 0 <= b < limit:
            picks.add(b)
    if wl.frame_rows:
        for f in range(1, wl.n_video // wl.frame_rows):
            if f * wl.frame_rows < limit:
                picks |= {f * wl.frame_rows - 1, f * wl.frame_rows}
    for o in outlier_rows(wl)[:8]:
        if o < limit:
            picks.add(int(o))
    return np.array(sorted(picks), dtype=np.int64)
