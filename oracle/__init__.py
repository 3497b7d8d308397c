"""fp64 CPU oracle for the fused DiT-block elementwise path (numpy front end).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import this package; the library
under ``rope_tfk_rmsnorm_gb300`` never does, and nothing here imports it.
The arithmetic lives in ``oracle.c`` (plain loops in double precision); this
file only marshals numpy arrays and optionally splits rows over threads.

Every function returns unrounded float64 results; ``round_bf16`` applies the
single final rounding (nearest, ties to even).  bf16 arrays are numpy
``uint16`` arrays of raw bits.  Pins against the definitions live in
``tests/test_oracle_pins.py``; every function here is pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place with gcc (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def bind(path: str):
    """Load a compiled oracle library from `path` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
    sig = {
        "oracle_bf16_to_f64": (dbl, [ctypes.c_uint16]),
        "oracle_f64_to_bf16": (ctypes.c_uint16, [dbl]),
        "oracle_round_bf16": (None, [vp, i64, vp]),
        "oracle_rmsnorm_adaln_indexed": (None, [vp, i64, i64, i32, vp, vp, vp, vp, i32, dbl, vp]),
        "oracle_head_rmsnorm": (None, [vp, i64, i64, i32, i32, vp, dbl, vp]),
        "oracle_rope_neox": (None, [vp, vp, i64, i32, i32, dbl]),
        "oracle_qk_rmsnorm_rope_neox": (None, [vp, vp, i64, i64, i32, i32, vp, vp, vp, dbl, dbl, vp, vp]),
        "oracle_swiglu": (None, [vp, i64, i64, i32, vp]),
        "oracle_valid_gather": (None, [vp, i64, i32, vp]),
        "oracle_zero_tail_merge": (None, [vp, i64, i64, i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind(_LIB)
    return _lib


def _p(a: np.ndarray, offset_elems: int = 0):
    return ctypes.c_void_p(a.ctypes.data + offset_elems * a.itemsize)


def _rows2d(a: np.ndarray, dtype) -> tuple[np.ndarray, int]:
    """A 2-D array whose columns are contiguous; returns it with its row stride in elements."""
    assert a.ndim == 2 and a.dtype == dtype, (a.shape, a.dtype)
    if a.strides[1] != a.itemsize or a.strides[0] % a.itemsize:
        a = np.ascontiguousarray(a)
    return a, a.strides[0] // a.itemsize


def _split(rows: int, threads: int):
    threads = max(1, min(threads, rows))
    per = (rows + threads - 1) // threads
    return [(s, min(rows, s + per)) for s in range(0, rows, per)]


def _run(fn_rows, rows: int, threads: int):
    if threads <= 1 or rows < 2:
        fn_rows(0, rows)
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda se: fn_rows(*se), _split(rows, threads)))


# ---- conversions ----------------------------------------------------------

def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(v: np.ndarray, threads: int = 1) -> np.ndarray:
    """fp64 -> bf16 bits, nearest with ties to even (one rounding); `threads` splits the
    elements over host threads (the result does not depend on the split)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    if v.size:
        lib = _load()

        def part(s, e):
            if e > s:
                lib.oracle_round_bf16(_p(v, s), e - s, _p(out, s))
        _run(part, v.size, threads)
    return out


# ---- the five operations ---------------------------------------------------

def rmsnorm_adaln_indexed(x: np.ndarray, weight: np.ndarray, shift: np.ndarray, scale: np.ndarray,
                          mod_idx: np.ndarray, eps: float, hidden: int | None = None,
                          threads: int = 1) -> np.ndarray:
    """RMSNorm of each row, times weight, then (1 + scale[m]) and + shift[m], m = mod_idx[row]."""
    x, stride = _rows2d(x, np.uint16)
    rows = x.shape[0]
    hidden = x.shape[1] if hidden is None else hidden
    weight = np.ascontiguousarray(weight, dtype=np.float32)
    shift = np.ascontiguousarray(shift, dtype=np.float32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    mod_idx = np.ascontiguousarray(mod_idx, dtype=np.int32)
    n_mod = shift.shape[0]
    assert weight.shape == (hidden,) and shift.shape == scale.shape == (n_mod, hidden)
    assert mod_idx.shape == (rows,) and (rows == 0 or (mod_idx.min() >= 0 and mod_idx.max() < n_mod))
    y = np.empty((rows, hidden), dtype=np.float64)
    lib = _load()

    def part(s, e):
        if e > s:
            lib.oracle_rmsnorm_adaln_indexed(_p(x, s * stride), stride, e - s, hidden, _p(weight),
                                             _p(shift), _p(scale), _p(mod_idx, s), n_mod, eps,
                                             _p(y, s * hidden))
    _run(part, rows, threads)
    return y


def head_rmsnorm(v: np.ndarray, n_heads: int, head_dim: int, weight: np.ndarray, eps: float,
                 threads: int = 1) -> np.ndarray:
    """Per-head RMSNorm of v [rows, >= n_heads*head_dim] -> float64 [rows, n_heads, head_dim]."""
    v, stride = _rows2d(v, np.uint16)
    rows = v.shape[0]
    weight = np.ascontiguousarray(weight, dtype=np.float32)
    assert weight.shape == (head_dim,)
    out = np.empty((rows, n_heads, head_dim), dtype=np.float64)
    lib = _load()

    def part(s, e):
        if e > s:
            lib.oracle_head_rmsnorm(_p(v, s * stride), stride, e - s, n_heads, head_dim, _p(weight),
                                    eps, _p(out, s * n_heads * head_dim))
    _run(part, rows, threads)
    return out


def rope_neox(v: np.ndarray, pos: np.ndarray, base: float, threads: int = 1) -> np.ndarray:
    """NeoX rotate-half RoPE of float64 v [rows, n_heads, head_dim] (returns a new array)."""
    out = np.array(v, dtype=np.float64, order="C", copy=True)
    rows, n_heads, head_dim = out.shape
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert pos.shape == (rows,)
    lib = _load()

    def part(s, e):
        if e > s:
            lib.oracle_rope_neox(_p(out, s * n_heads * head_dim), _p(pos, s), e - s, n_heads,
                                 head_dim, base)
    _run(part, rows, threads)
    return out


def qk_rmsnorm_rope_neox(q: np.ndarray, k: np.ndarray, q_weight: np.ndarray, k_weight: np.ndarray,
                         pos: np.ndarray, n_heads: int, head_dim: int, base: float, eps: float,
                         threads: int = 1):
    """(RoPE(head_rmsnorm(q)), RoPE(head_rmsnorm(k))) as float64 [rows, n_heads, head_dim]."""
    q, qs = _rows2d(q, np.uint16)
    k, ks = _rows2d(k, np.uint16)
    assert qs == ks and q.shape[0] == k.shape[0]
    rows = q.shape[0]
    q_weight = np.ascontiguousarray(q_weight, dtype=np.float32)
    k_weight = np.ascontiguousarray(k_weight, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    qo = np.empty((rows, n_heads, head_dim), dtype=np.float64)
    ko = np.empty_like(qo)
    lib = _load()
    hd = n_heads * head_dim

    def part(s, e):
        if e > s:
            lib.oracle_qk_rmsnorm_rope_neox(_p(q, s * qs), _p(k, s * ks), qs, e - s, n_heads, head_dim,
                                            _p(q_weight), _p(k_weight), _p(pos, s), base, eps,
                                            _p(qo, s * hd), _p(ko, s * hd))
    _run(part, rows, threads)
    return qo, ko


def swiglu(gate_up: np.ndarray, ffn: int | None = None, threads: int = 1) -> np.ndarray:
    """silu(gate) * up for gate_up [rows, 2*ffn] = [gate | up] -> float64 [rows, ffn]."""
    gate_up, stride = _rows2d(gate_up, np.uint16)
    rows = gate_up.shape[0]
    ffn = gate_up.shape[1] // 2 if ffn is None else ffn
    out = np.empty((rows, ffn), dtype=np.float64)
    lib = _load()

    def part(s, e):
        if e > s:
            lib.oracle_swiglu(_p(gate_up, s * stride), stride, e - s, ffn, _p(out, s * ffn))
    _run(part, rows, threads)
    return out


def valid_gather(padded: np.ndarray, valid_rows: int) -> np.ndarray:
    """The first valid_rows rows of padded [N, hidden] (bit copy)."""
    padded = np.ascontiguousarray(padded, dtype=np.uint16)
    hidden = padded.shape[1]
    assert 0 <= valid_rows <= padded.shape[0]
    out = np.empty((valid_rows, hidden), dtype=np.uint16)
    if valid_rows and hidden:
        _load().oracle_valid_gather(_p(padded), valid_rows, hidden, _p(out))
    return out


def zero_tail_merge(compact: np.ndarray, padded_rows: int) -> np.ndarray:
    """compact [L, hidden] written into a [padded_rows, hidden] buffer whose tail rows are +0.0."""
    compact = np.ascontiguousarray(compact, dtype=np.uint16)
    valid_rows, hidden = compact.shape
    assert valid_rows <= padded_rows
    out = np.empty((padded_rows, hidden), dtype=np.uint16)
    if padded_rows and hidden:
        _load().oracle_zero_tail_merge(_p(compact), valid_rows, padded_rows, hidden, _p(out))
    return out


# ---- fixed-valid mode: the same definitions on the valid prefix, +0.0 after it ----

def rmsnorm_adaln_fixed_valid(x_padded: np.ndarray, valid_rows: int, weight, shift, scale, mod_idx, eps,
                              threads: int = 1) -> np.ndarray:
    """rmsnorm_adaln_indexed on rows [0, valid_rows); +0.0 on the rest of the padded rows."""
    out = np.zeros((x_padded.shape[0], x_padded.shape[1]), dtype=np.float64)
    out[:valid_rows] = rmsnorm_adaln_indexed(x_padded[:valid_rows], weight, shift, scale,
                                             np.asarray(mod_idx)[:valid_rows], eps, threads=threads)
    return out


def qk_rmsnorm_rope_neox_fixed_valid(q_padded, k_padded, valid_rows: int, q_weight, k_weight, pos,
                                     n_heads: int, head_dim: int, base: float, eps: float, threads: int = 1):
    """qk_rmsnorm_rope_neox on rows [0, valid_rows); +0.0 on the rest of the padded rows."""
    shape = (q_padded.shape[0], n_heads, head_dim)
    qo, ko = np.zeros(shape), np.zeros(shape)
    qo[:valid_rows], ko[:valid_rows] = qk_rmsnorm_rope_neox(q_padded[:valid_rows], k_padded[:valid_rows],
                                                            q_weight, k_weight, np.asarray(pos)[:valid_rows],
                                                            n_heads, head_dim, base, eps, threads=threads)
    return qo, ko


# ---- Ulysses relayout (TeleFuser PR #23, section Changes Made; packing fused into
#      Q/K RMSNorm + RoPE, TeleFuser PR #38, section 2) ----

def ulysses_pack(rows_layout: np.ndarray, n_heads: int, head_dim: int, sp_degree: int) -> np.ndarray:
    """[rows, n_heads*head_dim] -> [sp_degree, rows, n_heads/sp_degree, head_dim]: block p holds the
    heads p*H/P .. (p+1)*H/P - 1 of every row, the block that sequence-parallel rank p receives."""
    rows = rows_layout.shape[0]
    a = np.asarray(rows_layout)[:, :n_heads * head_dim].reshape(rows, sp_degree, n_heads // sp_degree, head_dim)
    return np.ascontiguousarray(a.transpose(1, 0, 2, 3))


def ulysses_unpack(grouped: np.ndarray, n_heads: int, head_dim: int, sp_degree: int) -> np.ndarray:
    """Inverse of ulysses_pack: [sp_degree, rows, n_heads/sp_degree, head_dim] -> [rows, n_heads*head_dim]."""
    g = np.asarray(grouped).reshape(sp_degree, -1, n_heads // sp_degree, head_dim)
    return np.ascontiguousarray(g.transpose(1, 0, 2, 3)).reshape(g.shape[1], n_heads * head_dim)
