"""Python binding of libtfk, the GB300 (sm_103a) fused DiT-block elementwise kernels.

Argument marshalling only: every function below checks tensor dtypes and
layouts, allocates the output with PyTorch when none is given, and passes raw
device pointers, sizes and the current CUDA stream to the C ABI of the same
name (``include/tfk.h``).  All arithmetic runs in the CUDA kernels; there is
no CPU fallback.  If ``libtfk.so`` is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtfk.so")

TFK_OK = 0
STATUS = {0: "TFK_OK", 1: "TFK_ERR_INVALID_ARGUMENT", 2: "TFK_ERR_MISALIGNED",
          3: "TFK_ERR_UNSUPPORTED", 4: "TFK_ERR_CUDA"}

# (name, restype, argtypes) of every symbol include/tfk.h declares
_vp, _i64, _i32, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
SIGNATURES = [
    ("tfk_abi_version", ctypes.c_int, []),
    ("tfk_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("tfk_last_error_message", ctypes.c_char_p, []),
    ("tfk_debug_fail_next_launch", ctypes.c_int, [_i32]),
    ("tfk_rmsnorm_adaln_indexed", ctypes.c_int,
     [_vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _f32, _vp, _vp]),
    ("tfk_rmsnorm_adaln_indexed_noalloc", ctypes.c_int,
     [_vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _f32, _vp]),
    ("tfk_qk_rmsnorm_rope_neox", ctypes.c_int,
     [_vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _vp]),
    ("tfk_rmsnorm_adaln_indexed_fixed_valid", ctypes.c_int,
     [_vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _f32, _vp, _vp]),
    ("tfk_qk_rmsnorm_rope_neox_fixed_valid", ctypes.c_int,
     [_vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _f32, _f32, _vp]),
    ("tfk_qk_rmsnorm_rope_neox_ulysses", ctypes.c_int,
     [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _f32, _f32, _vp]),
    ("tfk_ulysses_pack", ctypes.c_int, [_vp, _i64, _vp, _i64, _i32, _i32, _i32, _vp]),
    ("tfk_ulysses_unpack", ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp]),
    ("tfk_swiglu", ctypes.c_int, [_vp, _i64, _vp, _i64, _i64, _i32, _vp]),
    ("tfk_valid_gather", ctypes.c_int, [_vp, _vp, _i64, _i32, _vp]),
    ("tfk_zero_tail_merge", ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _vp]),
    ("tfk_velocity_cache_schedule", ctypes.c_int,
     [_i32, ctypes.c_double, ctypes.c_double, _i32, _i32, _vp, _vp]),
]

_lock = threading.Lock()
_lib = None

RMSNORM_WORKSPACE_BYTES = 2304  # TFK_RMSNORM_WORKSPACE_BYTES
_ws_lock = threading.Lock()
_ws: dict = {}  # (device index, stream handle) -> zeroed int64 tensor of the RMSNorm workspace


class TfkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libtfk.so (built by ``__graft_entry__.build()`` or ``build.py``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libtfk.so not built at {LIB_PATH}; run __graft_entry__.build()")
            lib = ctypes.CDLL(LIB_PATH)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int):
    if status != TFK_OK:
        raise TfkError(status, load().tfk_last_error_message().decode())


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        return torch.cuda.current_stream(t.device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int:
    return 0 if t is None else t.data_ptr()


def _workspace(device: torch.device, stream: int, workspace) -> int:
    """Device address of the RMSNorm workspace for a call on `stream`.

    workspace=None: one zeroed workspace per (device, stream), made on first use
    (its zero-fill ordered on that stream) and kept; calls on one stream never
    overlap, and every completed call leaves it zero.  No new one is made while a
    stream is being captured into a graph (the call then runs without one).
    workspace=False or 0: none.  A tensor: its own storage (CUDA, at least
    RMSNORM_WORKSPACE_BYTES bytes, zero before its first use)."""
    if workspace is None:
        key = (device.index, stream)
        ws = _ws.get(key)
        if ws is None:
            if torch.cuda.is_current_stream_capturing():
                return 0
            with _ws_lock:
                ws = _ws.get(key)
                if ws is None:
                    with torch.cuda.stream(torch.cuda.ExternalStream(stream, device=device)):
                        ws = torch.zeros(RMSNORM_WORKSPACE_BYTES // 8, dtype=torch.int64, device=device)
                    _ws[key] = ws
        return ws.data_ptr()
    if workspace is False or (isinstance(workspace, int) and workspace == 0):
        return 0
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or \
            workspace.numel() * workspace.element_size() < RMSNORM_WORKSPACE_BYTES:
        raise ValueError(f"workspace must be a CUDA tensor of at least {RMSNORM_WORKSPACE_BYTES} bytes")
    return workspace.data_ptr()


def _rows(t: torch.Tensor, name: str, dtype=torch.bfloat16) -> int:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with contiguous columns, got shape {tuple(t.shape)} "
                         f"strides {t.stride()}")
    return t.stride(0)


def _param(t: torch.Tensor, name: str, dtype=torch.float32):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def abi_version() -> int:
    return load().tfk_abi_version()


def tfk_rmsnorm_adaln_indexed(x: torch.Tensor, weight: torch.Tensor, shift: torch.Tensor,
                              scale: torch.Tensor, mod_idx: torch.Tensor, eps: float = 1e-6,
                              out: torch.Tensor | None = None, stream=None, workspace=None) -> torch.Tensor:
    """y = RMSNorm(x) * weight * (1 + scale[mod_idx]) + shift[mod_idx]; x, y [rows, hidden] bf16.
    `workspace`: see _workspace (default: one per stream, managed here)."""
    xs = _rows(x, "x")
    rows, hidden = x.shape
    for t, n in ((weight, "weight"), (shift, "shift"), (scale, "scale")):
        _param(t, n)
    _param(mod_idx, "mod_idx", torch.int32)
    if out is None:
        out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=x.device)
    ys = _rows(out, "out")
    st = _stream(x, stream)
    _check(load().tfk_rmsnorm_adaln_indexed(_ptr(x), xs, _ptr(out), ys, _ptr(weight), _ptr(shift),
                                            _ptr(scale), _ptr(mod_idx), shift.shape[0] if shift.dim() == 2 else 1,
                                            rows, hidden, eps, _workspace(x.device, st, workspace), st))
    return out


def tfk_rmsnorm_adaln_indexed_noalloc(x: torch.Tensor, weight: torch.Tensor, shift: torch.Tensor,
                                      scale: torch.Tensor, mod_idx: torch.Tensor, out: torch.Tensor,
                                      eps: float = 1e-6, stream=None) -> torch.Tensor:
    """tfk_rmsnorm_adaln_indexed into a caller-given `out`, with no workspace and no allocation
    (the row counters live in an array of the library; calls that overlap on one GPU race)."""
    xs = _rows(x, "x")
    rows, hidden = x.shape
    for t, n in ((weight, "weight"), (shift, "shift"), (scale, "scale")):
        _param(t, n)
    _param(mod_idx, "mod_idx", torch.int32)
    ys = _rows(out, "out")
    _check(load().tfk_rmsnorm_adaln_indexed_noalloc(_ptr(x), xs, _ptr(out), ys, _ptr(weight), _ptr(shift),
                                                    _ptr(scale), _ptr(mod_idx),
                                                    shift.shape[0] if shift.dim() == 2 else 1, rows, hidden, eps,
                                                    _stream(x, stream)))
    return out


def tfk_qk_rmsnorm_rope_neox(q: torch.Tensor, k: torch.Tensor, q_weight: torch.Tensor,
                             k_weight: torch.Tensor, positions: torch.Tensor, n_heads: int,
                             head_dim: int, theta: float = 10000.0, eps: float = 1e-6,
                             q_out: torch.Tensor | None = None, k_out: torch.Tensor | None = None,
                             stream=None):
    """Per-head RMSNorm then NeoX RoPE of q and k [rows, >= n_heads*head_dim] (same row stride)."""
    qs, ks = _rows(q, "q"), _rows(k, "k")
    if qs != ks or q.shape[0] != k.shape[0]:
        raise ValueError("q and k must have the same rows and row stride")
    rows = q.shape[0]
    width = n_heads * head_dim
    _param(q_weight, "q_weight")
    _param(k_weight, "k_weight")
    _param(positions, "positions", torch.int32)
    if q_out is None:
        q_out = torch.empty((rows, width), dtype=torch.bfloat16, device=q.device)
    if k_out is None:
        k_out = torch.empty((rows, width), dtype=torch.bfloat16, device=q.device)
    qos, kos = _rows(q_out, "q_out"), _rows(k_out, "k_out")
    if qos != kos:
        raise ValueError("q_out and k_out must have the same row stride")
    _check(load().tfk_qk_rmsnorm_rope_neox(_ptr(q), _ptr(k), qs, _ptr(q_out), _ptr(k_out), qos,
                                           _ptr(q_weight), _ptr(k_weight), _ptr(positions), rows,
                                           n_heads, head_dim, theta, eps, _stream(q, stream)))
    return q_out, k_out


def tfk_rmsnorm_adaln_indexed_fixed_valid(x: torch.Tensor, valid_rows: int, weight: torch.Tensor,
                                          shift: torch.Tensor, scale: torch.Tensor, mod_idx: torch.Tensor,
                                          eps: float = 1e-6, out: torch.Tensor | None = None,
                                          stream=None, workspace=None) -> torch.Tensor:
    """Fixed-valid RMSNorm+AdaLN on a padded buffer x [padded_rows, hidden]: rows < valid_rows
    as tfk_rmsnorm_adaln_indexed, the rest of out written +0.0; mod_idx holds valid_rows entries."""
    xs = _rows(x, "x")
    padded, hidden = x.shape
    for t, n in ((weight, "weight"), (shift, "shift"), (scale, "scale")):
        _param(t, n)
    _param(mod_idx, "mod_idx", torch.int32)
    if out is None:
        out = torch.empty((padded, hidden), dtype=torch.bfloat16, device=x.device)
    ys = _rows(out, "out")
    st = _stream(x, stream)
    _check(load().tfk_rmsnorm_adaln_indexed_fixed_valid(
        _ptr(x), xs, _ptr(out), ys, _ptr(weight), _ptr(shift), _ptr(scale), _ptr(mod_idx),
        shift.shape[0] if shift.dim() == 2 else 1, valid_rows, out.shape[0], hidden, eps,
        _workspace(x.device, st, workspace), st))
    return out


def tfk_qk_rmsnorm_rope_neox_fixed_valid(q: torch.Tensor, k: torch.Tensor, valid_rows: int,
                                         q_weight: torch.Tensor, k_weight: torch.Tensor,
                                         positions: torch.Tensor, n_heads: int, head_dim: int,
                                         theta: float = 10000.0, eps: float = 1e-6,
                                         q_out: torch.Tensor | None = None, k_out: torch.Tensor | None = None,
                                         stream=None):
    """Fixed-valid Q/K RMSNorm+RoPE on padded q, k [padded_rows, >= n_heads*head_dim]."""
    qs, ks = _rows(q, "q"), _rows(k, "k")
    if qs != ks or q.shape[0] != k.shape[0]:
        raise ValueError("q and k must have the same rows and row stride")
    padded = q.shape[0]
    width = n_heads * head_dim
    _param(q_weight, "q_weight")
    _param(k_weight, "k_weight")
    _param(positions, "positions", torch.int32)
    if q_out is None:
        q_out = torch.empty((padded, width), dtype=torch.bfloat16, device=q.device)
    if k_out is None:
        k_out = torch.empty((padded, width), dtype=torch.bfloat16, device=q.device)
    qos, kos = _rows(q_out, "q_out"), _rows(k_out, "k_out")
    if qos != kos or q_out.shape[0] != k_out.shape[0]:
        raise ValueError("q_out and k_out must have the same rows and row stride")
    _check(load().tfk_qk_rmsnorm_rope_neox_fixed_valid(
        _ptr(q), _ptr(k), qs, _ptr(q_out), _ptr(k_out), qos, _ptr(q_weight), _ptr(k_weight), _ptr(positions),
        valid_rows, q_out.shape[0], n_heads, head_dim, theta, eps, _stream(q, stream)))
    return q_out, k_out


def tfk_qk_rmsnorm_rope_neox_ulysses(q: torch.Tensor, k: torch.Tensor, q_weight: torch.Tensor,
                                     k_weight: torch.Tensor, positions: torch.Tensor, n_heads: int,
                                     head_dim: int, sp_degree: int, theta: float = 10000.0, eps: float = 1e-6,
                                     q_send: torch.Tensor | None = None, k_send: torch.Tensor | None = None,
                                     stream=None):
    """Q/K RMSNorm + RoPE written into Ulysses send buffers [sp_degree, rows, n_heads/sp_degree, head_dim]."""
    qs, ks = _rows(q, "q"), _rows(k, "k")
    if qs != ks or q.shape[0] != k.shape[0]:
        raise ValueError("q and k must have the same rows and row stride")
    rows = q.shape[0]
    shape = (sp_degree, rows, n_heads // max(1, sp_degree), head_dim)
    _param(q_weight, "q_weight")
    _param(k_weight, "k_weight")
    _param(positions, "positions", torch.int32)
    if q_send is None:
        q_send = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if k_send is None:
        k_send = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    for t, n in ((q_send, "q_send"), (k_send, "k_send")):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.numel() != rows * n_heads * head_dim:
            raise ValueError(f"{n} must be a contiguous CUDA bf16 tensor of {shape}")
    _check(load().tfk_qk_rmsnorm_rope_neox_ulysses(_ptr(q), _ptr(k), qs, _ptr(q_send), _ptr(k_send), _ptr(q_weight),
                                                   _ptr(k_weight), _ptr(positions), rows, n_heads, head_dim,
                                                   sp_degree, theta, eps, _stream(q, stream)))
    return q_send, k_send


def tfk_ulysses_pack(src: torch.Tensor, n_heads: int, head_dim: int, sp_degree: int,
                     dst: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """[rows, >= n_heads*head_dim] -> contiguous [sp_degree, rows, n_heads/sp_degree, head_dim]."""
    ss = _rows(src, "src")
    rows = src.shape[0]
    if dst is None:
        dst = torch.empty((sp_degree, rows, n_heads // max(1, sp_degree), head_dim), dtype=torch.bfloat16,
                          device=src.device)
    if dst.dtype != torch.bfloat16 or not dst.is_contiguous() or dst.numel() != rows * n_heads * head_dim:
        raise ValueError("dst must be a contiguous bf16 tensor of rows*n_heads*head_dim elements")
    _check(load().tfk_ulysses_pack(_ptr(src), ss, _ptr(dst), rows, n_heads, head_dim, sp_degree,
                                   _stream(src, stream)))
    return dst


def tfk_ulysses_unpack(src: torch.Tensor, n_heads: int, head_dim: int, sp_degree: int,
                       dst: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Contiguous [sp_degree, rows, n_heads/sp_degree, head_dim] -> [rows, n_heads*head_dim] (or dst's stride)."""
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA bf16 tensor")
    rows = src.numel() // (n_heads * head_dim)
    if dst is None:
        dst = torch.empty((rows, n_heads * head_dim), dtype=torch.bfloat16, device=src.device)
    ds = _rows(dst, "dst")
    _check(load().tfk_ulysses_unpack(_ptr(src), _ptr(dst), ds, rows, n_heads, head_dim, sp_degree,
                                     _stream(src, stream)))
    return dst


def tfk_swiglu(gate_up: torch.Tensor, out: torch.Tensor | None = None, ffn: int | None = None,
               stream=None) -> torch.Tensor:
    """silu(gate) * up for gate_up [rows, 2*ffn] = [gate | up] -> [rows, ffn] bf16."""
    gs = _rows(gate_up, "gate_up")
    rows = gate_up.shape[0]
    ffn = gate_up.shape[1] // 2 if ffn is None else ffn
    if out is None:
        out = torch.empty((rows, ffn), dtype=torch.bfloat16, device=gate_up.device)
    os_ = _rows(out, "out")
    _check(load().tfk_swiglu(_ptr(gate_up), gs, _ptr(out), os_, rows, ffn, _stream(gate_up, stream)))
    return out


def tfk_valid_gather(padded: torch.Tensor, valid_rows: int, compact: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """compact = padded[:valid_rows] (bit copy); both contiguous [*, hidden] bf16."""
    _rows(padded, "padded")
    if not padded.is_contiguous():
        raise ValueError("padded must be contiguous")
    hidden = padded.shape[1]
    if compact is None:
        compact = torch.empty((valid_rows, hidden), dtype=torch.bfloat16, device=padded.device)
    _rows(compact, "compact")
    if not compact.is_contiguous():
        raise ValueError("compact must be contiguous")
    _check(load().tfk_valid_gather(_ptr(padded), _ptr(compact), valid_rows, hidden, _stream(padded, stream)))
    return compact


def tfk_zero_tail_merge(compact: torch.Tensor, padded: torch.Tensor, valid_rows: int | None = None,
                        stream=None) -> torch.Tensor:
    """padded[:L] = compact, padded[L:] = +0.0, in one launch; both contiguous bf16."""
    _rows(compact, "compact")
    _rows(padded, "padded")
    if not (compact.is_contiguous() and padded.is_contiguous()):
        raise ValueError("compact and padded must be contiguous")
    L = compact.shape[0] if valid_rows is None else valid_rows
    _check(load().tfk_zero_tail_merge(_ptr(compact), _ptr(padded), L, padded.shape[0], padded.shape[1],
                                      _stream(padded, stream)))
    return padded


def tfk_velocity_cache_schedule(num_steps: int, start_ratio: float = 0.2, end_ratio: float = 0.8,
                                refresh_interval: int = 2, max_consecutive_reuse: int = 1) -> list:
    """Per step: True where the conservative velocity cache reuses the previous velocity."""
    buf = (ctypes.c_uint8 * max(1, num_steps))()
    hits = ctypes.c_int32(0)
    st = load().tfk_velocity_cache_schedule(num_steps, start_ratio, end_ratio, refresh_interval,
                                            max_consecutive_reuse, ctypes.cast(buf, ctypes.c_void_p),
                                            ctypes.cast(ctypes.pointer(hits), ctypes.c_void_p))
    _check(st)
    return [bool(buf[i]) for i in range(num_steps)]
