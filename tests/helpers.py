"""Shared helpers of the GPU parity tests: host<->device bf16 moves, guarded
output buffers, and the element-wise tolerance check against the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

# bf16 outputs with fp32 arithmetic: |gpu - oracle| <= ATOL + RTOL * |oracle|, per element
ATOL = 2e-2
RTOL = 1e-2
GUARD = 0xFFFF           # canary bit pattern around every output
THREADS = max(1, min(32, os.cpu_count() or 1))


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Raw bf16 bits (uint16) -> a bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def f32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def i32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    """bf16 CUDA tensor -> raw bits (uint16), keeping its shape."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Guarded:
    """A [rows, stride] bf16 output view with GUARD rows above and below and
    GUARD in the padding columns; check() verifies no canary was touched."""

    def __init__(self, rows: int, width: int, stride: int | None = None, guard_rows: int = 2,
                 device="cuda", fill: int = GUARD):
        self.rows, self.width = rows, width
        self.stride = width if stride is None else stride
        self.g = guard_rows
        self.buf = torch.full((rows + 2 * guard_rows, self.stride), -1, dtype=torch.int16, device=device)
        if fill != GUARD:
            self.buf[guard_rows:guard_rows + rows, :width] = np.int16(np.uint16(fill).view(np.int16))
        self.view = self.buf.view(torch.bfloat16)[guard_rows:guard_rows + rows, :width]

    def check(self):
        b = self.buf.cpu().numpy().view(np.uint16)
        assert np.all(b[:self.g] == GUARD), "guard rows before the output were written"
        assert np.all(b[self.g + self.rows:] == GUARD), "guard rows after the output were written"
        if self.stride > self.width:
            assert np.all(b[:, self.width:] == GUARD), "padding columns of the output were written"

    def host(self) -> np.ndarray:
        return to_host(self.view)


def check_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL) -> dict:
    """Element-wise |gpu - ref| <= atol + rtol*|ref| for bf16 GPU output vs fp64 oracle values."""
    g = oracle.bf16_to_f64(gpu_bits).reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    rounded = oracle.round_bf16(ref, threads=THREADS)
    stats = {
        "n": int(ref.size),
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel": float((err / np.maximum(np.abs(ref), 1e-30)).max()) if err.size else 0.0,
        "bit_equal": float(np.mean(gpu_bits.reshape(ref.shape) == rounded)) if err.size else 1.0,
    }
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} elements out of tolerance; worst at "
                             f"{i}: gpu {g[i]!r} oracle {ref[i]!r}; {stats}")
    return stats


class Stats:
    """Running totals of check_close results over the row blocks of one output."""

    def __init__(self, what: str):
        self.what, self.n, self.max_abs, self.max_rel, self.equal = what, 0, 0.0, 0.0, 0.0

    def add(self, s: dict):
        self.n += s["n"]
        self.max_abs = max(self.max_abs, s["max_abs"])
        self.max_rel = max(self.max_rel, s["max_rel"])
        self.equal += s["bit_equal"] * s["n"]

    def summary(self) -> dict:
        return {"what": self.what, "n": self.n, "max_abs": self.max_abs, "max_rel": self.max_rel,
                "bit_equal": self.equal / max(1, self.n)}
