"""The allocation-free RMSNorm+AdaLN entry point, called through the C ABI.

tfk_rmsnorm_adaln_indexed_noalloc serves callers that cannot allocate device
memory (no allocator of their own, or code where cudaMalloc, which
synchronises the device, is not allowed): its row counters live in an array
of the library instead of a caller workspace.  Two calls in a row, the second
reusing the array the first left behind, must give what the workspace entry
point gives, within the parity tolerance.  The shapes take the warp-per-row
kernel, which is the one that uses the counters.  This file runs last, so a
failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

import rope_tfk_rmsnorm_gb300 as tfk
from helpers import ATOL, RTOL, f32_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


def _inputs(rng, rows, hidden, n_mod):
    x = torch.from_numpy(rng.standard_normal((rows, hidden)).astype(np.float32)).to(torch.bfloat16)
    x = to_dev(x.view(torch.int16).numpy().view(np.uint16))
    w = f32_dev((1 + 0.1 * rng.standard_normal(hidden)).astype(np.float32))
    shift = f32_dev((0.1 * rng.standard_normal((n_mod, hidden))).astype(np.float32))
    scale = f32_dev((0.1 * rng.standard_normal((n_mod, hidden))).astype(np.float32))
    idx = i32_dev(rng.integers(0, n_mod, rows).astype(np.int32))
    return x, w, shift, scale, idx


def _noalloc(lib, x, w, shift, scale, idx, y, eps, stream):
    return lib.tfk_rmsnorm_adaln_indexed_noalloc(x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0), w.data_ptr(),
                                                 shift.data_ptr(), scale.data_ptr(), idx.data_ptr(), shift.shape[0],
                                                 x.shape[0], x.shape[1], eps, stream)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row(cuda):
    lib = tfk.load()
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(20261203)
    for rows, hidden, n_mod in [(30358, 3072, 2), (8192, 4352, 4)]:
        x, w, shift, scale, idx = _inputs(rng, rows, hidden, n_mod)
        expect = tfk.tfk_rmsnorm_adaln_indexed(x, w, shift, scale, idx, 1e-6)
        got = torch.full_like(expect, float("nan"))
        st = _noalloc(lib, x, w, shift, scale, idx, got, 1e-6, stream)
        assert st == 0, lib.tfk_last_error_message().decode()
        torch.cuda.synchronize()
        g, e = got.double(), expect.double()
        assert bool(torch.isfinite(g).all()), f"{rows}x{hidden}: rows left unwritten"
        bad = (g - e).abs() > ATOL + RTOL * e.abs()
        assert not bool(bad.any()), f"{rows}x{hidden}: {int(bad.sum())} elements out of tolerance"
