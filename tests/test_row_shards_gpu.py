"""The path shards by rows: every step computes each token row on its own, so
running a step over row shards of a buffer (offset pointers into the same
tensors, as each sequence-parallel rank would hold its slice of the packed
token sequence) gives the whole-buffer result bit for bit.  The Ulysses
sequence parallelism of the MiniMax H3 integration (TeleFuser PR #23,
Changes Made) shards the token sequence exactly this way before its
all-to-all.

The shards are of unequal size and their inner edges (all but the end of
the one 7-row shard) are odd, so they fall off the 2-, 4-, 16- and 24-row
chunk grids of the Q/K and RMSNorm schedules and each shard gets its own
grid, chunking and (for RMSNorm) row order."""
import numpy as np
import pytest
import torch

import rope_tfk_rmsnorm_gb300 as tfk
import synth
from helpers import f32_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


def _cuts(T: int, n: int) -> list:
    if n == 2:
        return [0, (T // 3) | 1, T]
    rng = np.random.default_rng(n)
    inner = set(int(c) for c in rng.choice(np.arange(1, T - 8), n - 2, replace=False))
    inner = {c + 1 if c % 2 == 0 else c for c in inner}   # odd: never on a chunk edge
    c = max(inner)
    inner.add(c + 7)                                       # a shard of 7 rows
    return [0, *sorted(inner), T]


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _upload(wl, tag):
    return to_dev(synth.activation(wl, tag))


@pytest.mark.parametrize("name", ["large", "per_frame"])
def test_row_shards_match_the_whole_buffer_bit_for_bit(cuda, name):
    wl = synth.get(name)
    T = wl.rows
    p = {k: f32_dev(v) for k, v in synth.params(wl).items()}
    idx, pos = i32_dev(synth.mod_index(wl)), i32_dev(synth.positions(wl))
    plans = {n: _cuts(T, n) for n in (2, 8)}
    for cuts in plans.values():
        assert len(cuts) - 1 >= 2 and all(b > a for a, b in zip(cuts, cuts[1:]))

    x = _upload(wl, "x")
    whole = tfk.tfk_rmsnorm_adaln_indexed(x, p["w"], p["shift"], p["scale"], idx, wl.eps)
    for n, cuts in plans.items():
        part = torch.empty_like(whole)
        for s, e in zip(cuts, cuts[1:]):
            tfk.tfk_rmsnorm_adaln_indexed(x[s:e], p["w"], p["shift"], p["scale"], idx[s:e], wl.eps, out=part[s:e])
        torch.cuda.synchronize()
        assert _same_bits(whole, part), f"{name} a1, {n} shards"
    del x, whole, part

    q, k = _upload(wl, "q"), _upload(wl, "k")
    wq, wk = tfk.tfk_qk_rmsnorm_rope_neox(q, k, p["w_q"], p["w_k"], pos, wl.n_heads, wl.head_dim, wl.theta, wl.eps)
    for n, cuts in plans.items():
        pq, pk = torch.empty_like(wq), torch.empty_like(wk)
        for s, e in zip(cuts, cuts[1:]):
            tfk.tfk_qk_rmsnorm_rope_neox(q[s:e], k[s:e], p["w_q"], p["w_k"], pos[s:e], wl.n_heads, wl.head_dim,
                                         wl.theta, wl.eps, q_out=pq[s:e], k_out=pk[s:e])
        torch.cuda.synchronize()
        assert _same_bits(wq, pq) and _same_bits(wk, pk), f"{name} a2, {n} shards"
    del q, k, wq, wk, pq, pk

    gu = _upload(wl, "gate_up")
    whole = tfk.tfk_swiglu(gu)
    for n, cuts in plans.items():
        part = torch.empty_like(whole)
        for s, e in zip(cuts, cuts[1:]):
            tfk.tfk_swiglu(gu[s:e], out=part[s:e])
        torch.cuda.synchronize()
        assert _same_bits(whole, part), f"{name} a3, {n} shards"
    del gu, whole, part
    torch.cuda.empty_cache()
