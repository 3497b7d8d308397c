"""Seeded random shapes against the oracle, through the C ABI.

The launchers pick among many kernel instantiations by shape: one, two,
three, four or eight vectors per thread (whole-vector widths without bounds
predicates) or one warp per row (6 to 24 vectors per lane, staged modulation
rows in one or several passes) for RMSNorm+AdaLN; one to four heads per lane group, masked last
groups and side-by-side token streams for Q/K; one chunk per CTA or several
whole rows for SwiGLU; 4-row tiles or the column walk for the relayouts.
Every case here draws its shape from a fixed seed, so a wrong choice or a bad
edge anywhere in those rules shows up as a parity failure with its shape in
the test id.
"""
import numpy as np
import pytest
import torch

import oracle
import rope_tfk_rmsnorm_gb300 as tfk
from helpers import Guarded, THREADS, check_close, f32_dev, i32_dev, to_dev
from test_parity_gpu import gpu_adaln, gpu_qk, gpu_swiglu, mod_params, ora_adaln, ora_qk, ora_swiglu, rand_bits

pytestmark = pytest.mark.gpu

_RNG = np.random.default_rng(20261202)


def _hidden(rng):
    """Widths near the shape thresholds as often as arbitrary multiples of 8."""
    if rng.random() < 0.5:
        return int(8 * rng.integers(1, 1025))
    base = int(rng.choice([512, 768, 1024]))
    return int(base * rng.integers(1, 9)) + int(rng.choice([0, 0, 8, -8]))


def _adaln_cases(n):
    out = []
    for _ in range(n):
        hidden = max(8, _hidden(_RNG))
        rows = int(_RNG.integers(1, max(2, min(700, 3_000_000 // hidden))))
        out.append((rows, hidden, int(_RNG.integers(1, 7)), int(_RNG.integers(0, 2 ** 31))))
    return out


def _qk_cases(n):
    out = []
    while len(out) < n:
        D = int(16 * _RNG.integers(1, 17)) if _RNG.random() < 0.85 else 512
        H = int(_RNG.integers(1, 49))
        if H * D > 8192:
            continue
        rows = int(_RNG.integers(1, 300))
        out.append((rows, H, D, int(_RNG.integers(0, 2 ** 31))))
    return out


def _swiglu_cases(n):
    return [(int(_RNG.integers(1, 400)), int(8 * _RNG.integers(1, 1200)), int(_RNG.integers(0, 2 ** 31)))
            for _ in range(n)]


def _ulysses_cases(n):
    out = []
    while len(out) < n:
        P = int(_RNG.integers(1, 9))
        H = P * int(_RNG.integers(1, 9))
        D = int(16 * _RNG.integers(1, 17))
        if H * D > 16384:
            continue
        out.append((int(_RNG.integers(1, 200)), H, D, P, int(_RNG.integers(0, 2 ** 31))))
    return out


def _adaln_warp_cases(n):
    """Widths of the warp-per-row RMSNorm kernel (multiples of 768 from 1536 to 6144, and the
    widths between 4096 and 6144 that are not multiples of 1024) at row counts that fill
    several warps per CTA, with up to 90 modulation rows drawn per token, so that a CTA's rows
    may need more modulation rows than fit in shared memory (several passes)."""
    whole = [768 * k for k in range(2, 9)]
    ragged = [h for h in range(4104, 6144, 8) if h % 1024]
    out = []
    for i in range(n):
        hidden = int(_RNG.choice(whole if i % 2 == 0 else ragged))
        rows = int(_RNG.integers(300, max(301, min(12000, 24_000_000 // hidden))))
        out.append((rows, hidden, int(_RNG.integers(1, 91)), int(_RNG.integers(0, 2 ** 31))))
    return out


def _adaln_handout_cases(n):
    """Warp-per-row widths at 60-140 MB of x, above the size from which rows are handed
    out to warps through a workspace, with up to 8 modulation rows (all staged at once)."""
    whole = [768 * k for k in range(2, 9)]
    ragged = [h for h in range(4104, 6144, 8) if h % 1024]
    out = []
    for i in range(n):
        hidden = int(_RNG.choice(whole if i % 2 == 0 else ragged))
        rows = int(_RNG.integers(60_000_000, 140_000_000) // (2 * hidden))
        out.append((rows, hidden, int(_RNG.integers(1, 9)), int(_RNG.integers(0, 2 ** 31))))
    return out


ADALN = _adaln_cases(40)
ADALN_WARP = _adaln_warp_cases(10)
ADALN_HANDOUT = _adaln_handout_cases(6)
QK = _qk_cases(40)
SWIGLU = _swiglu_cases(20)
ULYSSES = _ulysses_cases(16)


@pytest.mark.parametrize("rows,hidden,n_mod,seed", ADALN,
                         ids=[f"{r}x{h}m{m}" for r, h, m, _ in ADALN])
def test_adaln_random_shapes(cuda, rows, hidden, n_mod, seed):
    rng = np.random.default_rng(seed)
    x = rand_bits(rng, (rows, hidden), 2.0)
    w, sh, sc = mod_params(rng, n_mod, hidden)
    idx = rng.integers(0, n_mod, rows).astype(np.int32)
    check_close(gpu_adaln(x, w, sh, sc, idx, 1e-6), ora_adaln(x, w, sh, sc, idx, 1e-6),
                f"a1 {rows}x{hidden}")


@pytest.mark.parametrize("rows,hidden,n_mod,seed", ADALN_WARP,
                         ids=[f"{r}x{h}m{m}" for r, h, m, _ in ADALN_WARP])
def test_adaln_warp_kernel_random_shapes(cuda, rows, hidden, n_mod, seed):
    rng = np.random.default_rng(seed)
    x = rand_bits(rng, (rows, hidden), 2.0)
    w, sh, sc = mod_params(rng, n_mod, hidden)
    idx = rng.integers(0, n_mod, rows).astype(np.int32)
    check_close(gpu_adaln(x, w, sh, sc, idx, 1e-6), ora_adaln(x, w, sh, sc, idx, 1e-6),
                f"a1 {rows}x{hidden}")


@pytest.mark.parametrize("rows,hidden,n_mod,seed", ADALN_HANDOUT,
                         ids=[f"{r}x{h}m{m}" for r, h, m, _ in ADALN_HANDOUT])
def test_adaln_rows_handed_out_random_shapes(cuda, rows, hidden, n_mod, seed):
    """Rows handed out through a workspace give the bits of the split up front on every
    element, leave the workspace zero, and agree with the oracle on sampled rows."""
    rng = np.random.default_rng(seed)
    xh = rand_bits(rng, (rows, hidden), 2.0)
    x = to_dev(xh)
    w, sh, sc = mod_params(rng, n_mod, hidden)
    idx = rng.integers(0, n_mod, rows).astype(np.int32)
    args = (x, f32_dev(w), f32_dev(sh), f32_dev(sc), i32_dev(idx), 1e-6)
    ws = torch.zeros(tfk.RMSNORM_WORKSPACE_BYTES // 8, dtype=torch.int64, device="cuda")
    handed = tfk.tfk_rmsnorm_adaln_indexed(*args, workspace=ws)
    split = tfk.tfk_rmsnorm_adaln_indexed(*args, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(handed.view(torch.int16), split.view(torch.int16))
    assert int(ws.abs().sum()) == 0
    sample = np.unique(np.r_[0, rows - 1, rng.integers(0, rows, 254)])
    got = handed[torch.from_numpy(sample).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    check_close(got, ora_adaln(xh[sample], w, sh, sc, idx[sample], 1e-6), f"a1 handed out {rows}x{hidden}")


@pytest.mark.parametrize("rows,H,D,seed", QK, ids=[f"{r}x{h}x{d}" for r, h, d, _ in QK])
def test_qk_random_shapes(cuda, rows, H, D, seed):
    rng = np.random.default_rng(seed)
    q = rand_bits(rng, (rows, H * D), 2.0)
    k = rand_bits(rng, (rows, H * D))
    wq = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    pos = rng.integers(0, 200_000, rows).astype(np.int32)
    gq, gk = gpu_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6, fused=bool(seed & 1))
    rq, rk = ora_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    check_close(gq, rq, f"q {rows}x{H}x{D}")
    check_close(gk, rk, f"k {rows}x{H}x{D}")


@pytest.mark.parametrize("rows,ffn,seed", SWIGLU, ids=[f"{r}x{f}" for r, f, _ in SWIGLU])
def test_swiglu_random_shapes(cuda, rows, ffn, seed):
    rng = np.random.default_rng(seed)
    gu = rand_bits(rng, (rows, 2 * ffn), 3.0)
    check_close(gpu_swiglu(gu), ora_swiglu(gu), f"swiglu {rows}x{ffn}")


@pytest.mark.parametrize("rows,H,D,P,seed", ULYSSES, ids=[f"{r}x{h}x{d}p{p}" for r, h, d, p, _ in ULYSSES])
def test_ulysses_random_shapes(cuda, rows, H, D, P, seed):
    """Pack and unpack bit-exact against the oracle's permutation, and the fused
    Q/K send layout within tolerance."""
    rng = np.random.default_rng(seed)
    W = H * D
    src = rand_bits(rng, (rows, W))
    packed = tfk.tfk_ulysses_pack(to_dev(src), H, D, P)
    back = Guarded(rows, W)
    tfk.tfk_ulysses_unpack(packed, H, D, P, dst=back.view)
    torch.cuda.synchronize()
    back.check()
    want = oracle.ulysses_pack(src, H, D, P)
    got = packed.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(want.shape)
    assert np.array_equal(got, want)
    assert np.array_equal(back.host(), src)

    q = rand_bits(rng, (rows, W), 2.0)
    k = rand_bits(rng, (rows, W))
    wq = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    pos = rng.integers(0, 100_000, rows).astype(np.int32)
    qs, ks = tfk.tfk_qk_rmsnorm_rope_neox_ulysses(to_dev(q), to_dev(k), f32_dev(wq), f32_dev(wk), i32_dev(pos),
                                                  H, D, P)
    torch.cuda.synchronize()
    rq, rk = ora_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    for got_t, ref, name in ((qs, rq, "q"), (ks, rk, "k")):
        bits = got_t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        check_close(bits.reshape(-1), oracle.ulysses_pack(ref, H, D, P).reshape(-1), f"ulysses {name}")


def _fixed_valid_cases(n):
    out = []
    while len(out) < n:
        hidden = max(8, _hidden(_RNG))
        D = int(16 * _RNG.integers(1, 17))
        H = int(_RNG.integers(1, 33))
        if H * D > 8192:
            continue
        N = int(_RNG.integers(1, max(2, min(400, 2_000_000 // max(hidden, H * D)))))
        L = int(_RNG.integers(0, N + 1))
        out.append((N, L, hidden, H, D, int(_RNG.integers(0, 2 ** 31))))
    return out


FIXED = _fixed_valid_cases(16)


@pytest.mark.parametrize("N,L,hidden,H,D,seed", FIXED, ids=[f"N{n}L{l}h{hd}q{h}x{d}" for n, l, hd, h, d, _ in FIXED])
def test_fixed_valid_random_shapes(cuda, N, L, hidden, H, D, seed):
    """Fixed-valid mode: rows [0, L) computed from the padded buffer, whose NaN
    tail is never read, and the rest of every output +0.0."""
    import synth
    rng = np.random.default_rng(seed)
    x = rand_bits(rng, (N, hidden))
    q, k = rand_bits(rng, (N, H * D), 2.0), rand_bits(rng, (N, H * D))
    for a in (x, q, k):
        a[L:] = synth.BF16_NAN
    w, sh, sc = mod_params(rng, 3, hidden)
    idx = rng.integers(0, 3, max(L, 1)).astype(np.int32)
    pos = rng.integers(0, 100_000, max(L, 1)).astype(np.int32)
    wq = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    y = Guarded(N, hidden)
    tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(to_dev(x), L, f32_dev(w), f32_dev(sh), f32_dev(sc), i32_dev(idx),
                                              1e-6, out=y.view)
    qo, ko = Guarded(N, H * D), Guarded(N, H * D)
    tfk.tfk_qk_rmsnorm_rope_neox_fixed_valid(to_dev(q), to_dev(k), L, f32_dev(wq), f32_dev(wk), i32_dev(pos),
                                             H, D, 10000.0, 1e-6, q_out=qo.view, k_out=ko.view)
    torch.cuda.synchronize()
    for g in (y, qo, ko):
        g.check()
        assert np.all(g.host()[L:] == 0x0000)
    check_close(y.host(), oracle.rmsnorm_adaln_fixed_valid(x, L, w, sh, sc, idx[:L], 1e-6, threads=THREADS),
                f"fixed-valid a1 N={N} L={L}")
    rq, rk = oracle.qk_rmsnorm_rope_neox_fixed_valid(q, k, L, wq, wk, pos[:L], H, D, 10000.0, 1e-6, threads=THREADS)
    check_close(qo.host(), rq.reshape(N, -1), f"fixed-valid q N={N} L={L}")
    check_close(ko.host(), rk.reshape(N, -1), f"fixed-valid k N={N} L={L}")
