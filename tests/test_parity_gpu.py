"""GPU parity: every entry point, called through the C ABI, against the fp64
oracle on the same seeded inputs.

Bit-exact for gather/merge; |gpu - oracle| <= 2e-2 + 1e-2*|oracle| per
element for the floating-point kernels.  Every output buffer is surrounded by
canary rows (and canary padding columns where the stride is wider than the
row), which must come back untouched.  Small and ragged cases are compared in
full, and so are the full-size workloads (75,600 and 56,320 tokens, the
32,768-row valid-only buffer and the 8-rank Ulysses send layout), in blocks
of rows that bound host memory; a few extra shapes beyond the workloads are
compared on seeded samples of rows.
"""
import numpy as np
import pytest
import torch

import oracle
import rope_tfk_rmsnorm_gb300 as tfk
import synth
from helpers import Guarded, Stats, THREADS, check_close, f32_dev, i32_dev, to_dev, to_host

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# runners: inputs as host arrays, outputs as host bits (+ guard checks)
# ---------------------------------------------------------------------------

def gpu_adaln(x, w, shift, scale, idx, eps, x_stride=None, y_stride=None, inplace=False):
    rows, hidden = x.shape
    xs = hidden if x_stride is None else x_stride
    xbuf = Guarded(rows, hidden, xs)
    xbuf.view.copy_(to_dev(x))
    if inplace:
        out = xbuf
    else:
        out = Guarded(rows, hidden, y_stride)
    tfk.tfk_rmsnorm_adaln_indexed(xbuf.view, f32_dev(w), f32_dev(shift), f32_dev(scale), i32_dev(idx),
                                  eps, out=out.view)
    torch.cuda.synchronize()
    out.check()
    if not inplace:
        xbuf.check()
        assert np.array_equal(xbuf.host(), x), "input x was modified"
    return out.host()


def ora_adaln(x, w, shift, scale, idx, eps):
    return oracle.rmsnorm_adaln_indexed(x, w, shift, scale, idx, eps, threads=THREADS)


def gpu_qk(q, k, wq, wk, pos, H, D, theta, eps, fused=False, inplace=False, out_stride=None):
    rows = q.shape[0]
    width = H * D
    if fused:  # q and k as column slices of one [rows, 3*H*D] QKV buffer
        qkv = Guarded(rows, 3 * width)
        qkv.view[:, :width].copy_(to_dev(q))
        qkv.view[:, width:2 * width].copy_(to_dev(k))
        qv, kv = qkv.view[:, :width], qkv.view[:, width:2 * width]
    else:
        qb, kb = Guarded(rows, width), Guarded(rows, width)
        qb.view.copy_(to_dev(q))
        kb.view.copy_(to_dev(k))
        qv, kv = qb.view, kb.view
    if inplace:
        qo, ko = qv, kv
    else:
        ostride = 2 * width if fused and out_stride is None else out_stride
        if fused:
            ob = Guarded(rows, 2 * width, ostride)
            qo, ko = ob.view[:, :width], ob.view[:, width:]
        else:
            qob, kob = Guarded(rows, width, out_stride), Guarded(rows, width, out_stride)
            qo, ko = qob.view, kob.view
    tfk.tfk_qk_rmsnorm_rope_neox(qv, kv, f32_dev(wq), f32_dev(wk), i32_dev(pos), H, D, theta, eps,
                                 q_out=qo, k_out=ko)
    torch.cuda.synchronize()
    if fused:
        qkv.check()
        assert np.all(to_host(qkv.view[:, 2 * width:]) == 0xFFFF), "v columns of the QKV buffer were written"
        if not inplace:
            ob.check()
    elif not inplace:
        qob.check()
        kob.check()
    return to_host(qo), to_host(ko)


def ora_qk(q, k, wq, wk, pos, H, D, theta, eps):
    qo, ko = oracle.qk_rmsnorm_rope_neox(q, k, wq, wk, pos, H, D, theta, eps, threads=THREADS)
    return qo.reshape(q.shape[0], H * D), ko.reshape(k.shape[0], H * D)


def gpu_swiglu(gu, out_stride=None, in_stride=None):
    rows, two_f = gu.shape
    ffn = two_f // 2
    gbuf = Guarded(rows, two_f, in_stride)
    gbuf.view.copy_(to_dev(gu))
    out = Guarded(rows, ffn, out_stride)
    tfk.tfk_swiglu(gbuf.view, out=out.view)
    torch.cuda.synchronize()
    out.check()
    gbuf.check()
    return out.host()


def ora_swiglu(gu):
    return oracle.swiglu(gu, threads=THREADS)


def rand_bits(rng, shape, scale=1.0):
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def mod_params(rng, n_mod, hidden, std=0.1):
    w = (1 + 0.1 * rng.standard_normal(hidden)).astype(np.float32)
    return (w, (std * rng.standard_normal((n_mod, hidden))).astype(np.float32),
            (std * rng.standard_normal((n_mod, hidden))).astype(np.float32))


# ---------------------------------------------------------------------------
# RMSNorm + indexed AdaLN: ragged sizes, index patterns, strides, in place
# ---------------------------------------------------------------------------

ADALN_CASES = [
    # rows, hidden, n_mod, index pattern
    (1, 8, 1, "const"),
    (7, 296, 3, "random"),
    (333, 1000, 5, "random"),
    (300, 3072, 4, "pairs"),         # two rows alternate per token, then two others
    (129, 5120, 2, "blocks"),
    (1000, 4104, 6, "random"),       # 513 vectors: ragged last thread of a 2-vector layout
    (150, 1536, 3, "pairs"),         # multiples of 768 up to 6144: three vectors per thread
    (99, 2304, 5, "random"),
    (60, 5376, 2, "blocks"),
    (200, 6144, 3, "random"),
    (120, 7168, 3, "random"),        # 7168-8192: two vectors per thread, 448-512 threads
    (150, 8192, 2, "pairs"),
    (90, 8200, 3, "random"),         # 1025 vectors: back to four per thread, ragged
    (64, 16384, 3, "random"),
    (17, 32768, 2, "random"),        # largest hidden
    (2500, 512, 28, "blocks"),
    (301, 4352, 3, "random"),        # warp-per-row kernel: 17 of 20 vectors per lane
    (257, 5632, 2, "random"),        # 22 of 24 vectors per lane
    (130, 6144, 3, "pairs"),         # 24 whole vectors per lane
    (4560, 2304, 70, "random"),      # 30 rows per CTA over more modulation rows than slots: several passes
    (77, 12288, 2, "random"),        # 80 KB in flight per SM for rows of 16 KB and more
    (40, 16392, 3, "random"),        # eight vectors per thread, one CTA per row
    (29, 17416, 3, "random"),        # a pair of CTAs per row: halves of 1089 and 1088 vectors
    (33, 20480, 2, "pairs"),         # pair: 1280 whole vectors per CTA
    (200, 24576, 4, "random"),
]


def index_pattern(rng, rows, n_mod, kind):
    if kind == "const":
        return np.zeros(rows, np.int32)
    if kind == "random":
        return rng.integers(0, n_mod, rows).astype(np.int32)
    if kind == "pairs":
        half = rows // 2
        return np.r_[rng.integers(0, 2, half), 2 + rng.integers(0, 2, rows - half)].astype(np.int32) % n_mod
    return (np.arange(rows) * n_mod // rows).astype(np.int32)


@pytest.mark.parametrize("rows,hidden,n_mod,kind", ADALN_CASES)
def test_adaln_ragged(cuda, rows, hidden, n_mod, kind):
    rng = np.random.default_rng(rows * 7 + hidden)
    x = rand_bits(rng, (rows, hidden), 2.0)
    w, sh, sc = mod_params(rng, n_mod, hidden)
    idx = index_pattern(rng, rows, n_mod, kind)
    got = gpu_adaln(x, w, sh, sc, idx, 1e-6)
    check_close(got, ora_adaln(x, w, sh, sc, idx, 1e-6), f"adaln {rows}x{hidden}")


@pytest.mark.parametrize("rows,hidden,n_mod", [(30358, 3072, 2), (20001, 4352, 3), (40000, 1536, 2), (12000, 6144, 2),
                                           (10007, 5632, 4), (8192, 3072, 4), (3001, 1536, 2), (2000, 5120, 2),
                                           (20000, 2304, 70), (333, 1000, 5)])
def test_adaln_workspace_and_static_split_give_the_same_bits(cuda, rows, hidden, n_mod):
    """With a workspace the warp-per-row kernel hands rows out dynamically (calls of at least
    336 KiB of x per SM: the first five cases on a 152-SM GPU); without one it splits them up
    front.  Both give the same bits (a row's arithmetic does not depend on who computes it),
    and each call leaves the workspace zero for the next.  Also for the fixed-valid variant,
    for calls below that size, for more modulation rows than shared-memory slots (2304 x 70,
    several passes) and for widths the workspace does not change (CTA-per-row)."""
    rng = np.random.default_rng(rows + hidden)
    x = to_dev(rand_bits(rng, (rows, hidden)))
    w, sh, sc = (f32_dev(a) for a in mod_params(rng, n_mod, hidden))
    idx = i32_dev(rng.integers(0, n_mod, rows).astype(np.int32))
    ws = torch.zeros(tfk.RMSNORM_WORKSPACE_BYTES // 8, dtype=torch.int64, device="cuda")
    plain = tfk.tfk_rmsnorm_adaln_indexed(x, w, sh, sc, idx, 1e-6, workspace=False)
    first = tfk.tfk_rmsnorm_adaln_indexed(x, w, sh, sc, idx, 1e-6, workspace=ws)
    second = tfk.tfk_rmsnorm_adaln_indexed(x, w, sh, sc, idx, 1e-6, workspace=ws)
    L = rows - rows // 7
    fv_plain = tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(x, L, w, sh, sc, idx[:L], 1e-6, workspace=False)
    fv_ws = tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(x, L, w, sh, sc, idx[:L], 1e-6, workspace=ws)
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16)
    assert torch.equal(bits(plain), bits(first)) and torch.equal(bits(plain), bits(second))
    assert torch.equal(bits(fv_plain), bits(fv_ws))
    assert torch.equal(bits(fv_ws[:L]), bits(plain[:L])) and int((bits(fv_ws[L:]) != 0).sum()) == 0
    assert int(ws.abs().sum()) == 0, "the workspace is not left zero"


def test_adaln_strided_and_in_place(cuda):
    rng = np.random.default_rng(1)
    rows, hidden = 211, 3072
    x = rand_bits(rng, (rows, hidden))
    w, sh, sc = mod_params(rng, 3, hidden)
    idx = rng.integers(0, 3, rows).astype(np.int32)
    ref = ora_adaln(x, w, sh, sc, idx, 1e-6)
    check_close(gpu_adaln(x, w, sh, sc, idx, 1e-6, x_stride=hidden + 64, y_stride=hidden + 8), ref, "strided")
    check_close(gpu_adaln(x, w, sh, sc, idx, 1e-6, x_stride=hidden + 64, inplace=True), ref, "in place")


def test_adaln_degenerate_rows(cuda):
    # zero rows give shift exactly; a constant row gives c/sqrt(c^2+eps) modulated
    hidden = 512
    x = np.zeros((4, hidden), np.uint16)
    x[1] = 0x3F80  # 1.0
    x[2] = 0x3A83  # ~1e-3: eps matters
    x[3] = 0xC2C8  # -100
    rng = np.random.default_rng(3)
    w, sh, sc = mod_params(rng, 2, hidden)
    idx = np.array([0, 1, 0, 1], np.int32)
    got = gpu_adaln(x, w, sh, sc, idx, 1e-6)
    ref = ora_adaln(x, w, sh, sc, idx, 1e-6)
    check_close(got, ref, "degenerate rows")
    assert np.array_equal(got[0], oracle.round_bf16(sh[0].astype(np.float64)))


def test_adaln_empty_is_a_no_op(cuda):
    out = Guarded(0, 512)
    x = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(512, dtype=torch.float32, device="cuda")
    tfk.tfk_rmsnorm_adaln_indexed(x, z, z[None], z[None], torch.empty(0, dtype=torch.int32, device="cuda"),
                                  out=out.view)
    torch.cuda.synchronize()
    out.check()


def test_adaln_bad_arguments_raise_and_write_nothing(cuda):
    out = Guarded(8, 12)
    x = torch.zeros((8, 12), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(12, dtype=torch.float32, device="cuda")
    with pytest.raises(tfk.TfkError) as e:
        tfk.tfk_rmsnorm_adaln_indexed(x, z, z[None], z[None], torch.zeros(8, dtype=torch.int32, device="cuda"),
                                      out=out.view)
    assert e.value.status == 3  # hidden 12 is not a multiple of 8
    torch.cuda.synchronize()
    out.check()
    assert np.all(out.host() == 0xFFFF)


# ---------------------------------------------------------------------------
# Q/K RMSNorm + NeoX RoPE
# ---------------------------------------------------------------------------

QK_CASES = [
    # rows, heads, head_dim
    (5, 1, 16),
    (33, 3, 64),
    (65, 5, 96),       # 6 lanes per head in a group of 8
    (300, 24, 128),
    (77, 40, 128),
    (19, 128, 128),    # 4 heads per lane group, several head chunks
    (13, 201, 128),    # odd head count: the last lane group of q and of k holds 1 head
    (23, 30, 96),      # 2 of 4 heads in the last group, 6 data lanes in a group of 8
    (41, 6, 128),      # 3 heads per lane group
    (19, 9, 64),
    (33, 12, 128),
    (18, 20, 128),
    (7, 3, 128),       # 3 heads per group, two token streams per CTA; fewer rows than streams x 4
    (25, 2, 128),      # two streams of 16 lanes
    (9, 4, 64),        # four streams of 8 lanes
    (7, 300, 64),      # many heads: a 2-D grid of token runs x head chunks
    (11, 4, 256),
    (9, 2, 512),
]


@pytest.mark.parametrize("rows,H,D", QK_CASES)
def test_qk_ragged(cuda, rows, H, D):
    rng = np.random.default_rng(rows + H * D)
    q = rand_bits(rng, (rows, H * D), 3.0)
    k = rand_bits(rng, (rows, H * D), 0.5)
    wq = (1 + 0.2 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.2 * rng.standard_normal(D)).astype(np.float32)
    pos = rng.integers(0, 80000, rows).astype(np.int32)
    qo, ko = gpu_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    rq, rk = ora_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    check_close(qo, rq, f"q {rows}x{H}x{D}")
    check_close(ko, rk, f"k {rows}x{H}x{D}")


def test_qk_fused_qkv_layout_in_place_and_out_of_place(cuda):
    rng = np.random.default_rng(5)
    rows, H, D = 97, 8, 128
    q = rand_bits(rng, (rows, H * D))
    k = rand_bits(rng, (rows, H * D))
    wq = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    pos = np.arange(rows, dtype=np.int32) * 613
    rq, rk = ora_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    for inplace in (False, True):
        qo, ko = gpu_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6, fused=True, inplace=inplace)
        check_close(qo, rq, f"fused q inplace={inplace}")
        check_close(ko, rk, f"fused k inplace={inplace}")
    qo, ko = gpu_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6, out_stride=H * D + 24)
    check_close(qo, rq, "padded-stride q")


def test_qk_extreme_positions_and_bases(cuda):
    # negative positions and positions near 2^31 - 1: the angle reduction is exact mod one turn
    rng = np.random.default_rng(8)
    rows, H, D = 64, 2, 128
    q = rand_bits(rng, (rows, H * D))
    k = rand_bits(rng, (rows, H * D))
    w = np.ones(D, np.float32)
    pos = np.r_[rng.integers(-2**31, 2**31 - 1, rows - 4), [0, -1, 2**31 - 1, -2**31]].astype(np.int32)
    for theta in (10000.0, 500000.0, 10.0):
        qo, ko = gpu_qk(q, k, w, w, pos, H, D, theta, 1e-6)
        rq, rk = ora_qk(q, k, w, w, pos, H, D, theta, 1e-6)
        check_close(qo, rq, f"q theta={theta}")
        check_close(ko, rk, f"k theta={theta}")


def test_qk_position_zero_is_plain_head_rmsnorm(cuda):
    rng = np.random.default_rng(9)
    rows, H, D = 40, 6, 64
    q = rand_bits(rng, (rows, H * D))
    w = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    qo, _ = gpu_qk(q, q, w, w, np.zeros(rows, np.int32), H, D, 10000.0, 1e-6)
    ref = oracle.head_rmsnorm(q, H, D, w, 1e-6).reshape(rows, H * D)
    check_close(qo, ref, "pos 0")


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,ffn", [(1, 8), (5, 104), (300, 1024), (37, 13824), (3, 8200),
                                      (1001, 3072),    # 2 whole rows per block, odd row count
                                      (777, 520),      # 15 rows of 65 vectors per block, 49 slots idle
                                      (70, 4096), (70, 4104)])  # the last width with 2 rows per block, and the first without
def test_swiglu_ragged(cuda, rows, ffn):
    rng = np.random.default_rng(rows * 31 + ffn)
    gu = rand_bits(rng, (rows, 2 * ffn), 4.0)
    check_close(gpu_swiglu(gu), ora_swiglu(gu), f"swiglu {rows}x{ffn}")


def test_swiglu_strides_and_extremes(cuda):
    rng = np.random.default_rng(2)
    rows, ffn = 64, 512
    g = rng.standard_normal((rows, ffn)) * 3
    g[0, :8] = [0.0, -0.0, 1.0, -1.0, 90.0, -90.0, 300.0, -300.0]
    u = rng.standard_normal((rows, ffn))
    gu = torch.from_numpy(np.concatenate([g, u], 1).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    check_close(gpu_swiglu(gu, out_stride=ffn + 8, in_stride=2 * ffn + 16), ora_swiglu(gu), "swiglu strided")


# ---------------------------------------------------------------------------
# valid-only gather / zero-tail merge (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,L,hidden", [(1, 0, 8), (1, 1, 8), (100, 37, 24), (4096, 4095, 3072),
                                        (1000, 1000, 512), (513, 0, 64)])
def test_gather_merge_bit_exact(cuda, N, L, hidden):
    rng = np.random.default_rng(N + L)
    padded = rng.integers(0, 65536, (N, hidden), dtype=np.uint32).astype(np.uint16)
    padded[L:] = synth.BF16_NAN
    dev = to_dev(padded)
    comp = Guarded(L, hidden)
    tfk.tfk_valid_gather(dev, L, compact=comp.view)
    torch.cuda.synchronize()
    comp.check()
    assert np.array_equal(comp.host(), oracle.valid_gather(padded, L))
    back = Guarded(N, hidden)
    tfk.tfk_zero_tail_merge(comp.view, back.view)
    torch.cuda.synchronize()
    back.check()
    merged = back.host()
    assert np.array_equal(merged, oracle.zero_tail_merge(oracle.valid_gather(padded, L), N))
    assert np.all(merged[L:] == 0x0000)


# ---------------------------------------------------------------------------
# the workloads
# ---------------------------------------------------------------------------

def _inputs_dev(wl, tags, rows=None):
    host = {t: synth.activation(wl, t, rows=rows) for t in tags}
    return host, {t: to_dev(a) for t, a in host.items()}


def _params_dev(wl):
    p = synth.params(wl)
    return p, {k: f32_dev(v) for k, v in p.items()}


def _chain_full(wl):
    """Whole-workload chain on the GPU, full oracle comparison (small workloads)."""
    host, dev = _inputs_dev(wl, ["x", "q", "k", "gate_up"])
    p, pd = _params_dev(wl)
    idx, pos = synth.mod_index(wl), synth.positions(wl)
    y = tfk.tfk_rmsnorm_adaln_indexed(dev["x"], pd["w"], pd["shift"], pd["scale"], i32_dev(idx), wl.eps)
    qo, ko = tfk.tfk_qk_rmsnorm_rope_neox(dev["q"], dev["k"], pd["w_q"], pd["w_k"], i32_dev(pos),
                                          wl.n_heads, wl.head_dim, wl.theta, wl.eps)
    o = tfk.tfk_swiglu(dev["gate_up"])
    torch.cuda.synchronize()
    stats = {"a1": check_close(to_host(y), ora_adaln(host["x"], p["w"], p["shift"], p["scale"], idx, wl.eps),
                               f"{wl.name} a1")}
    rq, rk = ora_qk(host["q"], host["k"], p["w_q"], p["w_k"], pos, wl.n_heads, wl.head_dim, wl.theta, wl.eps)
    stats["a2q"] = check_close(to_host(qo), rq, f"{wl.name} a2 q")
    stats["a2k"] = check_close(to_host(ko), rk, f"{wl.name} a2 k")
    stats["a3"] = check_close(to_host(o), ora_swiglu(host["gate_up"]), f"{wl.name} a3")
    return stats


def test_tiny_chain(cuda):
    stats = _chain_full(synth.get("tiny"))
    assert all(s["bit_equal"] > 0.9 for s in stats.values()), stats


def test_medium_chain(cuda):
    _chain_full(synth.get("medium"))


def test_valid_only_pipeline(cuda):
    """gather X, Q, K -> a1 and a2 on the valid rows only -> merge back: the tail is exactly +0.0."""
    wl = synth.get("valid_only")
    N, L, hidden = wl.rows, synth.valid_len(wl), wl.hidden
    host, dev = _inputs_dev(wl, ["x", "q", "k"])
    p, pd = _params_dev(wl)
    idx = synth.mod_index(wl, np.arange(L))
    pos = synth.positions(wl, np.arange(L))
    compact = {}
    for t in ("x", "q", "k"):
        compact[t] = tfk.tfk_valid_gather(dev[t], L)
    torch.cuda.synchronize()
    for t in ("x", "q", "k"):
        assert np.array_equal(to_host(compact[t]), oracle.valid_gather(host[t], L)), f"gather {t}"
    y = tfk.tfk_rmsnorm_adaln_indexed(compact["x"], pd["w"], pd["shift"], pd["scale"], i32_dev(idx), wl.eps)
    qo, ko = tfk.tfk_qk_rmsnorm_rope_neox(compact["q"], compact["k"], pd["w_q"], pd["w_k"], i32_dev(pos),
                                          wl.n_heads, wl.head_dim, wl.theta, wl.eps)
    outs = {}
    for t, c in (("y", y), ("q", qo), ("k", ko)):
        g = Guarded(N, hidden)  # pre-filled with 0xFFFF: every row must be rewritten
        tfk.tfk_zero_tail_merge(c, g.view)
        outs[t] = (c, g)
    torch.cuda.synchronize()
    xc = oracle.valid_gather(host["x"], L)
    check_close(to_host(y), ora_adaln(xc, p["w"], p["shift"], p["scale"], idx, wl.eps), "valid-only a1")
    rq, rk = ora_qk(oracle.valid_gather(host["q"], L), oracle.valid_gather(host["k"], L), p["w_q"], p["w_k"],
                    pos, wl.n_heads, wl.head_dim, wl.theta, wl.eps)
    check_close(to_host(qo), rq, "valid-only a2 q")
    check_close(to_host(ko), rk, "valid-only a2 k")
    for t, (c, g) in outs.items():
        g.check()
        merged = g.host()
        assert np.array_equal(merged, oracle.zero_tail_merge(to_host(c), N)), f"merge {t}"
        assert np.all(merged[L:] == 0x0000) and not np.any(np.isnan(oracle.bf16_to_f64(merged)))


BLOCK = 4096  # rows per oracle block: bounds host memory on the full-size workloads


def _blocks(n: int, block: int = BLOCK):
    return [(s, min(n, s + block)) for s in range(0, n, block)]


def _host_and_dev(wl, tag: str, rows: int):
    """The first `rows` rows of an activation input, on the host and on the device."""
    host = synth.activation(wl, tag, rows=np.arange(rows))
    return host, to_dev(host)


def _report(stats: dict):
    for st in stats.values():
        print(st)


def _full_chain(wl):
    """Full-size chain on the GPU, every element of a1, a2 and a3 compared with the oracle,
    in blocks of rows (the oracle on all host threads)."""
    p, pd = _params_dev(wl)
    idx, pos = synth.mod_index(wl), synth.positions(wl)
    T = wl.rows
    stats = {k: Stats(f"{wl.name} {k}") for k in ("a1", "a2q", "a2k", "a3")}
    # one step at a time to bound host and device memory
    x, xd = _host_and_dev(wl, "x", T)
    y = tfk.tfk_rmsnorm_adaln_indexed(xd, pd["w"], pd["shift"], pd["scale"], i32_dev(idx), wl.eps)
    torch.cuda.synchronize()
    del xd
    for s, e in _blocks(T):
        stats["a1"].add(check_close(to_host(y[s:e]), ora_adaln(x[s:e], p["w"], p["shift"], p["scale"], idx[s:e],
                                                                wl.eps), f"{wl.name} a1 rows {s}:{e}"))
    del x, y
    q, qd = _host_and_dev(wl, "q", T)
    k, kd = _host_and_dev(wl, "k", T)
    qo, ko = tfk.tfk_qk_rmsnorm_rope_neox(qd, kd, pd["w_q"], pd["w_k"], i32_dev(pos), wl.n_heads, wl.head_dim,
                                          wl.theta, wl.eps)
    torch.cuda.synchronize()
    del qd, kd
    for s, e in _blocks(T):
        rq, rk = ora_qk(q[s:e], k[s:e], p["w_q"], p["w_k"], pos[s:e], wl.n_heads, wl.head_dim, wl.theta, wl.eps)
        stats["a2q"].add(check_close(to_host(qo[s:e]), rq, f"{wl.name} a2 q rows {s}:{e}"))
        stats["a2k"].add(check_close(to_host(ko[s:e]), rk, f"{wl.name} a2 k rows {s}:{e}"))
    del q, k, qo, ko
    gu, gud = _host_and_dev(wl, "gate_up", T)
    o = tfk.tfk_swiglu(gud)
    torch.cuda.synchronize()
    del gud
    for s, e in _blocks(T):
        stats["a3"].add(check_close(to_host(o[s:e]), ora_swiglu(gu[s:e]), f"{wl.name} a3 rows {s}:{e}"))
    del gu, o
    torch.cuda.empty_cache()
    out = {k: v.summary() for k, v in stats.items()}
    _report(out)
    assert out["a1"]["n"] == T * wl.hidden and out["a3"]["n"] == T * wl.ffn
    assert out["a2q"]["n"] == out["a2k"]["n"] == T * wl.n_heads * wl.head_dim
    return out


@pytest.mark.parametrize("rows,hidden", [(120000, 512), (50000, 3072), (20000, 16384), (12000, 20480)])
def test_adaln_chunked_schedule_sampled(cuda, rows, hidden):
    """Row counts where the CTA-per-row RMSNorm kernel hands out chunks (16 rows,
    24 for rows of 16 KB and more) instead of one persistent run per CTA (more than
    64 rows per resident CTA), the pair of CTAs per row at 20480, and the warp-per-row
    kernel at 3072: rows at chunk edges, the first and last rows and a seeded sample
    are recomputed by the oracle; the modulation row is drawn per token from three."""
    wl = synth.custom(f"chunked{hidden}", rows, hidden, 8, 64, 64, n_mod=3)
    rng = np.random.default_rng(rows + hidden)
    w, sh, sc = mod_params(rng, 3, hidden)
    idx = rng.integers(0, 3, rows).astype(np.int32)
    _, dev = _inputs_dev(wl, ["x"])
    y = tfk.tfk_rmsnorm_adaln_indexed(dev["x"], f32_dev(w), f32_dev(sh), f32_dev(sc), i32_dev(idx), 1e-6)
    torch.cuda.synchronize()
    del dev
    edges = np.arange(0, rows, 16 if hidden * 2 < 16384 else 24)
    sample = np.unique(np.r_[edges[::97], edges[::89] - 1, synth.sample_rows(wl, 160)].clip(0, rows - 1))
    got = to_host(y[torch.from_numpy(sample).cuda()])
    del y
    torch.cuda.empty_cache()
    xs = synth.activation(wl, "x", rows=sample)
    check_close(got, ora_adaln(xs, w, sh, sc, idx[sample], 1e-6), f"a1 chunked hidden {hidden}")


def test_large_full(cuda):
    """The 75,600-token workload: every output element of the chain (including all 756
    outlier rows) against the oracle."""
    _full_chain(synth.get("large"))


def test_per_frame_full(cuda):
    _full_chain(synth.get("per_frame"))


def test_over_2g_elements_indexing(cuda):
    """SwiGLU and the merge on buffers of more than 2^31 elements (64-bit indexing):
    a seeded block is tiled on the device and sampled rows are checked."""
    rng = np.random.default_rng(11)
    ffn, rows = 14336, 75000                           # gate_up: 75000 x 28672 = 2.15e9 elements
    block = rand_bits(rng, (64, 2 * ffn), 3.0)
    gu = to_dev(block).repeat(rows // 64 + 1, 1)[:rows]
    assert gu.numel() > 2**31
    o = tfk.tfk_swiglu(gu)
    torch.cuda.synchronize()
    sample = np.r_[0, 1, rng.integers(0, rows, 60), rows - 1]
    check_close(to_host(o[torch.from_numpy(sample).cuda()]), ora_swiglu(block[sample % 64]), "swiglu > 2^31")
    del o
    hidden, N = 8192, 270000                           # 2.2e9 elements
    L = N - 12345
    comp = to_dev(block[:, :hidden]).repeat(L // 64 + 1, 1)[:L]
    padded = torch.empty((N, hidden), dtype=torch.bfloat16, device="cuda")
    tfk.tfk_zero_tail_merge(comp, padded)
    torch.cuda.synchronize()
    tail = padded[L:].view(torch.int16)
    assert int((tail != 0).sum()) == 0
    idx = torch.from_numpy(np.r_[0, L - 1, rng.integers(0, L, 30)]).cuda()
    assert torch.equal(padded[idx].view(torch.int16), comp[idx].view(torch.int16))
    del gu, comp, padded
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# fixed-valid mode: the normalisation kernels on the padded buffer directly
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,L,H", [(64, 0, 8), (64, 64, 8), (1000, 777, 8), (4096, 1, 8),
                                   (1001, 555, 3)])   # 3 heads: two token streams per CTA, tail split too
def test_fixed_valid_adaln_and_qk(cuda, N, L, H):
    rng = np.random.default_rng(N + 3 * L)
    hidden, D = 1024, 128
    x = rand_bits(rng, (N, hidden))
    q = rand_bits(rng, (N, H * D), 2.0)
    k = rand_bits(rng, (N, H * D))
    for a in (x, q, k):
        a[L:] = synth.BF16_NAN                        # the padded tail must never be read
    w, sh, sc = mod_params(rng, 3, hidden)
    idx = rng.integers(0, 3, L).astype(np.int32)
    pos = rng.integers(0, 70000, L).astype(np.int32)
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
    check_close(y.host(), oracle.rmsnorm_adaln_fixed_valid(x, L, w, sh, sc, idx, 1e-6, threads=THREADS),
                "fixed-valid a1")
    rq, rk = oracle.qk_rmsnorm_rope_neox_fixed_valid(q, k, L, wq, wk, pos, H, D, 10000.0, 1e-6, threads=THREADS)
    check_close(qo.host(), rq.reshape(N, -1), "fixed-valid q")
    check_close(ko.host(), rk.reshape(N, -1), "fixed-valid k")


@pytest.mark.parametrize("N,L,hidden", [(500, 333, 20480), (300, 300, 6144), (257, 0, 32768)])
def test_fixed_valid_adaln_wide_rows(cuda, N, L, hidden):
    """Fixed-valid RMSNorm+AdaLN on the wide-row paths (a pair of CTAs per row; the warp
    kernel at 6144): valid rows against the oracle, the tail +0.0, NaN tail never read."""
    rng = np.random.default_rng(N + L + hidden)
    x = rand_bits(rng, (N, hidden))
    x[L:] = synth.BF16_NAN
    w, sh, sc = mod_params(rng, 3, hidden)
    idx = rng.integers(0, 3, L).astype(np.int32)
    y = Guarded(N, hidden)
    tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(to_dev(x), L, f32_dev(w), f32_dev(sh), f32_dev(sc), i32_dev(idx),
                                              1e-6, out=y.view)
    torch.cuda.synchronize()
    y.check()
    got = y.host()
    assert np.all(got[L:] == 0x0000)
    check_close(got, oracle.rmsnorm_adaln_fixed_valid(x, L, w, sh, sc, idx, 1e-6, threads=THREADS),
                f"fixed-valid a1 hidden {hidden}")


def test_fixed_valid_in_place_on_the_valid_only_workload(cuda):
    """The valid-only workload without gather and merge: in place on the padded buffers,
    every valid element against the oracle and every tail element +0.0."""
    wl = synth.get("valid_only")
    N, L = wl.rows, synth.valid_len(wl)
    host, dev = _inputs_dev(wl, ["x", "q", "k"])
    p, pd = _params_dev(wl)
    idx = synth.mod_index(wl, np.arange(L))
    pos = synth.positions(wl, np.arange(L))
    tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(dev["x"], L, pd["w"], pd["shift"], pd["scale"], i32_dev(idx),
                                              wl.eps, out=dev["x"])
    tfk.tfk_qk_rmsnorm_rope_neox_fixed_valid(dev["q"], dev["k"], L, pd["w_q"], pd["w_k"], i32_dev(pos),
                                             wl.n_heads, wl.head_dim, wl.theta, wl.eps,
                                             q_out=dev["q"], k_out=dev["k"])
    torch.cuda.synchronize()
    y, qo, ko = (to_host(dev[t]) for t in ("x", "q", "k"))
    del dev
    for a in (y, qo, ko):
        assert np.all(a[L:] == 0x0000)
    stats = {k: Stats(f"valid_only fixed-valid {k}") for k in ("a1", "a2q", "a2k")}
    for s, e in _blocks(L):
        stats["a1"].add(check_close(y[s:e], ora_adaln(host["x"][s:e], p["w"], p["shift"], p["scale"], idx[s:e],
                                                       wl.eps), f"valid-only fixed-valid a1 rows {s}:{e}"))
        rq, rk = ora_qk(host["q"][s:e], host["k"][s:e], p["w_q"], p["w_k"], pos[s:e], wl.n_heads,
                        wl.head_dim, wl.theta, wl.eps)
        stats["a2q"].add(check_close(qo[s:e], rq, f"valid-only fixed-valid q rows {s}:{e}"))
        stats["a2k"].add(check_close(ko[s:e], rk, f"valid-only fixed-valid k rows {s}:{e}"))
    out = {k: v.summary() for k, v in stats.items()}
    _report(out)
    assert out["a1"]["n"] == L * wl.hidden


# ---------------------------------------------------------------------------
# Ulysses: packing fused into Q/K norm + RoPE, and the standalone relayout
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,H,D,P", [(50, 8, 128, 1), (50, 8, 128, 2), (129, 24, 128, 4), (33, 40, 128, 8),
                                        (17, 6, 64, 3),
                                        (21, 25, 128, 5),   # 4 heads per lane group, the last one masked,
                                        (9, 30, 96, 3),     # groups spanning two ranks' blocks
                                        (15, 6, 128, 2), (11, 9, 64, 3),   # 3 heads per lane group
                                        (13, 12, 128, 4), (9, 4, 64, 2)])  # four token streams per CTA
def test_qk_ulysses_send_layout(cuda, rows, H, D, P):
    rng = np.random.default_rng(rows + 100 * P)
    q = rand_bits(rng, (rows, H * D))
    k = rand_bits(rng, (rows, H * D), 2.0)
    wq = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    pos = rng.integers(0, 75600, rows).astype(np.int32)
    qs, ks = tfk.tfk_qk_rmsnorm_rope_neox_ulysses(to_dev(q), to_dev(k), f32_dev(wq), f32_dev(wk), i32_dev(pos),
                                                  H, D, P)
    torch.cuda.synchronize()
    rq, rk = ora_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    check_close(to_host(qs).reshape(-1), oracle.ulysses_pack(rq, H, D, P).reshape(-1), f"ulysses q P={P}")
    check_close(to_host(ks).reshape(-1), oracle.ulysses_pack(rk, H, D, P).reshape(-1), f"ulysses k P={P}")


@pytest.mark.parametrize("rows,H,D,P,stride_pad", [(1, 1, 8, 1, 0), (100, 24, 128, 4, 0), (77, 40, 128, 8, 64),
                                                   (5, 6, 40, 3, 8),
                                                   (1003, 24, 128, 4, 0),   # many 4-row tiles, ragged last tile
                                                   (203, 64, 128, 8, 0),    # 8192 values per row: 4 vectors per thread
                                                   (37, 72, 128, 8, 16)])   # 9216 values: the column-walking kernel
def test_ulysses_pack_unpack_bit_exact(cuda, rows, H, D, P, stride_pad):
    rng = np.random.default_rng(rows * H + P)
    x = rng.integers(0, 65536, (rows, H * D), dtype=np.uint32).astype(np.uint16)
    src = Guarded(rows, H * D, H * D + stride_pad)
    src.view.copy_(to_dev(x))
    packed = tfk.tfk_ulysses_pack(src.view, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(packed), oracle.ulysses_pack(x, H, D, P))
    back = Guarded(rows, H * D, H * D + stride_pad)
    tfk.tfk_ulysses_unpack(packed, H, D, P, dst=back.view)
    torch.cuda.synchronize()
    back.check()
    src.check()
    assert np.array_equal(back.host(), x)


def test_qk_ulysses_full_size(cuda):
    """The fused Ulysses packing on the 75,600-token workload for 8 ranks (5 heads per rank):
    every element of both send buffers against the oracle's permutation of its Q/K result."""
    wl = synth.get("large")
    P, T, H, D = 8, wl.rows, wl.n_heads, wl.head_dim
    p, pd = _params_dev(wl)
    pos = synth.positions(wl)
    q, qd = _host_and_dev(wl, "q", T)
    k, kd = _host_and_dev(wl, "k", T)
    qs, ks = tfk.tfk_qk_rmsnorm_rope_neox_ulysses(qd, kd, pd["w_q"], pd["w_k"], i32_dev(pos), H, D, P)
    torch.cuda.synchronize()
    del qd, kd
    stats = {"q": Stats("ulysses q P=8"), "k": Stats("ulysses k P=8")}
    for s, e in _blocks(T):
        rq, rk = ora_qk(q[s:e], k[s:e], p["w_q"], p["w_k"], pos[s:e], H, D, wl.theta, wl.eps)
        stats["q"].add(check_close(to_host(qs[:, s:e]).reshape(-1), oracle.ulysses_pack(rq, H, D, P).reshape(-1),
                                   f"ulysses q P={P} rows {s}:{e}"))
        stats["k"].add(check_close(to_host(ks[:, s:e]).reshape(-1), oracle.ulysses_pack(rk, H, D, P).reshape(-1),
                                   f"ulysses k P={P} rows {s}:{e}"))
    out = {k: v.summary() for k, v in stats.items()}
    _report(out)
    assert out["q"]["n"] == out["k"]["n"] == T * H * D
    del qs, ks
    torch.cuda.empty_cache()


def test_qk_ulysses_full_size_sampled_p4(cuda):
    """The same on 4 ranks (10 heads per rank), on a seeded sample of rows."""
    wl = synth.get("large")
    P = 4
    p, pd = _params_dev(wl)
    rows = synth.sample_rows(wl, 96)
    _, dev = _inputs_dev(wl, ["q", "k"])
    qs, ks = tfk.tfk_qk_rmsnorm_rope_neox_ulysses(dev["q"], dev["k"], pd["w_q"], pd["w_k"],
                                                  i32_dev(synth.positions(wl)), wl.n_heads, wl.head_dim, P)
    torch.cuda.synchronize()
    sel = torch.from_numpy(rows).cuda()
    got_q = to_host(qs[:, sel])                    # [P, sample, H/P, D]
    got_k = to_host(ks[:, sel])
    del dev, qs, ks
    rq, rk = ora_qk(synth.activation(wl, "q", rows=rows), synth.activation(wl, "k", rows=rows), p["w_q"], p["w_k"],
                    synth.positions(wl, rows), wl.n_heads, wl.head_dim, wl.theta, wl.eps)
    check_close(got_q.reshape(-1), oracle.ulysses_pack(rq, wl.n_heads, wl.head_dim, P).reshape(-1), f"ulysses q P={P}")
    check_close(got_k.reshape(-1), oracle.ulysses_pack(rk, wl.n_heads, wl.head_dim, P).reshape(-1), f"ulysses k P={P}")
    torch.cuda.empty_cache()
