"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a closed form, a library routine
(torch fp64 ``rms_norm`` / ``silu``, numpy complex arithmetic, mpmath), an
invariant of the definition, or a special case that reduces to one of those,
chosen so that a plausible slip (a dropped term, a wrong sign or index, a
transposed operand, a mean taken over the wrong axis) fails at least one.
No GPU is involved.
"""
import math
import struct

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

RNG = np.random.default_rng(12345)


def bf16(a) -> np.ndarray:
    """float array -> raw bf16 bits through torch's RNE cast (test-side input helper)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------------------
# rounding and widening
# ---------------------------------------------------------------------------

def test_widening_matches_torch_for_every_bf16_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    a = oracle.bf16_to_f64(bits)
    b = f64(bits)
    finite = np.isfinite(b)
    assert np.array_equal(a[finite], b[finite])
    assert np.array_equal(np.isnan(a), np.isnan(b))


def test_round_is_identity_on_every_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_to_f64(bits)
    ok = np.isfinite(v)
    assert np.array_equal(oracle.round_bf16(v[ok]), bits[ok])


def test_round_matches_torch_rne_cast_of_fp32_values():
    # for doubles that are exactly fp32 values, one RNE rounding to bf16 is what
    # torch's float32 -> bfloat16 cast does
    x = np.concatenate([RNG.standard_normal(200000) * 10.0 ** RNG.integers(-30, 30, 200000),
                        RNG.standard_normal(1000) * 1e-39]).astype(np.float32)
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), bf16(x))


def test_round_thread_split_changes_nothing():
    v = RNG.standard_normal(100003) * 10.0 ** RNG.integers(-8, 8, 100003)
    assert np.array_equal(oracle.round_bf16(v, threads=7), oracle.round_bf16(v))


def test_round_ties_go_to_even_and_off_ties_go_to_nearest():
    lo = bf16(RNG.uniform(-100, 100, 5000))
    lo = lo[(lo & 0x7F80) != 0x7F80]
    lo = lo[(lo & 0x7F) != 0x7F]                    # next pattern stays in the binade
    hi = lo + 1
    a, b = oracle.bf16_to_f64(lo), oracle.bf16_to_f64(hi)
    mid = (a + b) / 2.0                              # exact in double
    got = oracle.round_bf16(mid)
    even = np.where((lo & 1) == 0, lo, hi)
    assert np.array_equal(got, even)
    gap = np.abs(b - a)
    assert np.array_equal(oracle.round_bf16(mid + np.sign(b - a) * gap * 1e-6), hi)
    assert np.array_equal(oracle.round_bf16(mid - np.sign(b - a) * gap * 1e-6), lo)


def test_round_special_values():
    r = oracle.round_bf16(np.array([0.0, -0.0, np.inf, -np.inf, 3.5e38, -3.5e38, 1e-45, np.nan]))
    assert r[0] == 0x0000 and r[1] == 0x8000
    assert r[2] == 0x7F80 and r[3] == 0xFF80
    assert r[4] == 0x7F80 and r[5] == 0xFF80            # above the largest bf16 (3.39e38)
    assert r[6] == 0x0000                               # far below the smallest subnormal 2^-133
    assert (r[7] & 0x7F80) == 0x7F80 and (r[7] & 0x7F)
    assert oracle.round_bf16(np.array([2.0 ** -133]))[0] == 0x0001
    assert oracle.round_bf16(np.array([3.0 * 2.0 ** -134]))[0] == 0x0002   # tie 1.5 -> 2


# ---------------------------------------------------------------------------
# RMSNorm + indexed AdaLN modulation
# ---------------------------------------------------------------------------

def _mod_inputs(rows, hidden, n_mod, seed=0):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal((rows, hidden)) * rng.uniform(0.1, 5, (rows, 1)))
    w = (1 + 0.1 * rng.standard_normal(hidden)).astype(np.float32)
    shift = (0.1 * rng.standard_normal((n_mod, hidden))).astype(np.float32)
    scale = (0.1 * rng.standard_normal((n_mod, hidden))).astype(np.float32)
    idx = rng.integers(0, n_mod, rows).astype(np.int32)
    return x, w, shift, scale, idx


@pytest.mark.parametrize("hidden", [8, 512, 3072])
def test_adaln_reduces_to_torch_rms_norm(hidden):
    x, w, shift, scale, idx = _mod_inputs(37, hidden, 3)
    zeros = np.zeros_like(shift)
    eps = 1e-6
    y = oracle.rmsnorm_adaln_indexed(x, np.ones(hidden, np.float32), zeros, zeros, idx, eps)
    ref = F.rms_norm(torch.from_numpy(f64(x)), (hidden,), eps=eps).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)
    yw = oracle.rmsnorm_adaln_indexed(x, w, zeros, zeros, idx, eps)
    refw = F.rms_norm(torch.from_numpy(f64(x)), (hidden,), weight=torch.from_numpy(w.astype(np.float64)),
                      eps=eps).numpy()
    np.testing.assert_allclose(yw, refw, rtol=1e-13, atol=1e-15)


def test_adaln_scale_minus_one_returns_the_selected_shift_row():
    x, w, shift, _, idx = _mod_inputs(64, 256, 5)
    scale = -np.ones_like(shift)
    y = oracle.rmsnorm_adaln_indexed(x, w, shift, scale, idx, 1e-6)
    assert np.array_equal(y, shift[idx].astype(np.float64))


def test_adaln_modulation_is_one_plus_scale_then_shift():
    # with w = 1: y - shift[m] = rmsnorm(x) * (1 + scale[m]); checked against torch's
    # rms_norm for two different modulation rows chosen per token
    x, _, shift, scale, idx = _mod_inputs(50, 384, 2)
    ones = np.ones(384, np.float32)
    y = oracle.rmsnorm_adaln_indexed(x, ones, shift, scale, idx, 1e-6)
    n = F.rms_norm(torch.from_numpy(f64(x)), (384,), eps=1e-6).numpy()
    expect = n * (1.0 + scale[idx].astype(np.float64)) + shift[idx].astype(np.float64)
    np.testing.assert_allclose(y, expect, rtol=1e-13, atol=1e-14)
    # swapping the two modulation rows changes every output row
    y2 = oracle.rmsnorm_adaln_indexed(x, ones, shift, scale, 1 - idx, 1e-6)
    assert np.all(np.abs(y2 - y).max(axis=1) > 1e-3)


def test_adaln_constant_row_closed_form_shows_eps_inside_the_root():
    hidden, eps = 64, 1e-6
    for c in (2.0 ** -10, 0.5, 3.0, -7.0):
        x = bf16(np.full((1, hidden), c))
        zeros = np.zeros((1, hidden), np.float32)
        y = oracle.rmsnorm_adaln_indexed(x, np.ones(hidden, np.float32), zeros, zeros,
                                         np.zeros(1, np.int32), eps)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-15)


def test_adaln_zero_row_gives_shift():
    hidden = 128
    x = np.zeros((3, hidden), np.uint16)
    _, w, shift, scale, _ = _mod_inputs(3, hidden, 3)
    idx = np.array([2, 0, 1], np.int32)
    y = oracle.rmsnorm_adaln_indexed(x, w, shift, scale, idx, 1e-6)
    assert np.array_equal(y, shift[idx].astype(np.float64))


def test_adaln_output_mean_square_with_unit_weight():
    x, _, _, _, idx = _mod_inputs(20, 1024, 1)
    zeros = np.zeros((1, 1024), np.float32)
    eps = 1e-2  # large enough that the eps term is visible
    y = oracle.rmsnorm_adaln_indexed(x, np.ones(1024, np.float32), zeros, zeros, np.zeros(20, np.int32), eps)
    ms = (f64(x) ** 2).mean(axis=1)
    np.testing.assert_allclose((y ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)


def test_adaln_row_stride_and_thread_split_do_not_change_results():
    x, w, shift, scale, idx = _mod_inputs(33, 256, 3)
    wide = np.zeros((33, 256 + 24), np.uint16) + 0x7FC0
    wide[:, :256] = x
    a = oracle.rmsnorm_adaln_indexed(x, w, shift, scale, idx, 1e-6)
    b = oracle.rmsnorm_adaln_indexed(wide[:, :256], w, shift, scale, idx, 1e-6, threads=4)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# per-head RMSNorm + NeoX RoPE
# ---------------------------------------------------------------------------

def test_head_rmsnorm_matches_torch_per_head_not_per_row():
    rows, H, D = 9, 6, 64
    rng = np.random.default_rng(3)
    v = rng.standard_normal((rows, H, D)) * (10.0 ** np.arange(H))[None, :, None]
    vb = bf16(v.reshape(rows, H * D))
    w = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    got = oracle.head_rmsnorm(vb, H, D, w, 1e-6)
    ref = F.rms_norm(torch.from_numpy(f64(vb).reshape(rows, H, D)), (D,),
                     weight=torch.from_numpy(w.astype(np.float64)), eps=1e-6).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def _rope_input(rows, H, D, seed=0):
    return np.random.default_rng(seed).standard_normal((rows, H, D))


def test_rope_position_zero_is_identity():
    v = _rope_input(5, 3, 128)
    out = oracle.rope_neox(v, np.zeros(5, np.int32), 10000.0)
    assert np.array_equal(out, v)


@pytest.mark.parametrize("D", [8, 128])
def test_rope_is_complex_rotation_with_hand_derived_frequencies(D):
    # NeoX pairing (i, i + D/2) read as z = v[i] + 1j*v[i + D/2]; RoPE multiplies z by
    # exp(1j*pos*f_i).  With base 10000, f_i = 10000^(-2i/D): for D=8 that is
    # 1, 0.1, 0.01, 0.001; for D=128, i = 0, 16, 32, 48 give 1, 0.1, 0.01, 0.001.
    hand = {8: {0: 1.0, 1: 0.1, 2: 0.01, 3: 0.001}, 128: {0: 1.0, 16: 0.1, 32: 0.01, 48: 0.001}}[D]
    rows, H = 6, 2
    v = _rope_input(rows, H, D, 7)
    pos = np.array([0, 1, 2, 17, 4096, 75599], np.int32)
    out = oracle.rope_neox(v, pos, 10000.0)
    half = D // 2
    for i, f in hand.items():
        z = v[:, :, i] + 1j * v[:, :, i + half]
        rot = z * np.exp(1j * (pos.astype(np.float64) * f))[:, None]
        np.testing.assert_allclose(out[:, :, i], rot.real, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(out[:, :, i + half], rot.imag, rtol=1e-9, atol=1e-9)


def test_rope_preserves_every_rotate_half_pair_norm():
    D = 64
    v = _rope_input(8, 4, D, 11)
    out = oracle.rope_neox(v, np.arange(8, dtype=np.int32) * 997, 10000.0)
    h = D // 2
    np.testing.assert_allclose(out[..., :h] ** 2 + out[..., h:] ** 2, v[..., :h] ** 2 + v[..., h:] ** 2,
                               rtol=1e-12)


def test_rope_composes_additively():
    v = _rope_input(4, 2, 32, 5)
    p1 = np.array([3, 100, 5000, 31], np.int32)
    p2 = np.array([11, 7, 20000, 0], np.int32)
    twice = oracle.rope_neox(oracle.rope_neox(v, p1, 10000.0), p2, 10000.0)
    once = oracle.rope_neox(v, p1 + p2, 10000.0)
    np.testing.assert_allclose(twice, once, rtol=1e-9, atol=1e-11)


def test_rope_dot_product_depends_only_on_relative_position():
    D = 128
    q = _rope_input(1, 1, D, 1)
    k = _rope_input(1, 1, D, 2)
    dots = []
    for m, n in [(10, 3), (1010, 1003), (70007, 70000)]:
        rq = oracle.rope_neox(q, np.array([m], np.int32), 10000.0)
        rk = oracle.rope_neox(k, np.array([n], np.int32), 10000.0)
        dots.append(float((rq * rk).sum()))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    rk = oracle.rope_neox(k, np.array([5], np.int32), 10000.0)
    rq = oracle.rope_neox(q, np.array([10], np.int32), 10000.0)
    assert abs(float((rq * rk).sum()) - dots[0]) > 1e-3   # a different offset gives a different dot


def test_rope_angles_at_large_positions_agree_with_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    D = 128
    v = np.zeros((3, 1, D))
    v[:, :, :D // 2] = 1.0                      # z_i = 1 -> out = (cos, sin)
    pos = np.array([1, 56319, 75599], np.int32)
    out = oracle.rope_neox(v, pos, 10000.0)
    for t, p in enumerate(pos):
        for i in (0, 1, 5, 31, 63):
            ang = mpmath.mpf(int(p)) * mpmath.power(10000, mpmath.mpf(-2 * i) / D)
            assert abs(out[t, 0, i] - float(mpmath.cos(ang))) < 1e-11
            assert abs(out[t, 0, i + D // 2] - float(mpmath.sin(ang))) < 1e-11


def test_qk_uses_its_own_weight_for_q_and_for_k():
    rows, H, D = 7, 4, 64
    rng = np.random.default_rng(9)
    q = bf16(rng.standard_normal((rows, H * D)))
    k = bf16(rng.standard_normal((rows, H * D)))
    wq = (1 + 0.3 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.3 * rng.standard_normal(D)).astype(np.float32)
    pos = np.zeros(rows, np.int32)
    qo, ko = oracle.qk_rmsnorm_rope_neox(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
    tq = F.rms_norm(torch.from_numpy(f64(q).reshape(rows, H, D)), (D,), torch.from_numpy(wq.astype(np.float64)), 1e-6)
    tk = F.rms_norm(torch.from_numpy(f64(k).reshape(rows, H, D)), (D,), torch.from_numpy(wk.astype(np.float64)), 1e-6)
    np.testing.assert_allclose(qo, tq.numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(ko, tk.numpy(), rtol=1e-13, atol=1e-15)
    # and with positions the fused call is norm followed by rotation
    pos = np.arange(rows, dtype=np.int32) * 1234
    qo, ko = oracle.qk_rmsnorm_rope_neox(q, k, wq, wk, pos, H, D, 10000.0, 1e-6, threads=3)
    assert np.array_equal(qo, oracle.rope_neox(oracle.head_rmsnorm(q, H, D, wq, 1e-6), pos, 10000.0))
    assert np.array_equal(ko, oracle.rope_neox(oracle.head_rmsnorm(k, H, D, wk, 1e-6), pos, 10000.0))


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def test_swiglu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 2.0, 1.0, -20.0, 20.0])
    u = np.array([5.0, 1.0, 1.0, 0.5, 2.0, 1.0, 1.0])
    gu = bf16(np.concatenate([g, u])[None, :])
    out = oracle.swiglu(gu)[0]
    assert out[0] == 0.0                                        # silu(0) = 0
    np.testing.assert_allclose(out[1], 0.7310585786300049, rtol=1e-15)   # 1/(1+e^-1)
    np.testing.assert_allclose(out[2], -0.2689414213699951, rtol=1e-15)  # -1/(1+e)
    np.testing.assert_allclose(out[3], 0.5 * 2.0 / (1.0 + math.exp(-2.0)), rtol=1e-15)
    np.testing.assert_allclose(out[4], 2.0 * 0.7310585786300049, rtol=1e-15)
    assert abs(out[5]) < 1e-7 and abs(out[6] - 20.0) < 1e-6


def test_swiglu_gate_is_the_first_half():
    rng = np.random.default_rng(4)
    g = rng.standard_normal((5, 96)) * 3
    gu = bf16(np.concatenate([g, np.ones_like(g)], axis=1))
    out = oracle.swiglu(gu)
    np.testing.assert_allclose(out, F.silu(torch.from_numpy(f64(gu)[:, :96])).numpy(), rtol=1e-14, atol=1e-300)


def test_swiglu_matches_torch_silu_times_up():
    rng = np.random.default_rng(5)
    gu = bf16(rng.standard_normal((17, 2 * 200)) * 4)
    wide = np.full((17, 400 + 16), 0x7FC0, np.uint16)
    wide[:, :400] = gu
    out = oracle.swiglu(wide[:, :400], threads=4)
    t = torch.from_numpy(f64(gu))
    ref = (F.silu(t[:, :200]) * t[:, 200:]).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-300)


# ---------------------------------------------------------------------------
# valid-only gather / zero-tail merge
# ---------------------------------------------------------------------------

def _padded(N, hidden, L, seed=0):
    rng = np.random.default_rng(seed)
    p = rng.integers(0, 65536, (N, hidden), dtype=np.uint32).astype(np.uint16)
    p[L:] = 0x7FC0
    return p


def test_gather_is_the_valid_prefix_and_merge_zeroes_the_tail():
    N, hidden, L = 40, 24, 29
    p = _padded(N, hidden, L)
    c = oracle.valid_gather(p, L)
    assert np.array_equal(c, p[:L])
    m = oracle.zero_tail_merge(c, N)
    assert np.array_equal(m[:L], p[:L])
    assert np.all(m[L:] == 0x0000)                    # +0.0, never -0.0 or NaN
    assert not np.any((m[L:] & 0x7F80) == 0x7F80)


def test_gather_merge_round_trip_keeps_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(2048, 32)
    N = 2048 + 100
    p = np.full((N, 32), 0x7FC0, np.uint16)
    p[:2048] = bits
    m = oracle.zero_tail_merge(oracle.valid_gather(p, 2048), N)
    assert np.array_equal(m[:2048], bits) and np.all(m[2048:] == 0)


def test_gather_merge_degenerate_lengths():
    p = _padded(16, 8, 16)
    assert np.array_equal(oracle.zero_tail_merge(oracle.valid_gather(p, 16), 16), p)
    z = oracle.zero_tail_merge(oracle.valid_gather(p, 0), 16)
    assert z.shape == (16, 8) and np.all(z == 0)


# ---------------------------------------------------------------------------
# the generator gives the oracle what the workload recipes state
# ---------------------------------------------------------------------------

def test_workload_recipes():
    t = synth.get("tiny")
    assert np.array_equal(synth.mod_index(t), np.r_[np.zeros(256), np.ones(64)].astype(np.int32))
    assert np.array_equal(synth.positions(t), np.arange(320))
    m = synth.get("medium")
    idx = synth.mod_index(m)
    assert set(idx[:7168]) == {0, 1} and set(idx[7168:]) == {2, 3}
    assert synth.positions(m)[7168] == 0 and synth.positions(m)[8191] == 1023
    v = synth.get("valid_only")
    L = synth.valid_len(v)
    assert 24000 <= L <= 32768
    xs = synth.activation(v, "x", rows=[L - 1, L, v.rows - 1])
    assert np.all(xs[1:] == synth.BF16_NAN) and not np.any(xs[0] == synth.BF16_NAN)
    lg = synth.get("large")
    out = synth.outlier_rows(lg)
    assert len(out) == 756 and len(set(out)) == 756
    a = f64(synth.activation(lg, "x", rows=out[:3]))
    b = f64(synth.activation(lg, "x", rows=[r for r in range(10) if r not in set(out)]))
    assert np.abs(a).mean() > 20 * np.abs(b).mean()
    pf = synth.get("per_frame")
    idx = synth.mod_index(pf)
    assert idx[0] == 0 and idx[2047] == 0 and idx[2048] == 1 and idx[55295] == 26 and idx[55296] == 27
    # a subset of rows is the same rows of the full tensor
    full = synth.activation(t, "gate_up")
    assert np.array_equal(synth.activation(t, "gate_up", rows=[3, 4, 200, 319]), full[[3, 4, 200, 319]])


# ---------------------------------------------------------------------------
# Ulysses relayout
# ---------------------------------------------------------------------------

def test_ulysses_pack_feeds_an_all_to_all_that_shards_heads():
    # P ranks each hold T tokens of all H heads; after pack on every rank and the
    # all-to-all (rank p receives block p from every rank, in rank order), rank p
    # must hold heads [p*H/P, (p+1)*H/P) of all P*T tokens in sequence order.
    P, T, H, D = 4, 5, 8, 16
    glob = np.random.default_rng(0).integers(0, 65536, (P * T, H * D)).astype(np.uint16)
    sent = [oracle.ulysses_pack(glob[s * T:(s + 1) * T], H, D, P) for s in range(P)]
    for p in range(P):
        received = np.concatenate([sent[s][p] for s in range(P)])          # [P*T, H/P, D]
        expect = glob.reshape(P * T, H, D)[:, p * H // P:(p + 1) * H // P, :]
        assert np.array_equal(received, expect)


def test_ulysses_degree_one_is_identity_and_unpack_inverts_pack():
    x = np.random.default_rng(1).integers(0, 65536, (7, 6 * 32)).astype(np.uint16)
    assert np.array_equal(oracle.ulysses_pack(x, 6, 32, 1).reshape(7, -1), x)
    for P in (1, 2, 3, 6):
        assert np.array_equal(oracle.ulysses_unpack(oracle.ulysses_pack(x, 6, 32, P), 6, 32, P), x)


def test_fixed_valid_oracle_is_the_plain_definition_then_zeros():
    x, w, shift, scale, idx = _mod_inputs(40, 128, 3)
    full = oracle.rmsnorm_adaln_indexed(x, w, shift, scale, idx, 1e-6)
    assert np.array_equal(oracle.rmsnorm_adaln_fixed_valid(x, 40, w, shift, scale, idx, 1e-6), full)
    part = oracle.rmsnorm_adaln_fixed_valid(x, 25, w, shift, scale, idx, 1e-6)
    assert np.array_equal(part[:25], full[:25]) and np.all(part[25:] == 0.0)
    assert np.all(oracle.round_bf16(part[25:]) == 0x0000)                 # +0.0, not -0.0
    q = bf16(np.random.default_rng(2).standard_normal((40, 2 * 64)))
    wq = np.ones(64, np.float32)
    pos = np.arange(40, dtype=np.int32)
    qf, kf = oracle.qk_rmsnorm_rope_neox(q, q, wq, wq, pos, 2, 64, 10000.0, 1e-6)
    qp, kp = oracle.qk_rmsnorm_rope_neox_fixed_valid(q, q, 30, wq, wq, pos, 2, 64, 10000.0, 1e-6)
    assert np.array_equal(qp[:30], qf[:30]) and np.all(qp[30:] == 0.0) and np.array_equal(kp[:30], kf[:30])


# ---------------------------------------------------------------------------
# brute force on 4 tokens: every operation restated as scalar long-double
# loops written here (no code of oracle.c), RoPE as an explicit D x D
# block-rotation matrix per token, compared with the oracle's loop form
# ---------------------------------------------------------------------------

LD = np.longdouble
BRUTE_POS = np.array([0, 1, 4096, 75599], np.int32)   # first, second, a mid and the largest workload position


def _bf16_value(bits: int) -> float:
    """Value of one raw bf16 pattern: the top half of an IEEE binary32 (struct, not the oracle)."""
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _row_ld(bits_row) -> list:
    return [LD(_bf16_value(b)) for b in bits_row]


def _brute_adaln(x_bits, w, shift, scale, idx, eps):
    rows, hidden = x_bits.shape
    out = np.empty((rows, hidden), LD)
    for t in range(rows):
        xs = _row_ld(x_bits[t])
        ss = LD(0)
        for v in xs:
            ss += v * v
        r = LD(1) / np.sqrt(ss / LD(hidden) + LD(eps))
        m = int(idx[t])
        for j in range(hidden):
            out[t, j] = xs[j] * r * LD(float(w[j])) * (LD(1) + LD(float(scale[m, j]))) + LD(float(shift[m, j]))
    return out


def _rotation_matrix(pos: int, D: int, base: float) -> np.ndarray:
    """The NeoX rotary map of one token as a D x D matrix: plane (i, i + D/2) turned by
    pos * base^(-2i/D), every other coordinate untouched by that plane's rotation."""
    half = D // 2
    R = np.zeros((D, D), LD)
    for i in range(half):
        ang = LD(int(pos)) * np.power(LD(base), LD(-2 * i) / LD(D))
        c, s_ = np.cos(ang), np.sin(ang)
        R[i, i], R[i, i + half] = c, -s_
        R[i + half, i], R[i + half, i + half] = s_, c
    return R


def _brute_head_norm(bits_row, H, D, w, eps) -> np.ndarray:
    out = np.empty((H, D), LD)
    for h in range(H):
        v = _row_ld(bits_row[h * D:(h + 1) * D])
        ss = LD(0)
        for a in v:
            ss += a * a
        r = LD(1) / np.sqrt(ss / LD(D) + LD(eps))
        for d in range(D):
            out[h, d] = v[d] * r * LD(float(w[d]))
    return out


def _rope_tol(pos, n) -> np.ndarray:
    """1e-12, plus what fp64 can do no better than: the oracle forms pos * base^(-2i/D) in
    double (pow within 1 ulp, the product within half an ulp), so its angle is off by at
    most ~3.3e-16 * |pos| rad, which moves a pair of norm <= sqrt(2) max|n| by that much."""
    return 1e-12 + 5e-16 * np.abs(pos.astype(np.float64))[:, None, None] * np.abs(n).max(axis=(1, 2))[:, None, None]


@pytest.mark.parametrize("D", [8, 64, 128])
def test_brute_force_4_tokens_qk_rotation_matrix(D):
    H, eps, base = 2, 1e-6, 10000.0
    rng = np.random.default_rng(D)
    q = bf16(rng.standard_normal((4, H * D)) * 2.0)
    k = bf16(rng.standard_normal((4, H * D)) * 0.5)
    wq = (1 + 0.2 * rng.standard_normal(D)).astype(np.float32)
    wk = (1 + 0.2 * rng.standard_normal(D)).astype(np.float32)
    qo, ko = oracle.qk_rmsnorm_rope_neox(q, k, wq, wk, BRUTE_POS, H, D, base, eps)
    for bits, w, got in ((q, wq, qo), (k, wk, ko)):
        n = np.stack([_brute_head_norm(bits[t], H, D, w, eps) for t in range(4)])     # [4, H, D]
        expect = np.stack([(_rotation_matrix(BRUTE_POS[t], D, base) @ n[t].T).T for t in range(4)])
        err = np.abs(got - expect.astype(np.float64))
        tol = _rope_tol(BRUTE_POS, n.astype(np.float64))
        assert np.all(err <= tol), f"D={D}: worst {err.max()!r} at {np.unravel_index(np.argmax(err - tol), err.shape)}"
    # the separate halves of the oracle agree with the same matrices
    rot = oracle.rope_neox(oracle.head_rmsnorm(q, H, D, wq, eps), BRUTE_POS, base)
    assert np.array_equal(rot, qo)


def test_brute_force_4_tokens_adaln():
    rng = np.random.default_rng(44)
    for hidden, n_mod in ((8, 1), (64, 3), (520, 4)):
        x = bf16(rng.standard_normal((4, hidden)) * np.array([[0.01], [1.0], [7.0], [50.0]]))
        w = (1 + 0.1 * rng.standard_normal(hidden)).astype(np.float32)
        shift = (0.2 * rng.standard_normal((n_mod, hidden))).astype(np.float32)
        scale = (0.2 * rng.standard_normal((n_mod, hidden))).astype(np.float32)
        idx = (np.arange(4) % n_mod).astype(np.int32)[::-1].copy()
        got = oracle.rmsnorm_adaln_indexed(x, w, shift, scale, idx, 1e-6)
        expect = _brute_adaln(x, w, shift, scale, idx, 1e-6).astype(np.float64)
        assert np.abs(got - expect).max() <= 1e-12, (hidden, np.abs(got - expect).max())


def test_brute_force_4_tokens_swiglu():
    rng = np.random.default_rng(45)
    ffn = 40
    gu = bf16(rng.standard_normal((4, 2 * ffn)) * 4.0)
    got = oracle.swiglu(gu)
    for t in range(4):
        row = _row_ld(gu[t])
        for j in range(ffn):
            g, u = row[j], row[ffn + j]
            expect = g / (LD(1) + np.exp(-g)) * u
            assert abs(got[t, j] - float(expect)) <= 1e-12, (t, j)


def test_brute_force_4_tokens_gather_merge_and_fixed_valid():
    rng = np.random.default_rng(46)
    hidden = 24
    padded = rng.integers(0, 65536, (4, hidden), dtype=np.uint32).astype(np.uint16)
    x = bf16(rng.standard_normal((4, hidden)))
    w = np.ones(hidden, np.float32)
    zeros = np.zeros((1, hidden), np.float32)
    for L in range(5):
        rows = [[int(b) for b in padded[i]] for i in range(4)]
        compact = [rows[i][:] for i in range(L)]
        merged = [compact[i][:] if i < L else [0] * hidden for i in range(4)]
        assert oracle.valid_gather(padded, L).tolist() == compact
        assert oracle.zero_tail_merge(oracle.valid_gather(padded, L), 4).tolist() == merged
        fv = oracle.rmsnorm_adaln_fixed_valid(x, L, w, zeros, zeros, np.zeros(L, np.int32), 1e-6)
        for i in range(4):
            if i < L:
                assert np.abs(fv[i] - _brute_adaln(x[i:i + 1], w, zeros, zeros, [0], 1e-6)[0].astype(np.float64)).max() <= 1e-12
            else:
                assert np.all(fv[i] == 0.0) and not np.any(np.signbit(fv[i]))


def test_brute_force_4_tokens_ulysses_pack():
    rng = np.random.default_rng(47)
    H, D = 6, 8
    x = rng.integers(0, 65536, (4, H * D), dtype=np.uint32).astype(np.uint16)
    for P in (1, 2, 3, 6):
        got = oracle.ulysses_pack(x, H, D, P)
        hp = H // P
        for p in range(P):
            for t in range(4):
                for j in range(hp):
                    for d in range(D):
                        assert got[p, t, j, d] == x[t, (p * hp + j) * D + d]
