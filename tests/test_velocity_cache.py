"""Conservative DiT velocity-cache schedule: the oracle against the page's own
counts, the library's host implementation against the oracle (no GPU), and
the schedule driving the chained GPU path over a 49-step run: a hit launches
nothing and hands back the previous step's velocity."""
import itertools
import os

import pytest

import rope_tfk_rmsnorm_gb300 as tfk
from oracle import velocity_cache
from rope_tfk_rmsnorm_gb300 import build as tfk_build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "velocity_cache_p1.txt")


def golden():
    kv = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            kv[k] = float(v) if "." in v else int(v)
    return kv


@pytest.fixture(scope="module")
def lib():
    tfk_build.build()
    return tfk.load()


def test_oracle_reproduces_the_pages_counts():
    g = golden()
    s = velocity_cache.schedule(g["steps"], g["start_ratio"], g["end_ratio"], g["refresh_interval"],
                                g["max_consecutive_reuse"])
    assert sum(s) == g["cache_hits"]
    assert len(s) - sum(s) == g["cached_dit_calls"]
    # the cache off (an empty window) is the baseline: every step calls the DiT
    assert sum(velocity_cache.schedule(g["steps"], 0.0, 0.0)) == 0
    assert g["baseline_dit_calls"] == g["steps"]


def test_oracle_schedule_properties():
    s = velocity_cache.schedule(49)
    hits = [i for i, r in enumerate(s) if r]
    assert all(0.2 <= i / 49 < 0.8 for i in hits)               # only inside the window
    assert all(not (a and b) for a, b in zip(s, s[1:]))          # never two reuses in a row
    assert not s[0]                                              # nothing to reuse on step 0
    # a longer reuse budget is still capped by the refresh interval, and vice versa
    assert velocity_cache.schedule(49, refresh_interval=2, max_consecutive_reuse=3) == s
    assert velocity_cache.schedule(49, refresh_interval=5, max_consecutive_reuse=1) == s
    s3 = velocity_cache.schedule(49, refresh_interval=4, max_consecutive_reuse=3)
    assert sum(s3) > sum(s)


def _library_matches_oracle():
    g = golden()
    assert sum(tfk.tfk_velocity_cache_schedule(49)) == g["cache_hits"]
    for n, (a, b), ri, mr in itertools.product([0, 1, 2, 5, 10, 48, 49, 50, 100, 257],
                                               [(0.2, 0.8), (0.0, 1.0), (0.25, 0.75), (0.5, 0.5), (0.1, 0.3)],
                                               [1, 2, 3, 5], [0, 1, 2, 4]):
        assert tfk.tfk_velocity_cache_schedule(n, a, b, ri, mr) == velocity_cache.schedule(n, a, b, ri, mr), \
            (n, a, b, ri, mr)


def test_library_schedule_matches_the_oracle(lib):
    _library_matches_oracle()


@pytest.mark.gpu
def test_library_schedule_matches_the_oracle_on_the_gpu_host(lib):
    """The same check in the GPU run, where the library is built on the GPU host itself."""
    _library_matches_oracle()


def test_library_schedule_rejects_bad_arguments(lib):
    for args, words in [((-1, 0.2, 0.8, 2, 1), "num_steps = -1"), ((10, 0.8, 0.2, 2, 1), "<= end_ratio"),
                        ((10, -0.1, 0.8, 2, 1), "0 <= start_ratio"), ((10, 0.2, 1.5, 2, 1), "<= 1"),
                        ((10, 0.2, 0.8, 0, 1), "refresh_interval = 0"),
                        ((10, 0.2, 0.8, 2, -1), "max_consecutive_reuse = -1"),
                        ((10, float("nan"), 0.8, 2, 1), "finite")]:
        with pytest.raises(tfk.TfkError) as e:
            tfk.tfk_velocity_cache_schedule(*args)
        assert e.value.status == 1 and "tfk_velocity_cache_schedule" in str(e.value) and words in str(e.value), \
            (args, str(e.value))


@pytest.mark.gpu
def test_schedule_gates_the_chain_on_the_gpu(lib, cuda):
    """49 denoising steps of the 320-token chain (RMSNorm+AdaLN, Q/K RMSNorm+RoPE, SwiGLU
    standing in for the DiT call), gated by the library's schedule with the page's defaults
    (TeleFuser PR #38, section 3 and the section 1 table: 34 DiT calls, 15 hits).  A DiT step
    runs the chain on that step's inputs and its outputs become the cached velocity; a hit
    launches nothing and returns the cached buffers.  Checked: 34 chain runs and 3 * 34
    calls into the library's launching entry points (counted at the C ABI by a proxy around
    the loaded library), every hit bit-identical to the step before it, every computed step
    within tolerance of the oracle."""
    import dataclasses

    import numpy as np
    import torch

    import oracle
    import synth
    from helpers import THREADS, check_close, f32_dev, i32_dev, to_dev, to_host

    g = golden()
    sched = tfk.tfk_velocity_cache_schedule(g["steps"])
    base = synth.get("tiny")
    p = synth.params(base)
    pd = {k: f32_dev(v) for k, v in p.items()}
    idx, pos = synth.mod_index(base), synth.positions(base)
    idx_d, pos_d = i32_dev(idx), i32_dev(pos)
    inputs = []
    for i in range(g["steps"]):  # the step's DiT inputs: a fresh draw per step
        wl = dataclasses.replace(base, seed=1000 + i)
        inputs.append({t: synth.activation(wl, t) for t in ("x", "q", "k", "gate_up")})
    dev_inputs = [{t: to_dev(a) for t, a in step.items()} for step in inputs]
    torch.cuda.synchronize()

    class CountingLib:
        """The loaded library with a count of calls to every entry point that launches."""

        def __init__(self, lib):
            self.lib, self.launches = lib, {}

        def __getattr__(self, name):
            fn = getattr(self.lib, name)
            if name in ("tfk_status_string", "tfk_last_error_message", "tfk_abi_version",
                        "tfk_velocity_cache_schedule", "tfk_debug_fail_next_launch"):
                return fn

            def counted(*args):
                self.launches[name] = self.launches.get(name, 0) + 1
                return fn(*args)
            return counted

    counting = CountingLib(tfk.load())
    velocity, calls, handed = None, [], []
    tfk._lib = counting
    try:
        for i, hit in enumerate(sched):
            if hit:
                assert velocity is not None, "a hit before any DiT call"
                out = velocity
            else:
                d = dev_inputs[i]
                y = tfk.tfk_rmsnorm_adaln_indexed(d["x"], pd["w"], pd["shift"], pd["scale"], idx_d, base.eps)
                qo, ko = tfk.tfk_qk_rmsnorm_rope_neox(d["q"], d["k"], pd["w_q"], pd["w_k"], pos_d, base.n_heads,
                                                      base.head_dim, base.theta, base.eps)
                o = tfk.tfk_swiglu(d["gate_up"])
                out = velocity = (y, qo, ko, o)
                calls.append(i)
            handed.append(out)
        torch.cuda.synchronize()
    finally:
        tfk._lib = counting.lib

    assert len(calls) == g["cached_dit_calls"] and g["steps"] - len(calls) == g["cache_hits"]
    assert counting.launches == {"tfk_rmsnorm_adaln_indexed": g["cached_dit_calls"],
                                 "tfk_qk_rmsnorm_rope_neox": g["cached_dit_calls"],
                                 "tfk_swiglu": g["cached_dit_calls"]}, counting.launches

    bits = [tuple(to_host(t) for t in out) for out in handed]
    for i, hit in enumerate(sched):
        if hit:
            assert handed[i] is handed[i - 1] or all(a is b for a, b in zip(handed[i], handed[i - 1]))
            assert all(np.array_equal(a, b) for a, b in zip(bits[i], bits[i - 1])), f"step {i}"
    for i in calls:
        x, q, k, gu = (inputs[i][t] for t in ("x", "q", "k", "gate_up"))
        y, qo, ko, o = bits[i]
        check_close(y, oracle.rmsnorm_adaln_indexed(x, p["w"], p["shift"], p["scale"], idx, base.eps,
                                                    threads=THREADS), f"step {i} a1")
        rq, rk = oracle.qk_rmsnorm_rope_neox(q, k, p["w_q"], p["w_k"], pos, base.n_heads, base.head_dim,
                                             base.theta, base.eps, threads=THREADS)
        check_close(qo, rq.reshape(base.rows, -1), f"step {i} a2 q")
        check_close(ko, rk.reshape(base.rows, -1), f"step {i} a2 k")
        check_close(o, oracle.swiglu(gu, threads=THREADS), f"step {i} a3")
    # consecutive DiT calls see different inputs, so a reused velocity is never a recomputation
    assert not np.array_equal(bits[calls[0]][0], bits[calls[1]][0])
