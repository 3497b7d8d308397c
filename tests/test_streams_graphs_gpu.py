"""The entry points as a caller uses them beyond the default stream: on side
streams, from several host threads at once, and captured into a CUDA graph and
replayed; results must equal the ones of a plain launch bit for bit."""
import threading

import numpy as np
import pytest
import torch

import rope_tfk_rmsnorm_gb300 as tfk
import synth
from helpers import f32_dev, i32_dev, to_dev, to_host

pytestmark = pytest.mark.gpu


def _problem(rows=3000, name="sg"):
    wl = synth.custom(name, rows, 3072, 24, 128, 8192, n_mod=4, n_audio=rows // 8)
    p = {k: f32_dev(v) for k, v in synth.params(wl).items()}
    d = {t: to_dev(synth.activation(wl, t)) for t in ("x", "q", "k", "gate_up")}
    d["idx"] = i32_dev(synth.mod_index(wl) % 4)
    d["pos"] = i32_dev(synth.positions(wl))
    return wl, p, d


def _chain(wl, p, d, stream=None):
    y = tfk.tfk_rmsnorm_adaln_indexed(d["x"], p["w"], p["shift"], p["scale"], d["idx"], wl.eps, stream=stream)
    qo, ko = tfk.tfk_qk_rmsnorm_rope_neox(d["q"], d["k"], p["w_q"], p["w_k"], d["pos"], wl.n_heads, wl.head_dim,
                                         wl.theta, wl.eps, stream=stream)
    o = tfk.tfk_swiglu(d["gate_up"], stream=stream)
    return y, qo, ko, o


def _bits(ts):
    return [to_host(t) for t in ts]


def test_side_streams_give_the_same_bits(cuda):
    wl, p, d = _problem()
    ref = _bits(_chain(wl, p, d))
    torch.cuda.synchronize()
    for _ in range(2):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs = _chain(wl, p, d, stream=s)
        s.synchronize()
        for a, b in zip(_bits(outs), ref):
            assert np.array_equal(a, b)


def test_concurrent_host_threads(cuda):
    wl, p, d = _problem(name="threads")
    ref = _bits(_chain(wl, p, d))
    torch.cuda.synchronize()
    results, errors = {}, []

    def worker(i):
        try:
            torch.cuda.set_device(cuda)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(3):
                    outs = _chain(wl, p, d, stream=s)
            s.synchronize()
            results[i] = _bits(outs)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(4):
        for a, b in zip(results[i], ref):
            assert np.array_equal(a, b)


def test_graph_capture_and_replay(cuda):
    wl, p, d = _problem(name="graph")
    ref = _bits(_chain(wl, p, d))
    out = {
        "y": torch.empty_like(d["x"]),
        "q": torch.empty_like(d["q"]), "k": torch.empty_like(d["k"]),
        "o": torch.empty((wl.rows, wl.ffn), dtype=torch.bfloat16, device=cuda),
    }

    def launch():
        tfk.tfk_rmsnorm_adaln_indexed(d["x"], p["w"], p["shift"], p["scale"], d["idx"], wl.eps, out=out["y"])
        tfk.tfk_qk_rmsnorm_rope_neox(d["q"], d["k"], p["w_q"], p["w_k"], d["pos"], wl.n_heads, wl.head_dim,
                                     wl.theta, wl.eps, q_out=out["q"], k_out=out["k"])
        tfk.tfk_swiglu(d["gate_up"], out=out["o"])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launch()                                   # warm the library's per-device caches
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in out.values():
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    for _ in range(2):
        for t in out.values():
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(_bits([out["y"], out["q"], out["k"], out["o"]]), ref):
            assert np.array_equal(a, b)


def test_a_failed_call_leaves_the_next_launch_unaffected(cuda):
    """After an injected launch failure, and after a call rejected on the host,
    the next call launches normally and computes the same bits."""
    wl, p, d = _problem(rows=512, name="after_error")
    ref = _bits(_chain(wl, p, d))
    lib = tfk.load()
    assert lib.tfk_debug_fail_next_launch(700) == 0
    with pytest.raises(tfk.TfkError) as e:
        tfk.tfk_swiglu(d["gate_up"])
    assert e.value.status == 4 and "[injected]" in str(e.value)
    with pytest.raises(tfk.TfkError):
        tfk.tfk_swiglu(d["gate_up"], ffn=12)          # rejected on the host
    for a, b in zip(_bits(_chain(wl, p, d)), ref):
        assert np.array_equal(a, b)


def _dependent_steps(wl, p, d, buf, iters, sync_each=False):
    """Each call reads what the call before it wrote (and the last one writes the
    next iteration's input), so every launch has a read-after-write and a
    write-after-read hazard on its predecessor: x -> RMSNorm+AdaLN -> y -> Q/K
    norm+RoPE (q = k = y) -> z -> Ulysses pack and unpack of z's q half ->
    SwiGLU(z) -> o -> RMSNorm+AdaLN in place on o -> gather of the valid rows ->
    zero-tail merge back into x."""
    x, y, z, o, c, s = buf["x"], buf["y"], buf["z"], buf["o"], buf["c"], buf["s"]
    hd, H, D = wl.hidden, wl.n_heads, wl.head_dim

    def done():
        if sync_each:
            torch.cuda.synchronize()

    for _ in range(iters):
        tfk.tfk_rmsnorm_adaln_indexed(x, p["w"], p["shift"], p["scale"], d["idx"], wl.eps, out=y); done()
        tfk.tfk_qk_rmsnorm_rope_neox(y, y, p["w_q"], p["w_k"], d["pos"], H, D, wl.theta, wl.eps,
                                     q_out=z[:, :hd], k_out=z[:, hd:]); done()
        tfk.tfk_ulysses_pack(z[:, :hd], H, D, 4, dst=s); done()
        tfk.tfk_ulysses_unpack(s, H, D, 4, dst=z[:, :hd]); done()
        tfk.tfk_swiglu(z, out=o); done()
        tfk.tfk_rmsnorm_adaln_indexed(o, p["w"], p["shift"], p["scale"], d["idx"], wl.eps, out=o); done()
        tfk.tfk_valid_gather(o, c.shape[0], compact=c); done()
        tfk.tfk_zero_tail_merge(c, x); done()


def test_back_to_back_dependent_launches_keep_stream_order(cuda):
    """The kernels may be scheduled while their predecessor on the stream drains
    (programmatic dependent launch) and must still see all of its writes and
    finish their reads before their successor writes: a chain of dependent
    calls launched back to back, eagerly and from a CUDA graph, equals the same
    chain with a device synchronisation after every call, bit for bit."""
    wl, p, d = _problem(rows=4000, name="dep")
    T, hd = wl.rows, wl.hidden

    def buffers():
        return {"x": d["x"].clone(), "y": torch.empty_like(d["x"]),
                "z": torch.empty((T, 2 * hd), dtype=torch.bfloat16, device=cuda),
                "o": torch.empty_like(d["x"]), "c": torch.empty((T - 123, hd), dtype=torch.bfloat16, device=cuda),
                "s": torch.empty(T * hd, dtype=torch.bfloat16, device=cuda)}

    iters = 12
    ref = buffers()
    _dependent_steps(wl, p, d, ref, iters, sync_each=True)
    want = to_host(ref["x"])
    assert np.isfinite(synth_f32(want)).all()
    assert np.any(want != to_host(d["x"]))

    eager = buffers()
    _dependent_steps(wl, p, d, eager, iters)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(eager["x"]), want)

    graphed = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _dependent_steps(wl, p, d, buffers(), 1)   # warm the library's caches outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _dependent_steps(wl, p, d, graphed, iters)
    for _ in range(2):
        graphed["x"].copy_(d["x"])
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_host(graphed["x"]), want)


def synth_f32(bits: np.ndarray) -> np.ndarray:
    """Raw bf16 bits -> float32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_graph_capture_of_the_fixed_valid_ulysses_and_handed_out_calls(cuda):
    """The entry points the chain tests do not capture: both fixed-valid kernels, Q/K
    written into the Ulysses send layout, and RMSNorm+AdaLN with rows handed out through
    a caller's workspace (18,000 x 3072: above the size from which rows are handed out),
    captured into a CUDA graph and replayed twice; each replay gives the eager bits and
    leaves the workspace zero."""
    wl, p, d = _problem(rows=18000, name="graph2")
    T, hd, H, D = wl.rows, wl.hidden, wl.n_heads, wl.head_dim
    L = T - 1234
    ws = torch.zeros(tfk.RMSNORM_WORKSPACE_BYTES // 8, dtype=torch.int64, device=cuda)

    def launch(out):
        tfk.tfk_rmsnorm_adaln_indexed(d["x"], p["w"], p["shift"], p["scale"], d["idx"], wl.eps, out=out["y"],
                                      workspace=ws)
        tfk.tfk_rmsnorm_adaln_indexed_fixed_valid(d["x"], L, p["w"], p["shift"], p["scale"], d["idx"][:L], wl.eps,
                                                  out=out["fy"], workspace=ws)
        tfk.tfk_qk_rmsnorm_rope_neox_fixed_valid(d["q"], d["k"], L, p["w_q"], p["w_k"], d["pos"][:L], H, D,
                                                 wl.theta, wl.eps, q_out=out["fq"], k_out=out["fk"])
        tfk.tfk_qk_rmsnorm_rope_neox_ulysses(d["q"], d["k"], p["w_q"], p["w_k"], d["pos"], H, D, 4, wl.theta,
                                             wl.eps, q_send=out["sq"], k_send=out["sk"])

    def outputs():
        send = (4, T, H // 4, D)
        return {"y": torch.empty_like(d["x"]), "fy": torch.empty_like(d["x"]),
                "fq": torch.empty_like(d["q"]), "fk": torch.empty_like(d["k"]),
                "sq": torch.empty(send, dtype=torch.bfloat16, device=cuda),
                "sk": torch.empty(send, dtype=torch.bfloat16, device=cuda)}

    ref = outputs()
    launch(ref)
    torch.cuda.synchronize()
    want = {k: to_host(v) for k, v in ref.items()}
    assert int(ws.abs().sum()) == 0

    got = outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        launch(outputs())                          # warm the library's per-device caches outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch(got)
    for _ in range(2):
        for t in got.values():
            t.fill_(-1.0)
        g.replay()
        torch.cuda.synchronize()
        for k, v in got.items():
            assert np.array_equal(to_host(v), want[k]), k
        assert int(ws.abs().sum()) == 0, "a replay left the workspace non-zero"
