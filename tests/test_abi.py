"""The C ABI without a GPU: libtfk.so loads, exports every symbol include/tfk.h
declares, and rejects bad arguments on the host before anything is launched.

No call here reaches the CUDA driver: every call either fails validation or
is replaced by an injected launch failure (tfk_debug_fail_next_launch), which
the library checks after validation and before any CUDA call.
"""
import ctypes
import os
import re

import pytest

import rope_tfk_rmsnorm_gb300 as tfk
from rope_tfk_rmsnorm_gb300 import build as tfk_build

HEADER = os.path.join(tfk_build.INCLUDE, "tfk.h")
OK, INVALID, MISALIGNED, UNSUPPORTED, CUDA = 0, 1, 2, 3, 4
INJECTED = 999  # an arbitrary CUDA error code reported by the injection hook

A = 0x10000000  # fake, 16-byte aligned "device" addresses: never dereferenced
B = 0x20000000
C = 0x30000000
W = 0x40000000
S = 0x50000000
P = 0x60000000


@pytest.fixture(scope="module")
def lib():
    tfk_build.build()
    lib = tfk.load()
    lib.tfk_debug_fail_next_launch(0)
    yield lib
    lib.tfk_debug_fail_next_launch(0)


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(tfk_\w+)\s*\(", text, re.M)))


def msg(lib):
    return lib.tfk_last_error_message().decode()


def passes_validation(lib, call):
    """True if `call` gets past validation: it then returns the injected CUDA error."""
    lib.tfk_debug_fail_next_launch(INJECTED)
    st = call()
    lib.tfk_debug_fail_next_launch(0)
    if st == CUDA:
        assert "[injected]" in msg(lib)
        return True
    return False


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) == 16, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in tfk.h but not exported"
    assert sorted(n for n, _, _ in tfk.SIGNATURES) == names


def test_abi_version_and_status_strings(lib):
    ver = int(re.search(r"#define TFK_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert lib.tfk_abi_version() == ver
    for code, name in tfk.STATUS.items():
        assert lib.tfk_status_string(code).decode() == name
    assert lib.tfk_status_string(77).decode() == "TFK_ERR_UNKNOWN"


WS = 0x70000000


def adaln(lib, x=A, xs=512, y=B, ys=512, w=W, sh=S, sc=S + 0x100000, idx=P, n_mod=2, rows=10,
          hidden=512, eps=1e-6, ws=WS):
    return lib.tfk_rmsnorm_adaln_indexed(x, xs, y, ys, w, sh, sc, idx, n_mod, rows, hidden, eps, ws, None)


def test_adaln_validation(lib):
    assert passes_validation(lib, lambda: adaln(lib))
    assert passes_validation(lib, lambda: adaln(lib, y=A))                  # in place
    assert adaln(lib, rows=0, x=0, y=0, w=0, sh=0, sc=0, idx=0) == OK       # empty: no-op
    assert adaln(lib, rows=-1) == INVALID
    assert adaln(lib, x=0) == INVALID and "null" in msg(lib)
    assert adaln(lib, hidden=0) == INVALID
    assert adaln(lib, hidden=12, xs=16, ys=16) == UNSUPPORTED
    assert adaln(lib, hidden=32776, xs=32776, ys=32776) == UNSUPPORTED
    assert adaln(lib, n_mod=0) == INVALID
    assert adaln(lib, eps=-1.0) == INVALID
    assert adaln(lib, eps=float("nan")) == INVALID
    assert adaln(lib, xs=504) == INVALID                                    # stride < hidden
    assert adaln(lib, xs=516) == MISALIGNED
    assert adaln(lib, x=A + 8) == MISALIGNED
    assert adaln(lib, w=W + 4) == MISALIGNED
    assert adaln(lib, idx=P + 2) == MISALIGNED
    assert adaln(lib, y=A + 16) == INVALID and "overlaps x" in msg(lib)     # partial overlap
    assert adaln(lib, y=A, ys=1024, xs=512) == INVALID                      # same base, other stride
    assert adaln(lib, y=W) == INVALID and "parameter" in msg(lib)
    assert passes_validation(lib, lambda: adaln(lib, ws=0))                  # no workspace: rows split up front
    assert adaln(lib, ws=WS + 4) == MISALIGNED and "workspace" in msg(lib)
    assert adaln(lib, ws=B + 64) == INVALID and "workspace overlaps" in msg(lib)   # inside y
    assert adaln(lib, ws=A + 8) == INVALID and "workspace overlaps" in msg(lib)    # inside x
    assert adaln(lib, ws=P) == INVALID and "workspace overlaps" in msg(lib)        # on mod_idx


def adaln_noalloc(lib, x=A, xs=512, y=B, ys=512, w=W, sh=S, sc=S + 0x100000, idx=P, n_mod=2, rows=10,
                  hidden=512, eps=1e-6):
    return lib.tfk_rmsnorm_adaln_indexed_noalloc(x, xs, y, ys, w, sh, sc, idx, n_mod, rows, hidden, eps, None)


def test_adaln_noalloc_validation(lib):
    """The allocation-free entry point checks its arguments as tfk_rmsnorm_adaln_indexed
    does, under its own name, before it touches its scratch array or the GPU."""
    assert passes_validation(lib, lambda: adaln_noalloc(lib))
    assert passes_validation(lib, lambda: adaln_noalloc(lib, y=A))          # in place
    assert adaln_noalloc(lib, rows=0, x=0, y=0, w=0, sh=0, sc=0, idx=0) == OK
    assert adaln_noalloc(lib, x=0) == INVALID and "tfk_rmsnorm_adaln_indexed_noalloc" in msg(lib)
    assert adaln_noalloc(lib, n_mod=0) == INVALID
    assert adaln_noalloc(lib, hidden=32776, xs=32776, ys=32776) == UNSUPPORTED
    assert adaln_noalloc(lib, xs=516) == MISALIGNED
    assert adaln_noalloc(lib, y=A + 16) == INVALID and "overlaps x" in msg(lib)
    assert adaln_noalloc(lib, eps=float("nan")) == INVALID


def qk(lib, q=A, k=A + 2 * 1024, ist=3 * 1024, qo=B, ko=B + 2 * 1024, ost=3 * 1024, wq=W, wk=W + 64,
       pos=P, rows=10, H=8, D=128, theta=10000.0, eps=1e-6):
    return lib.tfk_qk_rmsnorm_rope_neox(q, k, ist, qo, ko, ost, wq, wk, pos, rows, H, D, theta, eps, None)


def test_qk_validation(lib):
    # q and k as column slices of one fused QKV buffer [rows, 3*H*D]
    assert passes_validation(lib, lambda: qk(lib))
    assert passes_validation(lib, lambda: qk(lib, qo=A, ko=A + 2 * 1024))   # in place in the QKV buffer
    assert qk(lib, rows=0, q=0, k=0, qo=0, ko=0, wq=0, wk=0, pos=0) == OK
    assert qk(lib, D=120) == UNSUPPORTED
    assert qk(lib, D=8) == UNSUPPORTED
    assert qk(lib, D=1024, ist=3 * 8192, ost=3 * 8192, k=A + 2 * 8192, ko=B + 2 * 8192) == UNSUPPORTED
    assert passes_validation(lib, lambda: qk(lib, H=200, ist=3 * 200 * 128, ost=3 * 200 * 128,
                                             k=A + 2 * 200 * 128, ko=B + 2 * 200 * 128))  # many heads: 2-D grid
    assert qk(lib, H=0) == INVALID
    assert qk(lib, theta=0.0) == INVALID
    assert qk(lib, theta=float("inf")) == INVALID
    assert qk(lib, eps=-1e-6) == INVALID
    assert qk(lib, ist=512) == INVALID                                      # stride < H*D
    assert qk(lib, ost=3 * 1024 + 4) == MISALIGNED
    assert qk(lib, pos=P + 1) == MISALIGNED
    assert qk(lib, wk=W + 8) == MISALIGNED
    assert qk(lib, ko=B + 1024) == INVALID and "q_out and k_out overlap" in msg(lib)
    assert qk(lib, qo=A + 16) == INVALID and "q_out overlaps q" in msg(lib)
    assert qk(lib, qo=A + 2 * 1024, ko=B) == INVALID                        # q_out onto k's input columns
    assert qk(lib, qo=P) == INVALID and "positions" in msg(lib)


def swiglu(lib, gu=A, ist=2048, out=B, ost=1024, rows=4, ffn=1024):
    return lib.tfk_swiglu(gu, ist, out, ost, rows, ffn, None)


def test_swiglu_validation(lib):
    assert passes_validation(lib, lambda: swiglu(lib))
    assert passes_validation(lib, lambda: swiglu(lib, gu=A, ist=3072, out=A + 2 * 2048, ost=3072))  # disjoint columns
    assert swiglu(lib, rows=0, gu=0, out=0) == OK
    assert swiglu(lib, ffn=12, ist=24, ost=16) == UNSUPPORTED
    assert swiglu(lib, ffn=0) == INVALID
    assert swiglu(lib, ist=2040) == INVALID
    assert swiglu(lib, out=B + 2) == MISALIGNED
    assert swiglu(lib, out=A + 2048) == INVALID and "overlaps" in msg(lib)
    assert swiglu(lib, gu=A, ist=3072, out=A + 2 * 1024, ost=3072) == INVALID  # out onto the up half


def test_gather_merge_validation(lib):
    g = lambda p=A, c=B, L=100, h=64: lib.tfk_valid_gather(p, c, L, h, None)
    m = lambda c=B, p=A, L=100, N=128, h=64: lib.tfk_zero_tail_merge(c, p, L, N, h, None)
    assert passes_validation(lib, g) and passes_validation(lib, m)
    assert passes_validation(lib, lambda: m(L=0, c=0))                      # all-zero fill
    assert g(L=0, p=0, c=0) == OK and m(N=0, L=0, p=0, c=0) == OK
    assert g(L=-1) == INVALID and m(L=200) == INVALID and m(L=-1) == INVALID
    assert g(h=12) == UNSUPPORTED and m(h=0) == INVALID
    assert g(c=B + 8) == MISALIGNED and m(p=A + 4) == MISALIGNED
    assert g(c=A + 128) == INVALID and m(c=A + 64 * 2 * 127) == INVALID
    assert g(c=0) == INVALID


def test_injection_hook_contract(lib):
    assert lib.tfk_debug_fail_next_launch(-5) == INVALID
    assert lib.tfk_debug_fail_next_launch(2) == OK
    # a validation failure does not consume the injection ...
    assert swiglu(lib, ffn=0) == INVALID
    # ... the next valid call does, exactly once
    assert swiglu(lib) == CUDA and "CUDA error 2" in msg(lib) and "[injected]" in msg(lib)
    assert lib.tfk_debug_fail_next_launch(0) == OK


def test_python_binding_rejects_bad_tensors_before_the_abi():
    import torch
    x = torch.zeros(4, 16, dtype=torch.float32)
    with pytest.raises((TypeError, ValueError)):
        tfk.tfk_swiglu(x)
    xb = torch.zeros(4, 16, dtype=torch.bfloat16)   # CPU tensor: the library has no CPU path
    with pytest.raises(ValueError, match="CUDA"):
        tfk.tfk_swiglu(xb)


def test_fixed_valid_validation(lib):
    fa = lambda L=10, N=16, x=A, y=B, idx=P: lib.tfk_rmsnorm_adaln_indexed_fixed_valid(
        x, 512, y, 512, W, S, S + 0x100000, idx, 2, L, N, 512, 1e-6, WS, None)
    assert passes_validation(lib, fa)
    assert passes_validation(lib, lambda: fa(L=0, x=0, idx=0))              # the whole buffer becomes +0.0
    assert passes_validation(lib, lambda: fa(y=A))                          # in place
    assert fa(L=0, N=0, x=0, y=0, idx=0) == OK
    assert fa(L=17, N=16) == INVALID and fa(L=-1) == INVALID
    assert fa(y=0) == INVALID
    assert fa(y=A + 512 * 2 * 12) == INVALID                                # y's padded rows reach into x
    fq = lambda L=10, N=16, qo=B, ko=B + 2 * 1024: lib.tfk_qk_rmsnorm_rope_neox_fixed_valid(
        A, A + 2 * 1024, 3 * 1024, qo, ko, 3 * 1024, W, W + 64, P, L, N, 8, 128, 10000.0, 1e-6, None)
    assert passes_validation(lib, fq)
    assert passes_validation(lib, lambda: fq(qo=A, ko=A + 2 * 1024))
    assert fq(L=20) == INVALID and fq(ko=B + 1024) == INVALID


def test_velocity_cache_schedule_sets_the_error_message(lib):
    buf = (ctypes.c_uint8 * 16)()
    hits = ctypes.c_int32(0)
    vp = lambda o: ctypes.cast(o, ctypes.c_void_p)
    sched = lambda n=10, a=0.2, b=0.8, ri=2, mr=1, r=vp(buf): lib.tfk_velocity_cache_schedule(
        n, a, b, ri, mr, r, vp(ctypes.pointer(hits)))
    assert sched() == OK
    for kwargs, words in [(dict(n=-3), "num_steps = -3"), (dict(ri=0), "refresh_interval = 0"),
                          (dict(mr=-2), "max_consecutive_reuse = -2"), (dict(a=float("inf")), "finite"),
                          (dict(a=0.9), "start_ratio (0.9) <= end_ratio (0.8)"), (dict(b=1.5), "<= 1"),
                          (dict(a=-0.5), "0 <= start_ratio"), (dict(r=None), "reuse is NULL")]:
        lib.tfk_debug_fail_next_launch(0)
        assert sched(**kwargs) == INVALID, kwargs
        m = msg(lib)
        assert m.startswith("tfk_velocity_cache_schedule: ") and words in m, (kwargs, m)
    assert sched(n=0, r=None) == OK                                         # no steps: reuse may be NULL
