"""The boundary from plain C on the GPU: a C program (gcc, the CUDA runtime's C
API, no Python or torch in the process) allocates device memory, creates its
own stream, runs the five operations of the path through include/tfk.h on
inputs this test drew, and writes the outputs back to files; the test checks
them against the oracle (bit-exact for gather and merge)."""
import glob
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from helpers import check_close
from rope_tfk_rmsnorm_gb300 import build as tfk_build
from test_parity_gpu import mod_params, ora_adaln, ora_qk, ora_swiglu, rand_bits

pytestmark = pytest.mark.gpu

ROWS, HIDDEN, N_MOD, H, D, FFN, PADDED, VALID = 333, 512, 3, 4, 128, 776, 400, 333

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "tfk.h"

static void* load(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s.bin", dir, name);
    FILE* f = fopen(path, "rb");
    void* p = malloc(bytes);
    if (!f || !p || fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot read %s\n", path); exit(2); }
    fclose(f);
    return p;
}

static void save(const char* dir, const char* name, const void* p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s.out", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
    fclose(f);
}

static void* to_device(const void* host, size_t bytes) {
    void* d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess || cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device copy failed\n");
        exit(3);
    }
    return d;
}

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("FAILED %s (line %d): %s\n", #c, __LINE__, tfk_last_error_message()); ++fails; } } while (0)

int main(int argc, char** argv) {
    if (argc != 2) return 2;
    const char* dir = argv[1];
    const int64_t rows = ROWS, padded = PADDED, valid = VALID;
    const int32_t hidden = HIDDEN, n_mod = N_MOD, heads = H, dim = D, ffn = FFN;
    const size_t xb = (size_t)rows * hidden * 2, qb = (size_t)rows * heads * dim * 2, ob = (size_t)rows * ffn * 2;
    const size_t pb = (size_t)padded * hidden * 2;

    void* x = to_device(load(dir, "x", xb), xb);
    void* w = to_device(load(dir, "w", hidden * 4), hidden * 4);
    void* shift = to_device(load(dir, "shift", (size_t)n_mod * hidden * 4), (size_t)n_mod * hidden * 4);
    void* scale = to_device(load(dir, "scale", (size_t)n_mod * hidden * 4), (size_t)n_mod * hidden * 4);
    void* idx = to_device(load(dir, "idx", rows * 4), rows * 4);
    void* q = to_device(load(dir, "q", qb), qb);
    void* k = to_device(load(dir, "k", qb), qb);
    void* wq = to_device(load(dir, "wq", dim * 4), dim * 4);
    void* wk = to_device(load(dir, "wk", dim * 4), dim * 4);
    void* pos = to_device(load(dir, "pos", rows * 4), rows * 4);
    void* gu = to_device(load(dir, "gate_up", 2 * ob), 2 * ob);
    void* pad = to_device(load(dir, "padded", pb), pb);
    void *y, *qo, *ko, *o, *compact, *merged, *ws;
    cudaMalloc(&y, xb); cudaMalloc(&qo, qb); cudaMalloc(&ko, qb); cudaMalloc(&o, ob);
    cudaMalloc(&compact, (size_t)valid * hidden * 2); cudaMalloc(&merged, pb);
    cudaMalloc(&ws, TFK_RMSNORM_WORKSPACE_BYTES);
    cudaMemset(ws, 0, TFK_RMSNORM_WORKSPACE_BYTES);
    cudaMemset(merged, 0xFF, pb);
    cudaStream_t s;
    CHECK(cudaStreamCreate(&s) == cudaSuccess);

    CHECK(tfk_rmsnorm_adaln_indexed(x, hidden, y, hidden, w, shift, scale, idx, n_mod, rows, hidden, 1e-6f, ws, s) == TFK_OK);
    CHECK(tfk_qk_rmsnorm_rope_neox(q, k, heads * dim, qo, ko, heads * dim, wq, wk, pos, rows, heads, dim,
                                   10000.0f, 1e-6f, s) == TFK_OK);
    CHECK(tfk_swiglu(gu, 2 * ffn, o, ffn, rows, ffn, s) == TFK_OK);
    CHECK(tfk_valid_gather(pad, compact, valid, hidden, s) == TFK_OK);
    CHECK(tfk_zero_tail_merge(compact, merged, valid, padded, hidden, s) == TFK_OK);
    CHECK(cudaStreamSynchronize(s) == cudaSuccess);

    unsigned char* host = malloc(pb > 2 * ob ? pb : 2 * ob);
    unsigned long long wsh[TFK_RMSNORM_WORKSPACE_BYTES / 8];
    CHECK(cudaMemcpy(wsh, ws, sizeof wsh, cudaMemcpyDeviceToHost) == cudaSuccess);
    for (size_t i = 0; i < sizeof wsh / 8; ++i) CHECK(wsh[i] == 0ull);
    cudaMemcpy(host, y, xb, cudaMemcpyDeviceToHost); save(dir, "y", host, xb);
    cudaMemcpy(host, qo, qb, cudaMemcpyDeviceToHost); save(dir, "qo", host, qb);
    cudaMemcpy(host, ko, qb, cudaMemcpyDeviceToHost); save(dir, "ko", host, qb);
    cudaMemcpy(host, o, ob, cudaMemcpyDeviceToHost); save(dir, "o", host, ob);
    cudaMemcpy(host, compact, (size_t)valid * hidden * 2, cudaMemcpyDeviceToHost);
    save(dir, "compact", host, (size_t)valid * hidden * 2);
    CHECK(cudaMemcpy(host, merged, pb, cudaMemcpyDeviceToHost) == cudaSuccess);
    save(dir, "merged", host, pb);
    cudaStreamDestroy(s);
    printf("%s\n", fails ? "FAILED" : "OK");
    return fails != 0;
}
"""


def _cuda_dirs():
    root = os.path.dirname(os.path.dirname(os.path.realpath(tfk_build.nvcc())))
    libs = [d for d in [os.path.join(root, "lib64"), *glob.glob(os.path.join(root, "targets", "*", "lib"))]
            if os.path.exists(os.path.join(d, "libcudart.so"))]
    return os.path.join(root, "include"), libs


def test_c_program_runs_the_path_on_the_gpu(cuda):
    lib = tfk_build.build()
    libdir = os.path.dirname(lib)
    inc, cudalibs = _cuda_dirs()
    assert cudalibs, "libcudart.so not found next to nvcc"
    rng = np.random.default_rng(5)
    x = rand_bits(rng, (ROWS, HIDDEN))
    w, sh, sc = mod_params(rng, N_MOD, HIDDEN)
    idx = rng.integers(0, N_MOD, ROWS).astype(np.int32)
    q, k = rand_bits(rng, (ROWS, H * D)), rand_bits(rng, (ROWS, H * D))
    wq, wk = (1 + 0.1 * rng.standard_normal((2, D))).astype(np.float32)
    pos = rng.integers(0, 80000, ROWS).astype(np.int32)
    gu = rand_bits(rng, (ROWS, 2 * FFN), 3.0)
    pad = rand_bits(rng, (PADDED, HIDDEN))
    pad[VALID:] = 0x7FC0  # NaN tail: never read
    with tempfile.TemporaryDirectory() as d:
        for name, a in dict(x=x, w=w, shift=sh, scale=sc, idx=idx, q=q, k=k, wq=wq, wk=wk, pos=pos,
                            gate_up=gu, padded=pad).items():
            np.ascontiguousarray(a).tofile(os.path.join(d, f"{name}.bin"))
        src, exe = os.path.join(d, "consumer.c"), os.path.join(d, "consumer")
        open(src, "w").write(C_SOURCE)
        defs = [f"-D{n}={v}" for n, v in dict(ROWS=ROWS, HIDDEN=HIDDEN, N_MOD=N_MOD, H=H, D=D, FFN=FFN,
                                              PADDED=PADDED, VALID=VALID).items()]
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", *defs, f"-I{tfk_build.INCLUDE}", f"-I{inc}", src,
                            os.path.join(libdir, "libtfk.so"), *[f"-L{p}" for p in cudalibs], "-lcudart",
                            f"-Wl,-rpath,{libdir}", *[f"-Wl,-rpath,{p}" for p in cudalibs], "-o", exe],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        r = subprocess.run([exe, d], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr

        def out(name, shape):
            return np.fromfile(os.path.join(d, f"{name}.out"), dtype=np.uint16).reshape(shape)

        check_close(out("y", (ROWS, HIDDEN)), ora_adaln(x, w, sh, sc, idx, 1e-6), "a1 from C")
        rq, rk = ora_qk(q, k, wq, wk, pos, H, D, 10000.0, 1e-6)
        check_close(out("qo", (ROWS, H * D)), rq, "a2 q from C")
        check_close(out("ko", (ROWS, H * D)), rk, "a2 k from C")
        check_close(out("o", (ROWS, FFN)), ora_swiglu(gu), "a3 from C")
        assert np.array_equal(out("compact", (VALID, HIDDEN)), oracle.valid_gather(pad, VALID))
        assert np.array_equal(out("merged", (PADDED, HIDDEN)),
                              oracle.zero_tail_merge(oracle.valid_gather(pad, VALID), PADDED))
