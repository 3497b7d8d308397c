"""The boundary from plain C: a C program includes include/tfk.h, links
libtfk.so and exercises the calls that need no GPU (version, status strings,
argument validation, injected launch failure, the velocity-cache schedule)."""
import os
import subprocess
import tempfile

import pytest

from rope_tfk_rmsnorm_gb300 import build as tfk_build

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "tfk.h"

static int fails = 0;
#define CHECK(c) do { if (!(c)) { printf("FAILED %s (line %d): %s\n", #c, __LINE__, tfk_last_error_message()); ++fails; } } while (0)

int main(void) {
    CHECK(tfk_abi_version() == TFK_ABI_VERSION);
    CHECK(strcmp(tfk_status_string(TFK_ERR_MISALIGNED), "TFK_ERR_MISALIGNED") == 0);
    /* empty problems are no-ops, even with NULL pointers */
    CHECK(tfk_swiglu(NULL, 16, NULL, 8, 0, 8, NULL) == TFK_OK);
    /* validation happens on the host, before any device work */
    CHECK(tfk_swiglu(NULL, 16, NULL, 8, 4, 8, NULL) == TFK_ERR_INVALID_ARGUMENT);
    CHECK(tfk_swiglu((const tfk_bf16*)0x1000, 16, (tfk_bf16*)0x2002, 8, 4, 8, NULL) == TFK_ERR_MISALIGNED);
    CHECK(tfk_qk_rmsnorm_rope_neox((const tfk_bf16*)0x1000, (const tfk_bf16*)0x9000, 1024, (tfk_bf16*)0x20000,
                                   (tfk_bf16*)0x40000, 1024, (const float*)0x60000, (const float*)0x60100,
                                   (const int32_t*)0x70000, 4, 8, 100, 10000.0f, 1e-6f, NULL) == TFK_ERR_UNSUPPORTED);
    /* an injected launch failure replaces the next valid call's launch */
    CHECK(tfk_debug_fail_next_launch(2) == TFK_OK);
    CHECK(tfk_valid_gather((const tfk_bf16*)0x100000, (tfk_bf16*)0x200000, 10, 64, NULL) == TFK_ERR_CUDA);
    CHECK(strstr(tfk_last_error_message(), "[injected]") != NULL);
    /* the host-side velocity-cache schedule of the page's validation run */
    uint8_t reuse[49];
    int32_t hits = -1;
    CHECK(tfk_velocity_cache_schedule(49, 0.2, 0.8, 2, 1, reuse, &hits) == TFK_OK);
    CHECK(hits == 15);
    int calls = 0;
    for (int i = 0; i < 49; ++i) calls += reuse[i] == 0;
    CHECK(calls == 34);
    printf("%s\n", fails ? "FAILED" : "OK");
    return fails != 0;
}
"""


def test_c_program_uses_the_abi():
    lib = tfk_build.build()
    libdir = os.path.dirname(lib)
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "consumer.c")
        exe = os.path.join(d, "consumer")
        open(src, "w").write(C_SOURCE)
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{tfk_build.INCLUDE}", src,
                            os.path.join(libdir, "libtfk.so"), f"-Wl,-rpath,{libdir}", "-o", exe],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
