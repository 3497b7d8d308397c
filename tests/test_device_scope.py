"""Which device a launch runs on, without a GPU: the entry points run each
launch with the device that owns the caller's stream current and make the
caller's device current again afterwards (csrc/device_scope.h).  The host
logic is compiled here against a fake runtime that records every device
switch and can fail any call."""
import os
import subprocess
import tempfile

from rope_tfk_rmsnorm_gb300 import build as tfk_build

CPP = r"""
#include <cstdio>
#include <vector>
#include "device_scope.h"

struct Fake {
    int current = 0;
    int stream_dev[4] = {0, 1, 3, 0};   // device of fake stream handles 0..3
    int fail_stream = 0, fail_current = 0, fail_set_to = -1, fail_restore = 0;
    std::vector<int> sets;
    int stream_device(int s, int* d) { if (fail_stream) return 700; *d = stream_dev[s]; return 0; }
    int current_device(int* d) { if (fail_current) return 701; *d = current; return 0; }
    int set_device(int d) {
        if (d == fail_set_to) return 702;
        if (fail_restore && !sets.empty()) return 703;
        sets.push_back(d); current = d; return 0;
    }
};

static int fails = 0;
#define CHECK(c) do { if (!(c)) { std::printf("FAILED line %d: %s\n", __LINE__, #c); ++fails; } } while (0)

int main() {
    {   // stream of the current device: no switch at all
        Fake rt; int ran_on = -1;
        CHECK(tfk::on_stream_device(rt, 0, [&] { ran_on = rt.current; return 0; }) == 0);
        CHECK(ran_on == 0 && rt.sets.empty() && rt.current == 0);
    }
    {   // stream of device 3 while device 0 is current: launch on 3, then back to 0
        Fake rt; int ran_on = -1;
        CHECK(tfk::on_stream_device(rt, 2, [&] { ran_on = rt.current; return 0; }) == 0);
        CHECK(ran_on == 3 && rt.sets.size() == 2 && rt.sets[0] == 3 && rt.sets[1] == 0 && rt.current == 0);
    }
    {   // a failing launch still restores the caller's device, and its error is returned
        Fake rt; rt.current = 1;
        CHECK(tfk::on_stream_device(rt, 2, [&] { return 98; }) == 98);
        CHECK(rt.current == 1);
    }
    {   // the stream's device cannot be read: nothing runs
        Fake rt; rt.fail_stream = 1; bool ran = false;
        CHECK(tfk::on_stream_device(rt, 1, [&] { ran = true; return 0; }) == 700);
        CHECK(!ran && rt.sets.empty());
    }
    {   // the current device cannot be read: nothing runs
        Fake rt; rt.fail_current = 1; bool ran = false;
        CHECK(tfk::on_stream_device(rt, 1, [&] { ran = true; return 0; }) == 701);
        CHECK(!ran);
    }
    {   // the stream's device cannot be made current: nothing runs, nothing changes
        Fake rt; rt.fail_set_to = 1; bool ran = false;
        CHECK(tfk::on_stream_device(rt, 1, [&] { ran = true; return 0; }) == 702);
        CHECK(!ran && rt.current == 0);
    }
    {   // the launch worked but restoring failed: that error is reported
        Fake rt; rt.fail_restore = 1; bool ran = false;
        CHECK(tfk::on_stream_device(rt, 1, [&] { ran = true; return 0; }) == 703);
        CHECK(ran);
    }
    std::printf("%s\n", fails ? "FAILED" : "OK");
    return fails != 0;
}
"""


def test_launch_runs_on_the_streams_device_and_restores_the_callers():
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "scope.cpp"), os.path.join(d, "scope")
        open(src, "w").write(CPP)
        csrc = os.path.join(tfk_build.HERE, "csrc")
        r = subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", f"-I{csrc}", src, "-o", exe],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
