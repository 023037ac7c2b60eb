"""Once-per-device set-up of kernel attributes (csrc/per_device.h), on the CPU.

Function attributes such as the GEMM's dynamic shared-memory limit belong to the context of
the device current when they are set, so a process that drives several GPUs must set them on
each device.  The header has no CUDA dependency; this test compiles a small C++ driver
against it with g++ and checks that the set-up runs once per device ordinal, is retried
after a failure, never caches an ordinal outside the tracked range, and runs at most a few
times when many host threads race on one device.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "transposed_convolution_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "per_device.h"

int main() {
    ctr::PerDeviceOnce once;
    int calls[3] = {0, 0, 0};
    auto setup_on = [&](int dev, int err) {
        return once.run(dev, 0, [&] { ++calls[dev < 0 ? 2 : dev]; return err; });
    };
    // Device 0: the first call runs the set-up, later calls do not.
    if (setup_on(0, 0) != 0 || setup_on(0, 0) != 0 || calls[0] != 1) return 1;
    if (!once.done(0) || once.done(1)) return 2;
    // Device 1 has a flag of its own.
    if (setup_on(1, 0) != 0 || calls[1] != 1 || !once.done(1)) return 3;
    // A failing set-up is reported and retried on the next call.
    ctr::PerDeviceOnce twice;
    int n = 0;
    if (twice.run(5, 0, [&] { ++n; return 7; }) != 7 || twice.done(5)) return 4;
    if (twice.run(5, 0, [&] { ++n; return 0; }) != 0 || !twice.done(5) || n != 2) return 5;
    // An ordinal that cannot be tracked (-1: the device could not be read) runs every time.
    setup_on(-1, 0);
    setup_on(-1, 0);
    if (calls[2] != 2 || once.done(-1)) return 6;
    // Many threads on one fresh device: the set-up runs at least once and the flag ends set.
    ctr::PerDeviceOnce raced;
    std::atomic<int> runs{0};
    std::vector<std::thread> ts;
    for (int i = 0; i < 16; ++i)
        ts.emplace_back([&] { raced.run(3, 0, [&] { runs.fetch_add(1); return 0; }); });
    for (auto &t : ts) t.join();
    if (runs.load() < 1 || runs.load() > 16 || !raced.done(3)) return 7;
    std::printf("ok\n");
    return 0;
}
"""


def test_set_up_runs_once_per_device(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("needs g++")
    src = tmp_path / "per_device_test.cpp"
    exe = tmp_path / "per_device_test"
    src.write_text(DRIVER)
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, "failed check %d" % r.returncode
    assert r.stdout.strip() == "ok"
