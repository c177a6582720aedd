"""The launchers' per-device attribute record, compiled on its own with g++.

cudaFuncSetAttribute acts on the device current at the call, so the
record of the shared-memory limit already set must be kept per device: a
launch on a second device (or with a handle made there) must make the call
again even though the first device has the value.  The setter here is a
fake that counts its calls per device, so no GPU is needed.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "deformable_convolution_vision_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "dcn_attr_cache.h"
#define CHECK(expr) do { if (!(expr)) { std::printf("FAIL %s\n", #expr); return 1; } } while (0)
int calls[8];
int fail_next = 0;
dcn::PerDeviceValue<4> rec;
int launch(int dev, int smem) {
    return rec.ensure(dev, smem, [&] {
        ++calls[dev < 0 ? 7 : dev % 8];
        if (fail_next) { fail_next = 0; return 1; }   // an error code
        return 0;
    });
}
int main() {
    CHECK(launch(0, 1000) == 0 && calls[0] == 1);
    CHECK(launch(0, 1000) == 0 && calls[0] == 1);      // recorded on device 0
    CHECK(launch(1, 1000) == 0 && calls[1] == 1);      // device 1 sets its own
    CHECK(launch(1, 1000) == 0 && calls[1] == 1);
    CHECK(launch(0, 2000) == 0 && calls[0] == 2);      // a new value is set again
    CHECK(launch(1, 1000) == 0 && calls[1] == 1);      // device 1 unchanged
    fail_next = 1;
    CHECK(launch(2, 500) == 1 && calls[2] == 1);       // a failed set is not recorded
    CHECK(launch(2, 500) == 0 && calls[2] == 2);
    CHECK(launch(2, 500) == 0 && calls[2] == 2);
    CHECK(launch(5, 500) == 0 && launch(5, 500) == 0 && calls[5] == 2);   // outside the table
    CHECK(launch(-1, 500) == 0 && calls[7] == 1);
    std::printf("ok\n");
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_attribute_record_is_per_device(tmp_path):
    src = tmp_path / "attr.cpp"
    exe = tmp_path / "attr"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-O2", "-Wall", "-Werror", "-I", CSRC, str(src), "-o",
                    str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout
