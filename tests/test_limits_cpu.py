"""The entry points' element-count check, compiled on its own with g++.

`within_index_limit` must accept a product of dimensions exactly when it is
at most 2^31 - 1, whatever the factors: products that overflow 64 bits
must not wrap round into accepted ones.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "deformable_convolution_vision_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "dcn_limits.h"
using dcn::within_index_limit;
#define CHECK(expr, want) do { if ((expr) != (want)) { std::printf("FAIL %s\n", #expr); return 1; } } while (0)
int main() {
    const long long lim = (1ll << 31) - 1;
    CHECK(within_index_limit({lim}), true);
    CHECK(within_index_limit({lim + 1}), false);
    CHECK(within_index_limit({1, lim, 1}), true);
    CHECK(within_index_limit({2, lim}), false);
    CHECK(within_index_limit({65536, 32767}), true);        // 2^31 - 2^16
    CHECK(within_index_limit({65536, 32768}), false);       // 2^31
    CHECK(within_index_limit({46341, 46340}), true);        // 2147441940
    CHECK(within_index_limit({46341, 46341}), false);       // 2147488281
    // 2^64 and 2^63: a plain 64-bit product wraps to 0 or goes negative
    CHECK(within_index_limit({65536, 65536, 65536, 65536}), false);
    CHECK(within_index_limit({1ll << 15, 1ll << 20, 1ll << 14, 1ll << 15}), false);
    CHECK(within_index_limit({1, 1ll << 30, 1ll << 30, 1, 16}), false);
    CHECK(within_index_limit({1, 5792, 5792, 64}), true);   // the largest problem tested
    CHECK(within_index_limit({0, lim}), true);
    CHECK(within_index_limit({-1, 4}), false);
    CHECK(within_index_limit({}), true);
    std::printf("ok\n");
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_within_index_limit(tmp_path):
    src = tmp_path / "limits.cpp"
    exe = tmp_path / "limits"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-O2", "-Wall", "-Werror", "-I", CSRC, str(src), "-o",
                    str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout
