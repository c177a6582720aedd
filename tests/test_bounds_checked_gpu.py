"""The forward, backward and sampling-operator parity suites against the
bounds-checked build.

compute-sanitizer is closed on this machine, so this stands in for its memory
check on the hot path: libdcn_checked.so is the library compiled with
DCN_CHECK_BOUNDS.  In it the convolution's forward kernels (tensor-core and
CUDA-core) check every corner load, offset and mask fetch, and output store
against the byte ranges of the caller's tensors; an access outside is
skipped and raises a status bit that dcn_sync_status reports as
DCN_ERR_BOUNDS.  The convolution's tensor-core backward kernels (the column
gradient with its scatter, and the weight gradient) check the same way
every offset, mask and corner load and every reduction into grad_x,
grad_offset, grad_mask and grad_weight; the CUDA-core backward kernels are
not instrumented.  The multi-scale and single-scale sampling kernels,
forward and backward, check every corner-row load of the value tensor and
every reduction into the value gradient; their entry points take no handle,
so a thread that meets an access outside writes NaN into every output it
owns, which the suites' oracle comparisons reject.  The suites run against
that build in a child process: every case must still match the oracle (and
the convolution's report a clean status), so no gather, reduction or store
of theirs leaves its tensor.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_parity_gpu.py", "tests/test_parity_general_gpu.py",
          "tests/test_parity_channels_gpu.py", "tests/test_parity_f16_gpu.py",
          "tests/test_abi_gpu.py", "tests/test_zz_no_alloc.py",
          "tests/test_backward_gpu.py", "tests/test_backward_full_gpu.py",
          "tests/test_msda_gpu.py", "tests/test_msda_backward_gpu.py",
          "tests/test_attn_gpu.py", "tests/test_attn_backward_gpu.py"]


def test_forward_suites_pass_bounds_checked():
    from deformable_convolution_vision_gb300 import build
    lib = build.build(checked=True)
    env = dict(os.environ, DCN_TEST_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-x", "-m", "gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1500)
    tail = "\n".join(r.stdout.splitlines()[-15:])
    assert r.returncode == 0, f"parity suites against the bounds-checked build failed:\n{tail}\n{r.stderr[-2000:]}"
    # the child ran against the checked library (its report header names it)
    assert f"dcn library under test: {lib}" in r.stdout
