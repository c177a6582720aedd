"""Build the CUDA library ``libdcn.so`` in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel, then linked
into one shared library next to this file.  The C runtime is linked
statically, so the library loads on a machine without a GPU (its entry
points then report DCN_ERR_NO_DEVICE).
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBRARY = os.path.join(HERE, "libdcn.so")
CHECKED_LIBRARY = os.path.join(HERE, "libdcn_checked.so")

SOURCES = ["dcn_api.cu", "dcn_simt.cu", "dcn_tc.cu", "dcn_noalloc.cu", "dcn_backward.cu",
           "dcn_bwd_tc.cu", "dcn_bwd_wgrad_tc.cu", "dcn_msda.cu", "dcn_msda_bwd.cu", "dcn_attn.cu", "dcn_attn_bwd.cu",
           "dcn_layout.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdcn.so")
    return exe


def _compile(src, extra, bdir=None):
    obj = os.path.join(bdir or BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False, extra=(), checked=False):
    """Compile every CUDA source for sm_103a and link libdcn.so; returns its
    path.  checked=True builds the bounds-checked variant instead
    (DCN_CHECK_BOUNDS: the forward kernels check every gather and store
    against the caller's tensors and report a skipped access through the
    status word), as libdcn_checked.so beside it."""
    out_lib = CHECKED_LIBRARY if checked else LIBRARY
    bdir = BUILD + "_checked" if checked else BUILD
    os.makedirs(bdir, exist_ok=True)
    extra = list(extra) + (["-DDCN_CHECK_BOUNDS"] if checked else [])
    if verbose:
        extra += ["-Xptxas", "-v"]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, bdir), SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = out_lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
