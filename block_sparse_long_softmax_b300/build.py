"""Build libskipsm.so (the C-ABI library) in-tree for sm_103a.

    python -m block_sparse_long_softmax_b300.build

Compiles every .cu under csrc/ with nvcc into
block_sparse_long_softmax_b300/libskipsm.so next to this file.

    python -m block_sparse_long_softmax_b300.build --trace

builds the test-only instrumented copy, libskipsm_trace.so (-DSKIPSM_TRACE=1: the
prefill kernel stamps clock64 at fixed points of one CTA's tile loop; see
tests/test_gpu_trace.py).  The package never loads it.
"""

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libskipsm.so")
TRACE_LIB = os.path.join(HERE, "libskipsm_trace.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def sources():
    return sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")))


def build(verbose: bool = False, extra=(), trace: bool = False) -> str:
    srcs = sources()
    out = TRACE_LIB if trace else LIB
    deps = srcs + glob.glob(os.path.join(HERE, "csrc", "*.h")) + \
        glob.glob(os.path.join(HERE, "csrc", "*.cuh")) + [os.path.join(ROOT, "include", "skipsm.h")]
    if os.path.exists(out) and not extra and \
            os.path.getmtime(out) >= max(os.path.getmtime(d) for d in deps):
        return out
    defs = ["-DSKIPSM_TRACE=1"] if trace else []
    cmd = [nvcc(), *ARCH, *FLAGS, *defs, *extra, *srcs, "-o", out + ".tmp", "-lcudart_static"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    args = sys.argv[1:]
    trace = "--trace" in args
    extra = [a for a in args if a != "--trace"]
    print(build(verbose=True, extra=extra, trace=trace))
