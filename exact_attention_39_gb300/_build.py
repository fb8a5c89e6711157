"""Builds the sm_103a shared library (libfa_sm103.so) in-tree with nvcc."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_NAME = "libfa_sm103.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
SOURCES = ["fa_api.cu"]
DEPS = ["fa_fwd_kernel.cuh", "fa_bwd_kernel.cuh", "ptx.cuh"]
HEADERS = ["fa.h", "fa_selftest.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _stale():
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    inputs = [os.path.join(CSRC, f) for f in SOURCES + DEPS]
    inputs += [os.path.join(INCLUDE, h) for h in HEADERS]
    return any(os.path.getmtime(f) > t for f in inputs)


def build(force=False, verbose=False):
    """Compile libfa_sm103.so unless it is newer than its sources."""
    if not force and not _stale():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "-I", INCLUDE, "-o", tmp]
    if verbose:
        cmd.append("-Xptxas=-v")
    cmd += [os.path.join(CSRC, f) for f in SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
