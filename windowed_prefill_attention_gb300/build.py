"""Build libpa.so (the C-ABI library) in-tree with nvcc for sm_103a."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("pa_api.cu", "pa_kernels.cu", "pa_attention.cu", "pa_noalloc.cu", "pa_decode.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("pa_internal.h", "pa_ptx.cuh", "pa_tiles.cuh")] + [
    os.path.join(HERE, "..", "include", "pa.h")]
LIB = os.path.join(HERE, "libpa.so")
# the tensor-core throughput probe the benchmark's roofline uses (its own library)
PEAK_SOURCES = [os.path.join(CSRC, "pa_peak.cu")]
PEAK_HEADERS = [os.path.join(HERE, "..", "include", "pa_peak.h")]
PEAK_LIB = os.path.join(HERE, "libpa_peak.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "--threads", "0"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def stale(lib, sources, headers) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in sources + headers)


def _compile(lib, sources, verbose):
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + sources + ["-o", tmp]
    return subprocess.Popen(cmd), tmp, lib


def build(force: bool = False, verbose: bool = False) -> str:
    jobs = []
    if force or stale(LIB, SOURCES, HEADERS):
        jobs.append(_compile(LIB, SOURCES, verbose))
    if force or stale(PEAK_LIB, PEAK_SOURCES, PEAK_HEADERS):
        jobs.append(_compile(PEAK_LIB, PEAK_SOURCES, verbose))
    for proc, tmp, lib in jobs:
        if proc.wait() != 0:
            raise subprocess.CalledProcessError(proc.returncode, "nvcc -> " + os.path.basename(lib))
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
