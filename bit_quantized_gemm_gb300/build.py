"""Build the library's CUDA sources into an in-tree shared library.

nvcc compiles each translation unit for sm_103a (in parallel), then links
them, with the CUDA runtime statically, into ``libqgemm.so`` next to this
file. No cmake, no torch extension machinery.
"""
import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
SO = os.path.join(HERE, "libqgemm.so")
BUILD = os.path.join(HERE, "_build")
SOURCES = ["api.cu", "quantize.cu", "pack.cu", "gemm_small.cu", "gemm_large.cu", "gemm_skinny.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xptxas", "-v", "-I", os.path.join(HERE, "..", "include")]


def nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "qgemm.h"))
    return max(os.path.getmtime(f) for f in files)


def _compile(src):
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, p.stdout, p.stderr))
    with open(os.path.join(BUILD, src + ".ptxas.txt"), "w") as f:
        f.write(p.stderr)
    return obj


def build(force=False, verbose=False):
    """Compile (if stale) and return the path of libqgemm.so."""
    if not force and os.path.exists(SO) and os.path.getmtime(SO) >= _deps():
        return SO
    os.makedirs(BUILD, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = SO + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs, "-cudart", "static"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (p.stdout, p.stderr))
    os.replace(tmp, SO)
    if verbose:
        for src in SOURCES:
            print(open(os.path.join(BUILD, src + ".ptxas.txt")).read())
    return SO


if __name__ == "__main__":
    build(force=True, verbose=True)
