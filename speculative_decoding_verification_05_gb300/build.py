"""Build libspecverify.so in-tree with nvcc for sm_103a (GB300).

    python -m speculative_decoding_verification_05_gb300.build

compiles each CUDA translation unit in parallel into ``_build/`` and links
the shared library next to this file. Nothing is installed elsewhere.
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libspecverify.so")
SOURCES = ["csrc/api.cu", "csrc/rows.cu", "csrc/argmax.cu", "csrc/mentor.cu", "csrc/noalloc.cu",
           "csrc/tree_build.cu", "csrc/beta.cu", "csrc/planner.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-Xptxas", "-v", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(HERE, "csrc")]


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")
    return nvcc


def _compile(src):
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *CFLAGS, "-c", os.path.join(HERE, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False):
    """Compile every translation unit and link libspecverify.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
