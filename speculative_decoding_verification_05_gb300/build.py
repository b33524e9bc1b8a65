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
# the same sources with device-side index checks (-DSPEC_DEBUG): failed checks
# skip the access and are counted (spec_debug_failures), nothing traps
DEBUG_LIB = os.path.join(HERE, "libspecverify_debug.so")
SOURCES = ["csrc/api.cu", "csrc/rows.cu", "csrc/rows_smem.cu", "csrc/argmax.cu", "csrc/mentor.cu",
           "csrc/noalloc.cu", "csrc/tree_build.cu", "csrc/beta.cu", "csrc/planner.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-Xptxas", "-v", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(HERE, "csrc")]


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")
    return nvcc


def _compile(job):
    src, debug = job
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", "_debug.o" if debug else ".o"))
    cmd = [_nvcc(), *ARCH, *CFLAGS, *(["-DSPEC_DEBUG"] if debug else []), "-c", os.path.join(HERE, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(objs, lib):
    tmp = lib + ".tmp"
    r = subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(verbose=False, debug=True):
    """Compile every translation unit and link libspecverify.so (and, with
    `debug`, libspecverify_debug.so with device-side index checks), all
    translation units in parallel; returns the release library's path."""
    os.makedirs(BUILD, exist_ok=True)
    jobs = [(src, False) for src in SOURCES] + ([(src, True) for src in SOURCES] if debug else [])
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(_compile, jobs))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (obj, log), (src, dbg) in zip(results, jobs):
            if not dbg:
                f.write(f"==== {src}\n{log}\n")
    _link([o for (o, _), (_, dbg) in zip(results, jobs) if not dbg], LIB)
    if debug:
        _link([o for (o, _), (_, dbg) in zip(results, jobs) if dbg], DEBUG_LIB)
    if verbose:
        print(f"built {LIB}" + (f" and {DEBUG_LIB}" if debug else ""))
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
