"""Build the CUDA library libgdn_cpr.so in-tree with nvcc (sm_103a only).

Each translation unit in csrc/ is compiled in parallel, then linked into one shared
library exporting the C ABI of include/gdn_cpr.h.  --fmad=false keeps the compiler from
contracting any floating-point expression on its own: the kernels spell out every fused
multiply-add they want, which is part of what keeps all modes bit-identical.

build(checked=True) makes the bounds-checked debug variant libgdn_cpr_checked.so
(-DGDN_CHECKED=1: every kernel checks the index ranges it derives from device data against
its buffers and records GDN_DEVERR_BOUNDS instead of touching memory outside them); the
binding loads it instead of the ordinary library when GDN_CPR_CHECKED=1 is set.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgdn_cpr.so")
LIB_CHECKED = os.path.join(HERE, "libgdn_cpr_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include"), "-Xptxas", "-warn-spills"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "gdn_cpr.h")]


def needs_build(checked: bool = False) -> bool:
    lib = LIB_CHECKED if checked else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    if not force and not needs_build(checked):
        return lib
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(bdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if checked:
        extra += ["-DGDN_CHECKED=1"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
