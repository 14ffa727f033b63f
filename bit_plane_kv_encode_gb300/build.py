"""Build libbpkv.so in-tree with nvcc for sm_103a (one -gencode, parallel
compile of the translation units, then one shared-library link)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["encode.cu", "depths.cu", "scan.cu", "select.cu", "attend.cu", "abi.cu", "noalloc.cu",
           "calibrate.cu", "vdepth.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def lib_path(checks: bool | None = None) -> str:
    """The library (checks: the bounds-checked build; None: as the
    BPKV_CHECKS environment variable says)."""
    if checks is None:
        checks = os.environ.get("BPKV_CHECKS") == "1"
    return os.path.join(HERE, f"libbpkv_{'checks_' if checks else ''}{platform.machine()}.so")


def _nvcc() -> str:
    for cand in [shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def build(force: bool = False, verbose: bool = False, checks: bool | None = None) -> str:
    """Compile and link the library; checks: the bounds-checked variant
    (-DBPKV_CHECKS=1, its own objects and library file)."""
    if checks is None:
        checks = os.environ.get("BPKV_CHECKS") == "1"
    out = lib_path(checks)
    deps = ([os.path.join(CSRC, s) for s in SOURCES] +
            [os.path.join(CSRC, h) for h in sorted(os.listdir(CSRC)) if h.endswith(".cuh")] +
            [os.path.join(INCLUDE, "bpkv.h")])
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(os.path.getmtime(d) for d in deps):
        return out
    nvcc = _nvcc()
    objdir = os.path.join(HERE, "_build", platform.machine() + ("_checks" if checks else ""))
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src: str) -> tuple:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *(["-DBPKV_CHECKS=1"] if checks else []), "-I", INCLUDE, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    objs = [o for o, _ in results]
    tmp = out + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{_cuda_lib_dir(nvcc)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
