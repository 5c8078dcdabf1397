"""Builds libspec_verify.so in-tree from csrc/ with nvcc for sm_103a only, and its checked
build libspec_verify_checked.so (the same sources compiled with SPEC_CHECKED).

Each translation unit is compiled in its own nvcc process (in parallel), then linked into one
shared library per variant with the CUDA runtime linked statically.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libspec_verify.so")
CHECKED_LIB_PATH = os.path.join(PKG, "libspec_verify_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspec_verify.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def lib_path(checked: bool = False) -> str:
    """The normal library, or the checked build (compiled with SPEC_CHECKED: every index the
    kernels compute is range-checked and a violation reported through the status word)."""
    return CHECKED_LIB_PATH if checked else LIB_PATH


def up_to_date(checked: bool = False) -> bool:
    path = lib_path(checked)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool = False) -> str:
    """Builds one library (the normal one, or the checked build); returns its path."""
    return build_all(force, verbose, ptxas_info, variants=(checked,))[0]


def build_all(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
              variants=(False, True)):
    """Builds the requested variants (False: normal, True: checked), all translation units
    compiled in parallel; returns their paths."""
    todo = [v for v in variants if force or not up_to_date(v)]
    if not todo:
        return [lib_path(v) for v in variants]
    cc = nvcc()
    srcs = sources()
    jobs = []
    for v in todo:
        bdir = BUILD_DIR + ("_checked" if v else "")
        os.makedirs(bdir, exist_ok=True)
        jobs += [(v, src, os.path.join(bdir, os.path.basename(src)[:-3] + ".o")) for src in srcs]

    def compile_one(job):
        v, src, obj = job
        cmd = [cc] + NVCC_FLAGS + (["-DSPEC_CHECKED"] if v else []) + (
            ["-Xptxas", "-v"] if ptxas_info else []) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return v, obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_info:
        for _, _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    for v in todo:
        path = lib_path(v)
        tmp = path + f".tmp{os.getpid()}"
        objs = [o for vv, o, _ in results if vv == v]
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
    return [lib_path(v) for v in variants]


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                    variants=(False, True) if "--checked" in sys.argv else (False,)))
