"""Build libattnres_gb300.so in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then the
objects are linked into one shared library next to this file. build(checked=
True) makes the range-checked variant, libattnres_gb300_checked.so (AR_CHECKED
defined: every kernel access is checked against the launch's buffers), from
the same sources in its own object folder.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libattnres_gb300.so")
LIB_CHECKED = os.path.join(HERE, "libattnres_gb300_checked.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_CHECKED if checked else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool | None = None) -> str:
    """Build the library (checked=None: the variant the binding loads, the
    range-checked one when AR_CHECKED=1 is set) and return its path."""
    if checked is None:
        checked = os.environ.get("AR_CHECKED", "") == "1"
    lib, bdir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and not ptxas_info and up_to_date(checked):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()
    objs = [os.path.join(bdir, os.path.basename(s) + ".o") for s in srcs]
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DAR_CHECKED"] if checked else [])

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{p.stderr}")
        return src, p.stderr

    workers = max(1, min(len(srcs), os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    if verbose or ptxas_info:
        for src, err in logs:
            if err.strip():
                print(f"== {os.path.basename(src)}\n{err}", file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    p = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checked=True if "--checked" in sys.argv else None))
