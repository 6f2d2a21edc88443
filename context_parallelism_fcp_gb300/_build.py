"""Build of the in-tree shared library ``libfcp.so`` (C ABI of include/fcp.h) for sm_103a.

Each translation unit is compiled in parallel with nvcc (one -gencode, sm_103a only) and
linked with the static CUDA runtime, so the library needs only the NVIDIA driver at run
time. A content hash of the sources and flags skips rebuilding when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys
from typing import List, Optional

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libfcp.so")

SOURCES = ["fcp_plan.cpp", "fcp_solver.cpp", "fcp_validate.cpp", "fcp_fwd.cu", "fcp_bwd.cu", "fcp_bwd_tile.cu", "fcp_merge.cu"]
HEADERS = ["fcp_internal.h", "fcp_cuda_util.h", "fcp_sm100.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INCLUDE,
          "-I", CSRC]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfcp.so")


def _digest(extra: List[str]) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(INCLUDE, "fcp.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + COMMON + extra).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile libfcp.so if the sources changed; return its path."""
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    digest = _digest([])
    stamp = LIB_PATH + ".stamp"
    if not force and not ptxas_info and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(name: str):
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD_DIR, name + ".o")
        cmd = [nvcc] + ARCH + COMMON + extra + ["-c", src, "-o", obj]
        if name.endswith(".cpp"):
            cmd = [nvcc] + COMMON + ["-x", "c++", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, obj, r

    objs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for name, obj, r in ex.map(compile_one, SOURCES):
            if verbose or ptxas_info:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
            objs.append(obj)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


def main(argv: Optional[List[str]] = None) -> None:
    argv = sys.argv[1:] if argv is None else argv
    path = build(verbose="-v" in argv, ptxas_info="--ptxas" in argv, force="--force" in argv)
    print(path)


if __name__ == "__main__":
    main()
