"""In-tree build of libbsgemm.so for sm_103a with nvcc (no cmake, no torch).

Each translation unit compiles in its own nvcc process (in parallel), then
nvcc links the shared library next to this file. Rebuilds only when a source
or header is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = PKG / "libbsgemm.so"
SOURCES = ("api.cu", "gemm_persistent.cu", "gemm_pair.cu", "gemm_skinny.cu", "swizzle.cu", "noalloc.cu",
           "quantize.cu", "probe.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden,-O2",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbsgemm.so")


def _inputs() -> list[Path]:
    return [*(CSRC.glob("*.cu")), *(CSRC.glob("*.cuh")), *(CSRC.glob("*.h")),
            INCLUDE / "bsgemm.h", Path(__file__)]


def is_stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> Path:
    """Compile (if needed) and return the path of libbsgemm.so."""
    if not force and not is_stale():
        return LIB
    BUILD.mkdir(parents=True, exist_ok=True)
    exe = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(src: str):
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [exe, *ARCH, *FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log:
                print(log)
    tmp = LIB.with_suffix(f".tmp{os.getpid()}.so")
    cmd = [exe, *ARCH, "-shared", "-o", str(tmp), *(str(o) for o, _ in results)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":  # pragma: no cover
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
