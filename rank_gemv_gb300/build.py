"""Build step for libsgmv.so: nvcc, sm_103a only, in-tree.

Compiles every ``csrc/*.cu`` in parallel into ``_build/`` and links
``libsgmv.so`` next to this file.  A build is skipped when the library is
newer than every source and header.  ``python -m rank_gemv_gb300.build [-v]``
rebuilds from the command line (``-v`` prints ptxas register / spill / shared
memory usage).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

HERE = Path(__file__).resolve().parent
ROOT = HERE.parent
CSRC = HERE / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = HERE / "_build"
LIB = HERE / "libsgmv.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]
CUDA_LIB = "/usr/local/cuda/lib64"


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists() and not shutil.which(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _deps():
    return [*CSRC.iterdir(), INCLUDE / "sgmv.h", Path(__file__)]


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    newest = max(p.stat().st_mtime for p in _deps())
    return LIB.stat().st_mtime >= newest


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and not verbose and up_to_date():
        return LIB
    BUILD_DIR.mkdir(exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src: Path) -> Path:
        obj = BUILD_DIR / (src.stem + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", str(src), "-o", str(obj)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{res.stderr}")
        if verbose:
            sys.stderr.write(res.stderr)
        return obj

    sources = sorted(CSRC.glob("*.cu"))
    with ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources))
    tmp = LIB.with_name(f".libsgmv.{os.getpid()}.so")
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *map(str, objs),
           "-Xlinker", f"-rpath,{CUDA_LIB}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
