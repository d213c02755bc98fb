"""Build libpa.so, the CUDA library behind the C ABI in include/pa.h, for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one shared
library next to this file (git-ignored).  The CUDA runtime is linked statically, so
the library needs only the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = ROOT / "_build"
LIBRARY = PKG / "libpa.so"
SOURCES = ["pa_api.cu", "pa_cache.cu", "pa_decode.cu", "pa_prefix.cu", "pa_multi.cu", "pa_multi_tc.cu", "pa_noalloc.cu", "pa_blocks.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libpa.so")


def compile_flags(ptxas_verbose: bool = False) -> list[str]:
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
             "-I", str(INCLUDE), "-I", str(CSRC)]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    return flags


def _stale(output: Path, inputs: list[Path]) -> bool:
    if not output.exists():
        return True
    t = output.stat().st_mtime
    return any(p.stat().st_mtime > t for p in inputs)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> Path:
    """Compile and link libpa.so (skipped when it is newer than every source)."""
    BUILD.mkdir(exist_ok=True)
    headers = sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + sorted(INCLUDE.glob("*.h"))
    cc = nvcc()
    objects = []
    jobs = []
    for src in SOURCES:
        s = CSRC / src
        o = BUILD / (s.stem + ".o")
        objects.append(o)
        if force or ptxas_verbose or _stale(o, [s, *headers, Path(__file__)]):
            jobs.append([cc, *compile_flags(ptxas_verbose), "-c", str(s), "-o", str(o)])

    def run(cmd):
        return subprocess.run(cmd, capture_output=True, text=True)

    with ThreadPoolExecutor(max_workers=len(jobs) or 1) as pool:
        results = list(pool.map(run, jobs))
    for cmd, res in zip(jobs, results):
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}:\n{res.stderr}")
        if not quiet or ptxas_verbose:
            sys.stderr.write(res.stderr)
    if force or jobs or _stale(LIBRARY, objects):
        tmp = LIBRARY.with_suffix(f".{os.getpid()}.tmp")
        cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objects)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv, quiet=False)
    print(LIBRARY)
