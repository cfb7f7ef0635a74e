"""Builds libkda.so (all CUDA and host C++ sources under csrc/) for sm_103a with nvcc.

Each translation unit compiles in parallel with
``-gencode arch=compute_103a,code=sm_103a``; the objects link into
``_build/libkda.so`` next to this file (git-ignored).  Run as a module or via
``__graft_entry__.build()``.
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
BUILD = PKG / "_build"
LIB = BUILD / "libkda.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found")
    return cand


def sources() -> list[Path]:
    """CUDA translation units and host-only C++ ones (compiled by nvcc too)."""
    return sorted([*CSRC.glob("*.cu"), *CSRC.glob("*.cpp")])


def _stale(obj: Path, src: Path) -> bool:
    if not obj.exists():
        return True
    deps = [src, INCLUDE / "kda.h", *CSRC.glob("*.h"), *CSRC.glob("*.cuh"), Path(__file__)]
    return any(d.stat().st_mtime > obj.stat().st_mtime for d in deps if d.exists())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> Path:
    BUILD.mkdir(parents=True, exist_ok=True)
    cc = nvcc()
    extra = list(extra_flags or [])

    def compile_one(src: Path) -> Path:
        obj = BUILD / (src.stem + ".o")
        if force or extra or _stale(obj, src):
            cmd = [cc, *ARCH, *FLAGS, *extra, "-I", str(INCLUDE), "-I", str(CSRC), "-c", str(src), "-o", str(obj)]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src.name}")
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if force or extra or not LIB.exists() or any(o.stat().st_mtime > LIB.stat().st_mtime for o in objs):
        tmp = BUILD / f"libkda.{os.getpid()}.tmp.so"
        cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("nvcc link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
