"""Builds libtq.so (the C-ABI library) in-tree for sm_103a.

Usage: ``python -m kv_cache_quantization_store_gb300.build`` or ``build()``.
Each source compiles in parallel with nvcc (one -gencode, -lineinfo);
objects go to ``_build/`` next to this file and the library to
``libtq.so`` beside it.  CUDA's runtime is linked statically.
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
OUT_DIR = PKG / "_build"
LIB = PKG / "libtq.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = [
    "tq_host.cpp", "tq_store.cu", "tq_decode.cu", "tq_decode_mma.cu", "tq_decode_mma_d64.cu",
    "tq_decode_mma_d128.cu", "tq_decode_mma_d256.cu", "tq_dequant.cu", "tq_noalloc.cu", "tq_dense.cu",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtq.so")


def _flags(extra=()) -> list[str]:
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            f"-I{INCLUDE}", f"-I{CSRC}", *extra]


def _compile(src: str, extra) -> Path:
    obj = OUT_DIR / (Path(src).stem + ".o")
    cmd = [nvcc(), *_flags(extra), "-c", str(CSRC / src), "-o", str(obj)]
    if src.endswith(".cu"):
        cmd.insert(1, "--expt-relaxed-constexpr")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if os.environ.get("TQ_BUILD_VERBOSE"):
        sys.stderr.write(res.stdout + res.stderr)
    return obj


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = list(CSRC.glob("*")) + list(INCLUDE.glob("*.h")) + [Path(__file__)]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, extra_flags=()) -> Path:
    """Compiles and links libtq.so unless it is newer than every source."""
    if not force and not _stale():
        return LIB
    OUT_DIR.mkdir(exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra_flags), SOURCES))
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
