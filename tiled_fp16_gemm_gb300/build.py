"""Build libtgemm.so in-tree with nvcc for sm_103a (no CMake, one translation unit)."""

from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libtgemm.so")
ARCH = "arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libtgemm needs the CUDA toolkit to build")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in sources())


def nvcc_command(out: str = LIB, extra: list[str] | None = None) -> list[str]:
    return [
        _nvcc(), "-gencode", ARCH, "-O3", "-std=c++17", "-lineinfo",
        "-Xcompiler", "-fPIC", "-shared", "--expt-relaxed-constexpr",
        "-I", INCLUDE, "-I", CSRC,
        os.path.join(CSRC, "tgemm.cu"), "-o", out,
    ] + (extra or [])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libtgemm.so next to this file unless it is newer than every source."""
    if not force and up_to_date():
        return LIB
    tmp = LIB + ".tmp"
    cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else None)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose:
        print(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
