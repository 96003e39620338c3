"""Build libwkv.so in-tree with nvcc for sm_103a (B300).

    python -m rwkv_linear_attention_backward_b300.build [--verbose]

Compiles every ``csrc/*.cu`` into one shared library next to this file.
``--verbose`` adds ``-Xptxas -v`` (registers, spills, shared memory per
kernel).  Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIBRARY = PKG / "libwkv.so"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libwkv.so")
    return cand


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _inputs() -> list[Path]:
    return sources() + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + sorted(INCLUDE.glob("*.h"))


def stale() -> bool:
    if not LIBRARY.exists():
        return True
    t = LIBRARY.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _inputs())


def command(verbose: bool = False, output: Path = LIBRARY) -> list[str]:
    cmd = [nvcc(), *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
           "-cudart", "shared", f"-I{INCLUDE}", f"-I{CSRC}", "-o", str(output)]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    return cmd + [str(s) for s in sources()]


def build(force: bool = False, verbose: bool = False) -> Path:
    if force or verbose or stale():
        tmp = LIBRARY.with_suffix(".so.tmp")
        proc = subprocess.run(command(verbose, tmp), capture_output=True, text=True)
        if proc.returncode != 0:
            sys.stderr.write(proc.stdout + proc.stderr)
            raise RuntimeError("nvcc failed building libwkv.so")
        if verbose:
            sys.stdout.write(proc.stdout + proc.stderr)
        os.replace(tmp, LIBRARY)
    return LIBRARY


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--verbose", action="store_true", help="print ptxas resource usage")
    ap.add_argument("--force", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    main()
