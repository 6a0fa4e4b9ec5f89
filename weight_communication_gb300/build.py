"""Build the CUDA library (libwc.so) in-tree for sm_103a.

    python -m weight_communication_gb300.build

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into one shared library with the CUDA runtime linked statically, so the
library needs only the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
BUILD = PKG / "_build"
LIB = BUILD / "libwc.so"
# The checked build (every kernel access compared with its buffer's extent,
# see wc_checked_violations in include/wc.h) goes to a folder of its own.
CHECKED_BUILD = BUILD / "checked"
CHECKED_LIB = CHECKED_BUILD / "libwc.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Exact IEEE arithmetic: no flush to zero, IEEE division and square root, no
# contraction of multiply-add pairs (the kernels also use explicitly rounded
# intrinsics wherever rounding matters).
NVCC_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-ftz=false", "-prec-div=true",
              "-prec-sqrt=true", "-fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", "-Xptxas", "-v"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(exe).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwc.so")
    return exe


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _compile(src: Path, out: Path, defines: list[str]) -> tuple[Path, str]:
    obj = out / (src.stem + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *defines, "-c", str(src), "-o", str(obj)]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src.name}:\n{proc.stdout}\n{proc.stderr}")
    return obj, proc.stderr


def build(verbose: bool = False, checked: bool = False) -> Path:
    """Compile every kernel file and link libwc.so; checked=True builds the
    bounds-checked library (WC_CHECKED=1) into its own folder instead."""
    out, lib = (CHECKED_BUILD, CHECKED_LIB) if checked else (BUILD, LIB)
    defines = ["-DWC_CHECKED=1"] if checked else []
    out.mkdir(parents=True, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda s: _compile(s, out, defines), srcs))
    log = "\n".join(f"== {o.name}\n{err}" for o, err in results)
    (out / "ptxas.log").write_text(log)
    if verbose:
        print(log)
    tmp = out / "libwc.so.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", str(tmp),
           *[str(o) for o, _ in results]]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, checked="--checked" in sys.argv))
