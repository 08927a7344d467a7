"""Build libbfp8.so in-tree for sm_103a with nvcc.

    python -m block_scaled_fp8_token_gb300.build

compiles every source under csrc/ in parallel, then links them into
block_scaled_fp8_token_gb300/libbfp8.so. The CUDA runtime is linked
statically, and TMA descriptors are encoded through the driver entry point
the runtime exposes, so nothing else has to be on the library path.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libbfp8.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cpp", "quant.cu", "gemm_sm103.cu", "gemv_decode.cu"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbfp8")
    return cand


def _compile(src: Path, obj: Path, verbose: bool) -> str:
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v" if verbose else "-O3", "-I", str(PKG.parent / "include"),
           "-c", str(src), "-o", str(obj)]
    if src.suffix == ".cpp":
        cmd.insert(1, "-x")
        cmd.insert(2, "cu")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src.name}:\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr


def _stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = list(CSRC.glob("*")) + [PKG.parent / "include" / "bfp8.h"]
    return any(p.stat().st_mtime > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile and link libbfp8.so if any source is newer than it."""
    if not force and not _stale():
        return LIB
    BUILD.mkdir(exist_ok=True)
    objs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        futs = {}
        for s in SOURCES:
            src = CSRC / s
            obj = BUILD / (src.stem + ".o")
            objs.append(obj)
            futs[ex.submit(_compile, src, obj, verbose)] = s
        for f in cf.as_completed(futs):
            out = f.result()
            if verbose and out.strip():
                print(f"== {futs[f]}\n{out}", file=sys.stderr)
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [_nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
