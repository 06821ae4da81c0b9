"""Builds libmoe_gb300.so in-tree with nvcc for sm_103a (no torch extension
machinery: the library is plain C ABI + CUDA)."""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libmoe_gb300.so"
SOURCES = ["moe_kernels.cu", "moe_decode.cu", "moe_abi.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> Path:
    headers = list(CSRC.glob("*.h")) + list((ROOT / "include").glob("*.h"))
    BUILD.mkdir(exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I", str(ROOT / "include"), "-I", str(CSRC)]
    if verbose:
        flags += ["-Xptxas", "-v"]
    procs, objs = [], []
    for src in SOURCES:
        obj = BUILD / (Path(src).stem + ".o")
        objs.append(obj)
        if force or _stale(obj, [CSRC / src] + headers):
            tmp = obj.with_suffix(".o.tmp%d" % os.getpid())
            procs.append((subprocess.Popen([nvcc(), *flags, "-c", str(CSRC / src), "-o", str(tmp)],
                                           stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True),
                          tmp, obj))
    errors = []
    for proc, tmp, obj in procs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            errors.append(out)
        else:
            os.replace(tmp, obj)
            if verbose and out:
                print(out)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    if force or _stale(LIB, objs):
        tmp = LIB.with_suffix(".so.tmp%d" % os.getpid())
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", str(tmp), *map(str, objs)], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    build_library(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
