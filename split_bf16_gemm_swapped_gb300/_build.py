"""Builds the package's native libraries in-tree (no pip install).

* ``_lib/libsplitk_sm103a.so``: the CUDA kernels and the C ABI declared in
  ``include/splitk.h``, compiled by nvcc for sm_103a only.
* ``_lib/libsynthetic.so``: the seeded input generator (plain C, gcc).

Both are rebuilt when a source is newer than the library.  Host code is
portable C/C++ (no x86 intrinsics, no -march=native), so the same sources
build on x86_64 and aarch64.
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
LIBDIR = PKG / "_lib"

SPLITK_LIB = LIBDIR / "libsplitk_sm103a.so"
SYNTHETIC_LIB = LIBDIR / "libsynthetic.so"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

# Translation units of the CUDA library; compiled in parallel, linked once.
SPLITK_SOURCES = ["splitk_kernel.cu", "splitk_persistent.cu", "splitk_copy.cu", "splitk_host.cu"]
SPLITK_HEADERS = ["splitk_device.cuh", "splitk_internal.h", "splitk_kernel_common.cuh"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return cand


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).exists() and Path(d).stat().st_mtime > t for d in deps)


def _run(cmd, cwd=None):
    res = subprocess.run(cmd, cwd=cwd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(
            "build command failed:\n  " + " ".join(map(str, cmd)) + "\n" +
            res.stdout[-4000:] + res.stderr[-8000:])
    return res


def build_synthetic(force: bool = False) -> Path:
    LIBDIR.mkdir(parents=True, exist_ok=True)
    src = CSRC / "synthetic.c"
    if force or _stale(SYNTHETIC_LIB, [src]):
        tmp = SYNTHETIC_LIB.with_suffix(f".{os.getpid()}.tmp")
        _run(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
              "-pthread", str(src), "-o", str(tmp), "-lm"])
        os.replace(tmp, SYNTHETIC_LIB)
    return SYNTHETIC_LIB


def build_splitk(force: bool = False, verbose_ptxas: bool = False) -> Path:
    LIBDIR.mkdir(parents=True, exist_ok=True)
    srcs = [CSRC / s for s in SPLITK_SOURCES]
    deps = srcs + [CSRC / h for h in SPLITK_HEADERS] + [INCLUDE / "splitk.h"]
    if not (force or _stale(SPLITK_LIB, deps)):
        return SPLITK_LIB
    nvcc = _nvcc()
    objdir = LIBDIR / f"obj.{os.getpid()}"
    objdir.mkdir(parents=True, exist_ok=True)
    common = [nvcc, *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", str(INCLUDE), "-I", str(CSRC)]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]

    def compile_one(src: Path):
        obj = objdir / (src.stem + ".o")
        res = _run(common + ["-c", str(src), "-o", str(obj)])
        return obj, res.stderr

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    tmp = SPLITK_LIB.with_suffix(f".{os.getpid()}.tmp")
    _run([nvcc, *ARCH_FLAGS, "-shared", "-o", str(tmp), *map(str, objs)])
    os.replace(tmp, SPLITK_LIB)
    shutil.rmtree(objdir, ignore_errors=True)
    if verbose_ptxas:
        for _, err in results:
            print(err)
    return SPLITK_LIB


def build_all(force: bool = False) -> None:
    build_synthetic(force)
    build_splitk(force)
