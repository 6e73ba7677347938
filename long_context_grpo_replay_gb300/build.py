"""Builds libls (the C-ABI CUDA library) in-tree for sm_103a.

Each .cu translation unit is compiled by its own nvcc process in parallel and
the objects are linked into ``_lib/libls.so`` next to this file.  The library
links the CUDA runtime dynamically so that it shares the runtime (and hence
streams and device pointers) with a PyTorch process that loaded it first.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

HERE = Path(__file__).resolve().parent
CSRC = HERE / "csrc"
INCLUDE = HERE.parent / "include"
LIBDIR = HERE / "_lib"
LIB = LIBDIR / "libls.so"
SOURCES = ["ls_api.cu", "ls_simt.cu", "ls_tc_fwd.cu", "ls_tc_bwd.cu", "ls_tc_dkdv.cu", "ls_noalloc.cu",
           "ls_gdn.cu", "ls_gdn_cp.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libls")
    return cand


def _cuda_home(nvcc: str) -> Path:
    return Path(nvcc).resolve().parent.parent


def _inputs():
    return [CSRC / s for s in SOURCES] + sorted(CSRC.glob("*.h")) + sorted(CSRC.glob("*.cuh")) + \
        sorted(INCLUDE.glob("*.h")) + [Path(__file__)]


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> Path:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    cuda = _cuda_home(nvcc)
    objdir = LIBDIR / "obj"
    objdir.mkdir(parents=True, exist_ok=True)
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                     f"-I{INCLUDE}", f"-I{CSRC}"] + list(extra_flags)
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = objdir / (Path(src).stem + ".o")
        cmd = [nvcc] + common + ["-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, err in results:
            sys.stderr.write(err)
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", str(tmp)] + \
        [str(o) for o, _ in results] + [f"-L{cuda / 'lib64'}",
                                          f"-Xlinker", f"-rpath,{cuda / 'lib64'}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    p = build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(p)
