"""Builds libh2o.so in-tree for sm_103a (GB300).

CUDA sources are compiled by nvcc with `-gencode arch=compute_103a,code=sm_103a`;
the C-ABI host file is compiled by g++ against PyTorch's c10 headers (for the
caching allocator and the current stream) and everything is linked into one
shared library next to this file. Objects go to `_build/` beside it.
Translation units compile in parallel; nothing is rebuilt when the library is
newer than every source and header.
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
BUILD = PKG / "_build"
LIB = PKG / "libh2o.so"

CU_SOURCES = ["decode.cu", "decode_multi.cu", "decode_ring.cu", "prefill.cu", "select.cu"]
CPP_SOURCES = ["h2o_api.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> Path:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home:
        return Path(home)
    nvcc = shutil.which("nvcc")
    if nvcc:
        return Path(nvcc).resolve().parent.parent
    return Path("/usr/local/cuda")


def _torch_paths():
    import torch
    from torch.utils import cpp_extension

    inc = [Path(p) for p in cpp_extension.include_paths()]
    lib = Path(torch.__file__).resolve().parent / "lib"
    abi = int(torch._C._GLIBCXX_USE_CXX11_ABI)
    return inc, lib, abi


def _sources():
    return ([CSRC / s for s in CU_SOURCES + CPP_SOURCES] + list(CSRC.glob("*.cuh"))
            + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h")))


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _sources())


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({r.returncode}):\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile every CUDA/C++ translation unit for sm_103a and link libh2o.so."""
    if not force and up_to_date():
        return LIB
    cuda = _cuda_home()
    nvcc = str(cuda / "bin" / "nvcc")
    tinc, tlib, abi = _torch_paths()
    BUILD.mkdir(exist_ok=True)
    common = [f"-I{INCLUDE}", f"-I{CSRC}"]
    jobs = []
    for s in CU_SOURCES:
        obj = BUILD / (s + ".o")
        jobs.append([nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", *common, "-c", str(CSRC / s), "-o", str(obj)])
    for s in CPP_SOURCES:
        obj = BUILD / (s + ".o")
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", f"-D_GLIBCXX_USE_CXX11_ABI={abi}",
                     *common, f"-I{cuda / 'include'}", *[f"-I{p}" for p in tinc],
                     "-c", str(CSRC / s), "-o", str(obj)])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for f in [ex.submit(_run, j) for j in jobs]:
            f.result()
    objs = [str(BUILD / (s + ".o")) for s in CU_SOURCES + CPP_SOURCES]
    tmp = LIB.with_suffix(".so.tmp")
    _run(["g++", "-shared", "-o", str(tmp), *objs,
          f"-L{cuda / 'lib64'}", "-lcudart", f"-L{tlib}", "-lc10_cuda", "-lc10",
          f"-Wl,-rpath,{tlib}", f"-Wl,-rpath,{cuda / 'lib64'}"])
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
