"""Builds libsmd.so (the sparse MLA decode C-ABI library) for sm_103a.

    python -m sparse_mla_decode_gb300.build [--force] [--trace]

--trace builds the tracing variant instead (-DSMD_TRACE: per-phase timestamps
of the decode kernels, smd_trace_read) into _build/trace/libsmd_trace.so; the
binding loads it when SMD_TRACE_BUILD=1.

nvcc compiles each translation unit in parallel and links a shared library
into sparse_mla_decode_gb300/_build/. Nothing is installed outside the tree.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libsmd.so")
TRACE_BUILD = os.path.join(BUILD, "trace")
TRACE_LIB = os.path.join(TRACE_BUILD, "libsmd_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the sparse MLA decode library needs the CUDA toolkit")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          trace: bool = False) -> str:
    lib, out_dir = (TRACE_LIB, TRACE_BUILD) if trace else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + ARCH + ["-I", INCLUDE, "-I", CSRC] + list(extra or [])
    if trace:
        flags.append("-DSMD_TRACE")

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [cc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, trace="--trace" in sys.argv))
