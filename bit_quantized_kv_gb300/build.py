"""Build the CUDA library libuq.so (sm_103a) in-tree with nvcc.

The translation units are compiled in parallel and linked into
``bit_quantized_kv_gb300/_build/libuq.so`` with the CUDA runtime linked
statically, so the library needs only the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libuq.so")

SOURCES = ["uq_api.cu", "uq_store.cu", "uq_decode.cu", "uq_dequant.cu", "uq_noalloc.cu"]
HEADERS = ["uq_device.cuh", "uq_decode_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _inputs():
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "uq.h"))
    paths.append(os.path.abspath(__file__))
    return paths


def _up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


# Test-only variants of the library, built beside it under their own names and
# never loaded by the package: name -> extra nvcc defines.  "stuck_tile" leaves
# one page copy of the decode kernel unissued and shortens the bounded waits,
# so that a test can watch a wait run out and the kernel return.
VARIANTS = {
    "stuck_tile": ["-DUQ_TEST_STUCK_TILE", "-DUQ_WAIT_SUSPEND_NS=1024u", "-DUQ_WAIT_SPIN_LIMIT=256u"],
}


def variant_path(name: str) -> str:
    return os.path.join(BUILD, f"libuq_{name}.so")


def build(force: bool = False, verbose: bool = False, variant: str | None = None) -> str:
    """Compile and link libuq.so (or a test variant of it) if any source
    changed; return its path."""
    lib = LIB if variant is None else variant_path(variant)
    defines = [] if variant is None else VARIANTS[variant]
    tag = "" if variant is None else f"_{variant}"
    if not force and _up_to_date(lib):
        return lib
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", f"{tag}.o"))
        cmd = [nvcc, *NVCC_FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
