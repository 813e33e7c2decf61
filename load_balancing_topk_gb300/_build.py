"""Build the in-tree CUDA library ``libmep.so`` for sm_103a with nvcc.

Each translation unit under ``csrc/`` is compiled in parallel, then linked
into a shared library beside this file. No CMake, no torch extension
machinery: the library exposes the plain C ABI of ``include/mep.h``.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libmep.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["abi.cu", "plan.cu", "permute.cu", "reduce_grad.cu", "prefetch.cu", "plan_static.cu",
           "grouped_gemm.cu", "permute_backward.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDACXX"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    files.append(os.path.join(INCLUDE, "mep.h"))
    return files


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, extra_flags: list[str] | None = None, lib: str = LIB_PATH,
          verbose: bool = False, src_dir: str | None = None) -> str:
    """Compile csrc/*.cu and link ``libmep.so``; returns its path.

    extra_flags, lib and src_dir build a separate copy (other macros, another
    output path, or a modified copy of csrc/) without touching the default
    library."""
    src = src_dir or CSRC
    if not force and extra_flags is None and src_dir is None and up_to_date(lib):
        return lib
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-I" + INCLUDE, "-Xcompiler", "-fPIC",
                    "-Xcompiler", "-fvisibility=hidden"] + list(extra_flags or [])
    tag = (str(abs(hash((tuple(extra_flags or []), src))))[:8]
           if (extra_flags or src_dir) else "main")

    def compile_one(name: str) -> str:
        obj = os.path.join(BUILD_DIR, f"{os.path.splitext(name)[0]}.{tag}.o")
        cmd = [cc] + flags + ["-I" + CSRC, "-c", os.path.join(src, name), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
