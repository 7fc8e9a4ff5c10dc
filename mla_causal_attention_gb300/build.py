"""Builds libmla_attn.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each .cu file is compiled in parallel, then linked into one shared library with a static
CUDA runtime.  Usage: ``python -m mla_causal_attention_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmla_attn.so")
SOURCES = ["host.cu", "decode.cu", "prefill.cu", "noalloc.cu", "rope.cu", "mask.cu", "latent.cu",
           "oproj.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
                   *extra]


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "mla_attn.h")]
    newest = max(os.path.getmtime(d) for d in deps)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest and not extra_flags:
        return LIB
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-Xlinker",
           "--exclude-libs,ALL"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def build_test_variant(name: str, source: str, defines) -> str:
    """A test-only copy of the library in which `source` is compiled with extra -D
    defines (the other objects are the library's own).  It lives under _build/test_<name>/
    and is never what the package loads; the product build sets none of these defines."""
    build_library()
    out_dir = os.path.join(BUILD, f"test_{name}")
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, f"libmla_attn_{name}.so")
    if os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(LIB):
        return lib
    cc = nvcc()
    obj = os.path.join(out_dir, source.replace(".cu", ".o"))
    r = subprocess.run([cc, *_flags(defines), "-c", os.path.join(CSRC, source), "-o", obj],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {source} ({name}):\n{r.stderr}")
    objs = [obj if s == source else os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
                        "-Xlinker", "--exclude-libs,ALL"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed ({name}):\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
