"""Build the CUDA library (libspecverify.so) in-tree for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then the
objects link into one shared library next to this file.  No CMake, no torch
extension machinery: the library exports a plain C ABI (include/spec_verify.h).
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libspecverify.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]

SOURCES = ["api.cu", "kv_cache.cu", "verify.cu", "verify_bf16.cu", "verify_f32.cu", "verify_mixed.cu",
           "verify_static.cu", "verify_topk_bf16.cu", "verify_topk_f32.cu", "verify_topk_mixed.cu",
           "tree_verify.cu", "tree_bf16.cu", "tree_f32.cu", "tree_opts_bf16.cu", "tree_opts_f32.cu",
           "stream.cu", "stream_more.cu"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, extra=(), out: str = LIB, only=None) -> str:
    """Compile the sources and link `out` (default: the package's library).
    `extra` nvcc flags apply to the translation units compiled; with `only`,
    just those sources are recompiled and the others' objects are reused."""
    os.makedirs(BUILD, exist_ok=True)
    todo = SOURCES if only is None else [s for s in SOURCES if s in only]
    with cf.ThreadPoolExecutor(max_workers=len(todo)) as ex:
        list(ex.map(lambda s: _compile(s, list(extra)), todo))
    objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print("built", out, file=sys.stderr)
    return out


if __name__ == "__main__":
    build(verbose=True)
