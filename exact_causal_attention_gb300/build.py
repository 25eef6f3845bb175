"""Builds the CUDA library in-tree: one nvcc invocation, sm_103a only."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libeca_attn.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
# The same sources with ECA_ANATOMY: the attention kernel records per-CTA milestone
# stamps (a measurement aid; nothing else changes).
ANATOMY_LIB_PATH = os.path.join(BUILD_DIR, "libeca_attn_anatomy.so")
SOURCES = ["attn_api.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))]
    files.append(os.path.join(INCLUDE, "attn.h"))
    return files


def _command(out: str, defines, verbose: bool):
    cuda_lib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC",
           "-cudart", "shared", "-I", INCLUDE, "-I", CSRC, "-Xlinker", f"-rpath,{cuda_lib}", *defines,
           "-o", out, *[os.path.join(CSRC, s) for s in SOURCES]]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ into _build/libeca_attn.so (and the anatomy variant beside it, in
    parallel) unless both are newer than every source.  Returns the main library."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(f) for f in _deps())
    todo = [(path, defines) for path, defines in ((LIB_PATH, []), (ANATOMY_LIB_PATH, ["-DECA_ANATOMY"]))
            if force or not os.path.exists(path) or os.path.getmtime(path) < newest]
    procs = []
    for path, defines in todo:
        tmp = path + f".tmp{os.getpid()}"
        procs.append((subprocess.Popen(_command(tmp, defines, verbose)), tmp, path))
    failed = [path for proc, _, path in procs if proc.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, f"nvcc for {failed}")
    for _, tmp, path in procs:
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
