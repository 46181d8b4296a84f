"""In-tree build of libkvp.so (nvcc, sm_103a only).

Each translation unit is compiled in parallel to an object under ``_build/``
and linked with ``nvcc -shared`` into ``_lib/libkvp.so``; an object is rebuilt
when it is older than its source or any header.  No cmake, no ninja.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libkvp.so")

SOURCES = [
    "kvp_api.cu",
    "kvp_append.cu",
    "kvp_decode_simt.cu",
    "kvp_decode_mma.cu",
    "kvp_decode_int8.cu",
    "kvp_decode_fp8.cu",
    "kvp_decode_fp8_umma.cu",
    "kvp_reduce.cu",
    "kvp_prefill.cu",
    "kvp_block_manager.cpp",
    "kvp_noalloc.cu",
    "kvp_selftest.cu",
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    hs += glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    s = os.path.join(CSRC, src)
    o = os.path.join(BUILD_DIR, src + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-c", s, "-o", o]
    if ptxas_verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return o, r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (incrementally) and link libkvp.so; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    hdr = _headers_mtime()
    todo = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src + ".o")
        objs.append(o)
        if force or ptxas_verbose or not os.path.exists(o) or \
                os.path.getmtime(o) < max(os.path.getmtime(s), hdr):
            todo.append(src)
    logs = []
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(len(todo), os.cpu_count() or 4)) as ex:
            for _, log in ex.map(lambda f: _compile(f, ptxas_verbose), todo):
                logs.append(log)
    if todo or force or not os.path.exists(LIB_PATH) or \
            os.path.getmtime(LIB_PATH) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp, "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_PATH)
    if verbose or ptxas_verbose:
        for log in logs:
            if log.strip():
                print(log)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv)
    print(LIB_PATH)
