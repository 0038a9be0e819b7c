"""In-tree build of libswiglu.so (nvcc, sm_103a only, no cmake).

Each CUDA translation unit is compiled in parallel into ``_build/`` beside this
file, then linked into ``libswiglu.so`` in this package directory with the
CUDA runtime linked statically and only the ``swiglu_*`` symbols exported. A
stamp of the sources and flags skips the work when nothing changed.

    python -m swiglu_gated_mlp_gb300.build        # build (or check) the library
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libswiglu.so")
STAMP = os.path.join(BUILD_DIR, "libswiglu.stamp")

SOURCES = ["swiglu_api.cu", "pack.cu", "fused_large_m.cu", "fused_large_m_pair.cu", "fused_small_m.cu",
           "fused_sequential.cu", "fused_split_k.cu", "fused_resident_pair.cu"]
HEADERS = ["kernels.h", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                 "-Xptxas", "-v", "-I" + INCLUDE, "-I" + CSRC]
VERSION_SCRIPT = "{ global: swiglu_*; local: *; };\n"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libswiglu")


def _stamp(nvcc: str) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "swiglu.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(CFLAGS).encode())
    h.update(subprocess.run([nvcc, "--version"], capture_output=True, text=True).stdout.encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libswiglu.so if it is missing or stale; return its path."""
    nvcc = _nvcc()
    stamp = _stamp(nvcc)
    if not force and os.path.exists(LIB_PATH) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == stamp:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(name: str):
        obj = os.path.join(BUILD_DIR, name.replace(".cu", ".o"))
        cmd = [nvcc, "-c", os.path.join(CSRC, name), "-o", obj] + CFLAGS
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for name, _, r in results:
        log.append(f"==== {name}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}{r.stderr}")
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    vs = os.path.join(BUILD_DIR, "exports.map")
    with open(vs, "w") as f:
        f.write(VERSION_SCRIPT)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + [o for _, o, _ in results] + ARCH + [
        "--cudart", "static", "-Xlinker", "--version-script=" + vs, "-Xlinker", "-z,defs",
        "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(STAMP, "w") as f:
        f.write(stamp + "\n")
    if verbose:
        print("\n".join(log))
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
