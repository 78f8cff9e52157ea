"""Builds libmemra.so in-tree from csrc/*.cu for sm_103a (nvcc, no cmake).

Each translation unit compiles in its own nvcc process, in parallel; the
shared library links the CUDA runtime statically, so it needs only the driver.

Staleness is decided by content, not by file times: a SHA-256 over the
sources, the headers, the public header, this file and the compiler flags is
written beside the library (libmemra.so.sha256), and the library is rebuilt
whenever the stamp is missing or differs.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(os.path.dirname(HERE), "_build")
LIB = os.path.join(HERE, "libmemra.so")
STAMP = LIB + ".sha256"

SOURCES = ["api.cu", "kv_append.cu", "combine.cu", "decode_d128.cu", "decode_d256.cu", "noalloc.cu", "cascade.cu"]
HEADERS = ["memra_device.cuh", "decode_kernel.cuh", "kv_quant.cuh", "cascade.cuh", "tcgen05.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmemra.so")
    return path


def source_hash() -> str:
    """SHA-256 (first 16 hex digits) of everything the library is built from."""
    h = hashlib.sha256()
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [__file__]
    files += [os.path.join(INCLUDE, f) for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h")]
    for f in files:
        h.update(os.path.basename(f).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS[:-1]).encode())
    return h.hexdigest()[:16]


def built_hash() -> str | None:
    """The source hash the present libmemra.so was built from (None if unstamped)."""
    try:
        with open(STAMP) as f:
            return f.read().strip() or None
    except FileNotFoundError:
        return None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (unless the library's stamp matches the sources) and return the path of libmemra.so."""
    want = source_hash()
    if not force and os.path.exists(LIB) and built_hash() == want:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP + ".tmp", "w") as f:
        f.write(want + "\n")
    os.replace(STAMP + ".tmp", STAMP)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
