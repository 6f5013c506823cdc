"""Builds libpa.so (the sm_103a kernels and the C ABI) in-tree with nvcc.

Each .cu translation unit compiles in parallel to an object under ``_build/``; the objects
link into ``paged_kv_cache_238_gb300/libpa.so`` with the CUDA runtime linked statically and
its symbols hidden, so the library does not bind to another copy of the runtime that a host
process (e.g. PyTorch) may have loaded. A stamp of the sources and flags skips rebuilds.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
# PA_SANITIZE=address,undefined (any -fsanitize list) builds the host code with gcc's
# sanitizers into libpa_san.so instead, under _build_san/; run the process with the sanitizer
# runtimes preloaded (LD_PRELOAD of libasan.so and libubsan.so).
SANITIZE = os.environ.get("PA_SANITIZE", "").strip()
if SANITIZE:
    BUILD = os.path.join(HERE, "_build_san")
    LIB = os.path.join(HERE, "libpa_san.so")
else:
    LIB = os.path.join(HERE, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# (nvcc's -Xcompiler splits at commas: one -fsanitize= per sanitizer)
_SAN = ",".join(f"-fsanitize={x.strip()}" for x in SANITIZE.split(",") if x.strip())
_HOST = "-fPIC,-fvisibility=hidden" + (f",{_SAN},-fno-omit-frame-pointer,-g" if SANITIZE else "")
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", _HOST,
                     "--expt-relaxed-constexpr", "-I", INCLUDE]
LINK_FLAGS = ARCH + ["-shared", "-Xlinker", "--exclude-libs,ALL", "-Xlinker", "-Bsymbolic"] + (
    ["-Xcompiler", _SAN] if SANITIZE else [])


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa")


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    deps = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    return cu, deps


def _stamp(extra_flags) -> str:
    cu, deps = _sources()
    h = hashlib.sha256()
    for f in cu + deps:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    with open(os.path.join(INCLUDE, "pa.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + LINK_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile libpa.so if its sources changed; returns its path."""
    stamp_file = os.path.join(BUILD, "stamp")
    stamp = _stamp(extra_flags)
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as fh:
            if fh.read().strip() == stamp:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = nvcc_path()
    cu, _ = _sources()

    def compile_one(name):
        obj = os.path.join(BUILD, name.rsplit(".", 1)[0] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + list(extra_flags) + ["-c", os.path.join(CSRC, name), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(cu))) as ex:
        objs = list(ex.map(compile_one, cu))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc] + LINK_FLAGS + objs + ["-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else ()))
