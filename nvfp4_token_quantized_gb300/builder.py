"""Build the sm_103a CUDA library in-tree.

Compiles every ``csrc/*.cu`` translation unit with nvcc (in parallel, one
``-gencode`` for sm_103a) and links them into
``nvfp4_token_quantized_gb300/_lib/libmoe_nvfp4.so``.  The CUDA runtime is
linked statically; the GEMM operands move by plain bulk copies, and the one
tensor map (the small-batch front kernel's router-weight ring) is encoded
through the runtime's driver entry point, so the library needs no link
against libcuda.  Works the same on x86_64 and aarch64 hosts (no
host-architecture flags).
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
LIB_DIR = os.path.join(PKG_DIR, "_lib")
LIB_NAME = "libmoe_nvfp4.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)

GENCODE = "arch=compute_103a,code=sm_103a"
NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo", f"-gencode={GENCODE}",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
]


def _nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _fingerprint() -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)) + ["../../include/moe_nvfp4.h"]:
        path = os.path.normpath(os.path.join(CSRC, f))
        if os.path.isfile(path):
            with open(path, "rb") as fh:
                h.update(f.encode() + fh.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if its sources changed; return the .so path."""
    os.makedirs(LIB_DIR, exist_ok=True)
    stamp = os.path.join(LIB_DIR, "build.stamp")
    fp = _fingerprint()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == fp:
                return LIB_PATH
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(LIB_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, "-shared", f"-gencode={GENCODE}", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    for o in objs:
        os.remove(o)
    with open(stamp, "w") as fh:
        fh.write(fp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
