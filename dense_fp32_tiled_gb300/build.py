"""Build step for the CUDA library libsgemm_f32.so (sm_103a only).

Compiles every csrc/*.cu with one nvcc call into the package directory
(in-tree, so the library that runs is the one built from this checkout).  A stamp of the
source hash and flags skips the compile when nothing changed.  The ptxas
report (registers, spills, shared memory) is kept in _build/ptxas.log.
"""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libsgemm_f32.so")
BUILD_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v", "-Xcompiler", "-fPIC",
                "-shared", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stamp() -> str:
    h = hashlib.sha256()
    for p in _sources():
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    return h.hexdigest()


def kernel_stamp(names) -> str:
    """Hash of the named csrc files and the compile flags: identifies one
    kernel's code, so a profile taken on it can be matched to the build."""
    h = hashlib.sha256()
    for n in sorted(names):
        h.update(n.encode())
        with open(os.path.join(CSRC, n), "rb") as f:
            h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, quiet: bool = True) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp_file = os.path.join(BUILD_DIR, "libsgemm_f32.stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB
    tmp = os.path.join(BUILD_DIR, f"libsgemm_f32.{os.getpid()}.so")
    cus = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cmd = [_nvcc(), *FLAGS, *cus, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libsgemm_f32.so")
    if not quiet:
        sys.stdout.write(r.stderr)
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))
