"""Build step for the CUDA library libsgemm_f32.so (sm_103a only).

Compiles every csrc/*.cu to an object file, all in parallel (one nvcc
process each), and links them into the package directory (in-tree, so the
library that runs is the one built from this checkout).  A stamp of the
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
# flags that shape the generated code (hashed into the stamps; no paths, so a
# checkout in another directory has the same stamps)
CODEGEN = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v", "-Xcompiler", "-fPIC"]
FLAGS = CODEGEN + [f"-I{INCLUDE}", f"-I{CSRC}"]


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
    """Hash of the named csrc files and the code-generation flags: identifies
    one kernel's code, so a profile taken on it can be matched to the build
    on any machine."""
    h = hashlib.sha256()
    for n in sorted(names):
        h.update(n.encode())
        with open(os.path.join(CSRC, n), "rb") as f:
            h.update(f.read())
    h.update(" ".join(CODEGEN).encode())
    return h.hexdigest()


def build(force: bool = False, quiet: bool = True) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    stamp_file = os.path.join(BUILD_DIR, "libsgemm_f32.stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB
    pid = os.getpid()
    tmp = os.path.join(BUILD_DIR, f"libsgemm_f32.{pid}.so")
    cus = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(BUILD_DIR, f"{os.path.basename(cu)[:-3]}.{pid}.o") for cu in cus]
    cmds = [[_nvcc(), *FLAGS, "-c", cu, "-o", obj] for cu, obj in zip(cus, objs)]
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for c in cmds]
    outs = [p.communicate() for p in procs]
    link = [_nvcc(), *ARCH, "-shared", *objs, "-o", tmp, "-ldl"]  # NVTX3 loads a profiler's hooks with dlopen
    log = ["\n".join([" ".join(c), o + e]) for c, (o, e) in zip(cmds, outs)]
    failed = any(p.returncode != 0 for p in procs)
    if not failed:
        r = subprocess.run(link, capture_output=True, text=True)
        log.append(" ".join(link) + "\n" + r.stdout + r.stderr)
        failed = r.returncode != 0
    for obj in objs:
        if os.path.exists(obj):
            os.remove(obj)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    if failed:
        sys.stderr.write("\n".join(log))
        raise RuntimeError("nvcc failed building libsgemm_f32.so")
    if not quiet:
        sys.stdout.write("\n".join(e for _, e in outs))
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))
