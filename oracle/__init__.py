"""FP64 CPU oracle for the FP32 tiled matrix multiply -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (``dense_fp32_tiled_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``oracle_f64.c`` (plain C, FP64 accumulation in
increasing k); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  What each function follows is cited in the C file:
the textbook product C = A x B of the shared-memory/vectorised-load pages,
leading dimensions as row strides, and the bank page's
``bank = (byte_address / 4) % 32`` with its conflict/broadcast rules.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_f64.c")
_LIB = os.path.join(_HERE, "liboracle_f64.so")
_STAMP = _LIB + ".src-sha256"

_lib = None


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile oracle_f64.c into liboracle_f64.so (OpenMP, -O2, portable C)."""
    h = _src_hash()
    if not force and os.path.exists(_LIB) and os.path.exists(_STAMP):
        with open(_STAMP) as f:
            if f.read().strip() == h:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(_STAMP, "w") as f:
        f.write(h)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p]
        lib.oracle_gemm_f64.restype = ctypes.c_int
        lib.oracle_gemm_sampled_f64.argtypes = [i64, p, p, i64, i64, i64, p, i64, p, i64, p, p]
        lib.oracle_gemm_sampled_f64.restype = ctypes.c_int
        lib.oracle_bank_of.argtypes = [ctypes.c_uint64]
        lib.oracle_bank_of.restype = ctypes.c_int
        ip = ctypes.POINTER(ctypes.c_int)
        lib.oracle_shared_request.argtypes = [ctypes.c_int, p, p, ctypes.c_int, ip, ip, ip, ip]
        lib.oracle_shared_request.restype = ctypes.c_int
        lib.oracle_transpose_f32.argtypes = [i64, i64, p, i64, p, i64]
        lib.oracle_transpose_f32.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _storage(x: np.ndarray, rows: int, cols: int, ld: int | None):
    """Return (base array, ld) for a float32 matrix given either as a dense 2-D
    array or as a flat buffer with an explicit row stride ``ld``."""
    if ld is None:
        x = np.ascontiguousarray(x, dtype=np.float32)
        assert x.shape == (rows, cols), (x.shape, rows, cols)
        return x, max(1, cols)
    assert x.dtype == np.float32 and x.flags.c_contiguous
    need = 0 if rows == 0 or cols == 0 else (rows - 1) * ld + cols
    assert x.size >= need, (x.size, need)
    return x, ld


def num_threads() -> int:
    return _load().oracle_num_threads()


def gemm(A, B, M=None, N=None, K=None, lda=None, ldb=None, with_abs=True):
    """C = A.B in FP64 (and |A|.|B| when ``with_abs``).

    A, B are float32 arrays: dense 2-D (M x K, K x N), or flat buffers with
    explicit ``lda`` / ``ldb`` row strides and M, N, K given.  Returns (C, S)
    as dense float64 M x N arrays (S is None without ``with_abs``).
    """
    if M is None:
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
    A_, lda_ = _storage(A, M, K, lda)
    B_, ldb_ = _storage(B, K, N, ldb)
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64) if with_abs else None
    rc = _load().oracle_gemm_f64(M, N, K, _ptr(A_), lda_, _ptr(B_), ldb_,
                                 _ptr(C), max(1, N), _ptr(S))
    if rc != 0:
        raise ValueError(f"oracle_gemm_f64 rejected the arguments (rc={rc})")
    return C, S


def gemm_sampled(A, B, rows, cols, M=None, N=None, K=None, lda=None, ldb=None):
    """FP64 values (and |A|.|B| values) of C = A.B at the outputs (rows[t], cols[t])."""
    if M is None:
        M, K = A.shape
        _, N = B.shape
    A_, lda_ = _storage(A, M, K, lda)
    B_, ldb_ = _storage(B, K, N, ldb)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.zeros(r.size, dtype=np.float64)
    absout = np.zeros(r.size, dtype=np.float64)
    rc = _load().oracle_gemm_sampled_f64(r.size, _ptr(r), _ptr(c), M, N, K,
                                         _ptr(A_), lda_, _ptr(B_), ldb_,
                                         _ptr(out), _ptr(absout))
    if rc != 0:
        raise ValueError(f"oracle_gemm_sampled_f64 rejected the arguments (rc={rc})")
    return out, absout


def transpose(x, rows=None, cols=None, ld_in=None, ld_out=None, out=None):
    """out[j][i] = x[i][j] for a float32 matrix (dense 2-D, or a flat buffer with
    an explicit ld_in).  Returns a dense cols x rows array, or fills the flat
    buffer ``out`` with row stride ``ld_out``."""
    if rows is None:
        rows, cols = x.shape
    x_, ldi = _storage(x, rows, cols, ld_in)
    if out is None:
        res = np.zeros((cols, rows), dtype=np.float32)
        ldo = max(1, rows)
    else:
        res, ldo = out, ld_out
    rc = _load().oracle_transpose_f32(rows, cols, _ptr(x_), ldi, _ptr(res), ldo)
    if rc != 0:
        raise ValueError(f"oracle_transpose_f32 rejected the arguments (rc={rc})")
    return res


def bank_of(byte_address: int) -> int:
    """bank = (byte_address / 4) % 32."""
    return _load().oracle_bank_of(int(byte_address))


def shared_request(byte_addresses, width_bytes: int = 4, active=None) -> dict:
    """Bank analysis of one warp-wide shared-memory request (see oracle_f64.c)."""
    addr = np.ascontiguousarray(byte_addresses, dtype=np.uint64)
    act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
    w, i, d, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = _load().oracle_shared_request(addr.size, _ptr(addr), _ptr(act), width_bytes,
                                       ctypes.byref(w), ctypes.byref(i),
                                       ctypes.byref(d), ctypes.byref(n))
    if rc != 0:
        raise ValueError("oracle_shared_request rejected the request")
    return {"wavefronts": w.value, "ideal": i.value, "degree": d.value, "distinct": n.value}
