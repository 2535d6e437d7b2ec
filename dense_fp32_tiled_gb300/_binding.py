"""ctypes binding of libsgemm_f32.so: argument marshalling only.

Every arithmetic step runs in the CUDA library.  PyTorch is used only for
device memory, strides and the current stream.  There is no fallback: if the
library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsgemm_f32.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "sgemm_f32.h")
HEADER_PATHS = [HEADER_PATH, os.path.join(os.path.dirname(_PKG), "include", "transpose_f32.h"),
                os.path.join(os.path.dirname(_PKG), "include", "smem_bank_probe.h")]

SGEMM_OK = 0
_lib = None


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str = "sgemm_f32"):
        self.status = status
        super().__init__(f"{what} failed with status {status}: {status_string(status)}")


def load_library():
    """Load libsgemm_f32.so from the package directory (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"CUDA library {LIB_PATH} is not built; run dense_fp32_tiled_gb300.build.build() "
            "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(LIB_PATH)
    i32, p, i64p = ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64)
    lib.sgemm_f32.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, p]
    lib.sgemm_f32.restype = i32
    lib.sgemm_f32_ws.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, p, ctypes.c_size_t, p]
    lib.sgemm_f32_ws.restype = i32
    lib.sgemm_f32_static_scratch.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, p]
    lib.sgemm_f32_static_scratch.restype = i32
    lib.sgemm_f32_3xtf32.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, p, ctypes.c_size_t, p]
    lib.sgemm_f32_3xtf32.restype = i32
    lib.sgemm_f32_3xtf32_workspace_size.argtypes = [i32, i32, i32]
    lib.sgemm_f32_3xtf32_workspace_size.restype = ctypes.c_size_t
    lib.sgemm_f32_3xtf32_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.sgemm_f32_3xtf32_timeouts.restype = i32
    lib.sgemm_f32_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.sgemm_f32_timeouts.restype = i32
    for name in ("sgemm_f32_wait_selftest", "sgemm_f32_3xtf32_wait_selftest"):
        getattr(lib, name).argtypes = [i32, ctypes.c_uint, ctypes.POINTER(ctypes.c_uint)]
        getattr(lib, name).restype = i32
    lib.sgemm_f32_host.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, p, ctypes.c_size_t, p]
    lib.sgemm_f32_host.restype = i32
    lib.sgemm_f32_host_workspace_size.argtypes = [i32, i32, i32]
    lib.sgemm_f32_host_workspace_size.restype = ctypes.c_size_t
    lib.sgemm_f32_ws_schedule.argtypes = [i32, i32, i32, p, i32, p, i32, p, i32, ctypes.c_size_t,
                                          ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_longlong)]
    lib.sgemm_f32_ws_schedule.restype = i32
    lib.sgemm_f32_workspace_size.argtypes = [i32, i32, i32]
    lib.sgemm_f32_workspace_size.restype = ctypes.c_size_t
    lib.sgemm_f32_workspace_size_for.argtypes = [i32, i32, i32, p, i32, p, i32]
    lib.sgemm_f32_workspace_size_for.restype = ctypes.c_size_t
    lib.sgemm_f32_status_string.argtypes = [i32]
    lib.sgemm_f32_status_string.restype = ctypes.c_char_p
    ip = ctypes.POINTER(ctypes.c_int)
    lib.transpose_f32.argtypes = [i32, i32, p, i32, p, i32, p]
    lib.transpose_f32.restype = i32
    lib.transpose_f32_layout.argtypes = [i32, i32, p, i32, p, i32, i32, p]
    lib.transpose_f32_layout.restype = i32
    lib.transpose_f32_smem_request.argtypes = [i32, i32, i32, i32, i64p, ip]
    lib.transpose_f32_smem_request.restype = i32
    lib.transpose_f32_status_string.argtypes = [i32]
    lib.transpose_f32_status_string.restype = ctypes.c_char_p
    lib.sgemm_f32_smem_shape.argtypes = [i32, ip, ip, ip]
    lib.sgemm_f32_smem_shape.restype = i32
    lib.sgemm_f32_smem_request.argtypes = [i32, i32, i32, i32, i64p, ip]
    lib.sgemm_f32_smem_request.restype = i32
    lib.smem_bank_stride_probe.argtypes = [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_longlong)]
    lib.smem_bank_stride_probe.restype = i32
    lib.smem_bank_pattern_probe.argtypes = [i32, ctypes.POINTER(ctypes.c_int), i32, i32,
                                            ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]
    lib.smem_bank_pattern_probe.restype = i32
    _lib = lib
    return lib


def declared_functions() -> list[str]:
    """Names of the functions the headers in include/ declare."""
    names = set()
    for path in HEADER_PATHS:
        with open(path) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        names |= set(re.findall(r"\b((?:sgemm|transpose)_f32\w*|smem_bank_\w+)\s*\(", text))
    return sorted(names)


def status_string(status: int) -> str:
    return load_library().sgemm_f32_status_string(int(status)).decode()


def sgemm_f32(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
              stream: int = 0) -> int:
    """Raw C-ABI call with integer device addresses; returns the status code."""
    return load_library().sgemm_f32(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None), int(lda),
                                    ctypes.c_void_p(int(B) or None), int(ldb),
                                    ctypes.c_void_p(int(C) or None), int(ldc),
                                    ctypes.c_void_p(int(stream) or None))


def sgemm_f32_ws(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                 workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Raw C-ABI call of the workspace variant; returns the status code."""
    return load_library().sgemm_f32_ws(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None), int(lda),
                                       ctypes.c_void_p(int(B) or None), int(ldb),
                                       ctypes.c_void_p(int(C) or None), int(ldc),
                                       ctypes.c_void_p(int(workspace) or None), int(workspace_bytes),
                                       ctypes.c_void_p(int(stream) or None))


def sgemm_f32_static_scratch(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                             stream: int = 0) -> int:
    """Raw C-ABI call of the allocation-free entry point (its scratch is a fixed
    array inside the library); returns the status code."""
    return load_library().sgemm_f32_static_scratch(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None),
                                                   int(lda), ctypes.c_void_p(int(B) or None), int(ldb),
                                                   ctypes.c_void_p(int(C) or None), int(ldc),
                                                   ctypes.c_void_p(int(stream) or None))


def sgemm_f32_3xtf32(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                     workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Raw C-ABI call of the tensor-core (3xTF32) variant; returns the status code."""
    return load_library().sgemm_f32_3xtf32(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None), int(lda),
                                           ctypes.c_void_p(int(B) or None), int(ldb),
                                           ctypes.c_void_p(int(C) or None), int(ldc),
                                           ctypes.c_void_p(int(workspace) or None), int(workspace_bytes),
                                           ctypes.c_void_p(int(stream) or None))


def sgemm_f32_host(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                   workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Raw C-ABI call for HOST operands (device workspace); returns the status code."""
    return load_library().sgemm_f32_host(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None), int(lda),
                                         ctypes.c_void_p(int(B) or None), int(ldb),
                                         ctypes.c_void_p(int(C) or None), int(ldc),
                                         ctypes.c_void_p(int(workspace) or None), int(workspace_bytes),
                                         ctypes.c_void_p(int(stream) or None))


def host_workspace_size(M: int, N: int, K: int) -> int:
    return int(load_library().sgemm_f32_host_workspace_size(int(M), int(N), int(K)))


def _host_matrix_args(t, rows: int, cols: int, name: str):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.is_cuda:
        raise TypeError(f"{name} must be a CPU float32 tensor")
    if t.dim() != 2 or tuple(t.shape) != (rows, cols):
        raise ValueError(f"{name} must have shape ({rows}, {cols}), got {tuple(t.shape)}")
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with unit column stride")
    ld = t.stride(0) if rows > 1 else max(1, cols)
    return t.data_ptr(), max(ld, cols, 1)


def sgemm_host(A, B, out=None, device=None, stream=None):
    """C = A @ B for CPU float32 tensors through sgemm_f32_host (copies in,
    product on the GPU, copy back).  Pinned tensors give asynchronous copies;
    the call synchronises the stream before returning, so `out` is ready."""
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch: {tuple(A.shape)} @ {tuple(B.shape)}")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=A.is_pinned())
    a, lda = _host_matrix_args(A, M, K, "A")
    b, ldb = _host_matrix_args(B, K, N, "B")
    c, ldc = _host_matrix_args(out, M, N, "out")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st_obj = stream or torch.cuda.current_stream(dev)
        nbytes = host_workspace_size(M, N, K)
        ws = _workspace("host", dev, st_obj, nbytes)
        st = sgemm_f32_host(M, N, K, a, lda, b, ldb, c, ldc, ws.data_ptr(), nbytes, st_obj.cuda_stream)
        if st != SGEMM_OK:
            raise SgemmError(st, "sgemm_f32_host")
        st_obj.synchronize()
    return out


def tc_workspace_size(M: int, N: int, K: int) -> int:
    return int(load_library().sgemm_f32_3xtf32_workspace_size(int(M), int(N), int(K)))


def tc_timeouts() -> int:
    n = ctypes.c_uint()
    st = load_library().sgemm_f32_3xtf32_timeouts(ctypes.byref(n))
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_f32_3xtf32_timeouts")
    return n.value


def copy_timeouts() -> int:
    """Flag of sgemm_f32_timeouts: 1 if a CUDA-core kernel gave up a copy wait."""
    n = ctypes.c_uint()
    st = load_library().sgemm_f32_timeouts(ctypes.byref(n))
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_f32_timeouts")
    return n.value


WAIT_SELFTESTS = {"copy_never": ("sgemm_f32_wait_selftest", 0), "flag_never": ("sgemm_f32_wait_selftest", 1),
                  "copy_done": ("sgemm_f32_wait_selftest", 2), "flag_done": ("sgemm_f32_wait_selftest", 3),
                  "tc_never": ("sgemm_f32_3xtf32_wait_selftest", 0), "tc_done": ("sgemm_f32_3xtf32_wait_selftest", 1)}


def wait_selftest(case: str, polls: int = 1000) -> bool:
    """Runs one bounded-wait self-test (WAIT_SELFTESTS); True if the wait gave up."""
    fn, which = WAIT_SELFTESTS[case]
    n = ctypes.c_uint(7)
    st = getattr(load_library(), fn)(which, int(polls), ctypes.byref(n))
    if st != SGEMM_OK:
        raise SgemmError(st, fn)
    assert n.value in (0, 1)
    return n.value == 1


def sgemm_tc(A, B, out=None, stream=None):
    """C = A @ B through the tensor-core 3xTF32 variant (same FP32 tolerance,
    not bit-identical to sgemm); the workspace is cached per device and stream."""
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch: {tuple(A.shape)} @ {tuple(B.shape)}")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    a, lda = _matrix_args(A, M, K, "A")
    b, ldb = _matrix_args(B, K, N, "B")
    c, ldc = _matrix_args(out, M, N, "out")
    nbytes = tc_workspace_size(M, N, K)
    st_obj = stream or torch.cuda.current_stream(A.device)
    with torch.cuda.device(A.device):
        ws = _workspace("tc", A.device, st_obj, nbytes)
        st = sgemm_f32_3xtf32(M, N, K, a, lda, b, ldb, c, ldc, ws.data_ptr(), max(nbytes, 256),
                              st_obj.cuda_stream)
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_f32_3xtf32")
    return out


def ws_schedule(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                workspace_bytes: int = None):
    """(status, kind, words): what sgemm_f32_ws runs for these arguments with a
    workspace of `workspace_bytes` (default: workspace_size_for these
    operands; 0 gives what sgemm_f32 runs): kind = schedule (bits 0-1) + 4 if
    A is repacked + 8 if B is + 16 if A is transposed into its k-major copy
    + 32 for the cluster split of K, with its cluster size in bits 8-12;
    words = the leading workspace words it zero-fills and leaves zero."""
    if workspace_bytes is None:
        workspace_bytes = workspace_size_for(M, N, K, A, lda, B, ldb)
    kind, words = ctypes.c_int(), ctypes.c_longlong()
    st = load_library().sgemm_f32_ws_schedule(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None), int(lda),
                                              ctypes.c_void_p(int(B) or None), int(ldb),
                                              ctypes.c_void_p(int(C) or None), int(ldc), int(workspace_bytes),
                                              ctypes.byref(kind), ctypes.byref(words))
    return st, kind.value, words.value


def workspace_size(M: int, N: int, K: int) -> int:
    return int(load_library().sgemm_f32_workspace_size(int(M), int(N), int(K)))


def workspace_size_for(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int) -> int:
    """Workspace bytes for these operands, room for the operand copies that pay
    (the k-major copy of A, repacked unaligned rows) included."""
    return int(load_library().sgemm_f32_workspace_size_for(int(M), int(N), int(K), ctypes.c_void_p(int(A) or None),
                                                           int(lda), ctypes.c_void_p(int(B) or None), int(ldb)))


def smem_shape(kind: int):
    nw, ns, nst = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = load_library().sgemm_f32_smem_shape(kind, ctypes.byref(nw), ctypes.byref(ns), ctypes.byref(nst))
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_f32_smem_shape")
    return nw.value, ns.value, nst.value


def smem_request(kind: int, warp: int, step: int, stage: int = 0):
    """(byte offsets of the 32 lanes, width in bytes) of one shared-memory access."""
    out = (ctypes.c_int64 * 32)()
    width = ctypes.c_int()
    st = load_library().sgemm_f32_smem_request(kind, warp, step, stage, out, ctypes.byref(width))
    if st != SGEMM_OK:
        raise SgemmError(st, "sgemm_f32_smem_request")
    return list(out), width.value


def _matrix_args(t, rows: int, cols: int, name: str):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if t.dim() != 2 or tuple(t.shape) != (rows, cols):
        raise ValueError(f"{name} must have shape ({rows}, {cols}), got {tuple(t.shape)}")
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with unit column stride")
    ld = t.stride(0) if rows > 1 else max(1, cols)
    return t.data_ptr(), max(ld, cols, 1)


_workspaces = {}


def _workspace(kind: str, device, stream, nbytes: int):
    """Scratch for one entry point on one stream of one device (torch memory,
    grown on demand).  Calls on one stream are ordered, so they can share it;
    calls on different streams get different buffers.  record_stream keeps
    torch from handing the memory out again while work queued on `stream`
    may still use it."""
    import torch
    key = (kind, torch.device(device), stream.cuda_stream)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 12), dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    buf.record_stream(stream)
    return buf


def sgemm(A, B, out=None, stream=None, balanced=True):
    """C = A @ B for CUDA float32 tensors (row-major, any row stride) via the C ABI.

    ``out`` (M x N, row-major) is written when given, else allocated.  Runs on
    ``stream`` (a torch.cuda.Stream) or the current stream; asynchronous.
    With ``balanced`` (default) the call goes through sgemm_f32_ws with a
    workspace cached per device and stream, which enables the balanced
    schedules and the repacking of unaligned rows; otherwise through
    sgemm_f32.
    """
    import torch
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch: {tuple(A.shape)} @ {tuple(B.shape)}")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    a, lda = _matrix_args(A, M, K, "A")
    b, ldb = _matrix_args(B, K, N, "B")
    c, ldc = _matrix_args(out, M, N, "out")
    st_obj = stream or torch.cuda.current_stream(A.device)
    s = st_obj.cuda_stream
    with torch.cuda.device(A.device):
        if balanced:
            # exactly the size asked for (not the cached buffer's), so the
            # schedule, and with it the summation order, depends only on the call
            nbytes = workspace_size_for(M, N, K, a, lda, b, ldb)
            ws = _workspace("ws", A.device, st_obj, nbytes) if nbytes else None
            st = sgemm_f32_ws(M, N, K, a, lda, b, ldb, c, ldc, ws.data_ptr() if ws is not None else 0,
                              nbytes if ws is not None else 0, s)
        else:
            st = sgemm_f32(M, N, K, a, lda, b, ldb, c, ldc, s)
    if st != SGEMM_OK:
        raise SgemmError(st)
    return out


# ---- transpose ------------------------------------------------------------
TRANSPOSE_LAYOUTS = {"padded": 0, "unpadded": 1, "swizzled": 2, "fast": 3, "fast_vec": 4}


def transpose_f32(rows: int, cols: int, inp: int, ld_in: int, out: int, ld_out: int, stream: int = 0,
                  layout: str | None = None) -> int:
    """Raw C-ABI call (transpose_f32, or transpose_f32_layout with a layout name)."""
    lib = load_library()
    args = (int(rows), int(cols), ctypes.c_void_p(int(inp) or None), int(ld_in),
            ctypes.c_void_p(int(out) or None), int(ld_out))
    if layout is None:
        return lib.transpose_f32(*args, ctypes.c_void_p(int(stream) or None))
    return lib.transpose_f32_layout(*args, TRANSPOSE_LAYOUTS[layout], ctypes.c_void_p(int(stream) or None))


def transpose_status_string(status: int) -> str:
    return load_library().transpose_f32_status_string(int(status)).decode()


def transpose_smem_request(layout: str, kind: int, warp: int, step: int):
    out = (ctypes.c_int64 * 32)()
    width = ctypes.c_int()
    st = load_library().transpose_f32_smem_request(TRANSPOSE_LAYOUTS[layout], kind, warp, step, out,
                                                   ctypes.byref(width))
    if st != 0:
        raise ValueError(f"transpose_f32_smem_request rejected ({st})")
    return list(out), width.value


def transpose(x, out=None, stream=None):
    """x.T for a CUDA float32 tensor (row-major, any row stride) via transpose_f32."""
    import torch
    if x.dim() != 2:
        raise ValueError("transpose expects a 2-D tensor")
    rows, cols = x.shape
    if out is None:
        out = torch.empty((cols, rows), dtype=torch.float32, device=x.device)
    a, lda = _matrix_args(x, rows, cols, "x")
    b, ldb = _matrix_args(out, cols, rows, "out")
    s = (stream or torch.cuda.current_stream(x.device)).cuda_stream
    with torch.cuda.device(x.device):
        st = transpose_f32(rows, cols, a, lda, b, ldb, s)
    if st != 0:
        raise RuntimeError(f"transpose_f32 failed with status {st}: {transpose_status_string(st)}")
    return out


# ---- shared-memory stride sweep ---------------------------------------------
def bank_stride_probe(stride: int, op: str = "load", warps: int = 8, iters: int = 4096):
    """(cycles per warp-wide access, checksum) of smem_bank_stride_probe."""
    cyc, chk = ctypes.c_double(), ctypes.c_longlong()
    st = load_library().smem_bank_stride_probe(int(stride), {"load": 0, "store": 1}[op], int(warps), int(iters),
                                               ctypes.byref(cyc), ctypes.byref(chk))
    if st != 0:
        raise RuntimeError(f"smem_bank_stride_probe failed with status {st}")
    return cyc.value, chk.value


def bank_pattern_probe(width_bytes: int, lane_word, warps: int = 8, iters: int = 4096):
    """(cycles per warp-wide load, checksum) of smem_bank_pattern_probe for the
    32 word offsets ``lane_word``."""
    arr = (ctypes.c_int * 32)(*[int(x) for x in lane_word])
    cyc, chk = ctypes.c_double(), ctypes.c_longlong()
    st = load_library().smem_bank_pattern_probe(int(width_bytes), arr, int(warps), int(iters), ctypes.byref(cyc),
                                                ctypes.byref(chk))
    if st != 0:
        raise RuntimeError(f"smem_bank_pattern_probe failed with status {st}")
    return cyc.value, chk.value
