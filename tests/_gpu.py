"""Helpers for GPU tests: upload seeded inputs, run sgemm_f32 through the C ABI."""
import numpy as np
import torch

import dense_fp32_tiled_gb300 as sg


def dev_buffer(x: np.ndarray, offset_elems: int = 0, fill: float = 0.0):
    """Device copy of flat float32 data placed `offset_elems` floats into a
    fresh allocation (to create 4- or 8-byte aligned base pointers)."""
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    t = torch.full((flat.size + offset_elems + 4,), fill, dtype=torch.float32, device="cuda")
    t[offset_elems:offset_elems + flat.size] = torch.from_numpy(flat).cuda()
    return t, t.data_ptr() + 4 * offset_elems


def run(M, N, K, A, lda, B, ldb, ldc=None, a_off=0, b_off=0, c_off=0, c_fill=np.nan, stream=None):
    """Run C = A.B on the GPU; A, B are flat (or 2-D dense) float32 host arrays.
    Returns (status, C as a (M, ldc)-strided host array view [M x N], raw C buffer)."""
    ldc = ldc or max(1, N)
    tA, pA = dev_buffer(A, a_off) if A is not None and np.size(A) else (None, 0)
    tB, pB = dev_buffer(B, b_off) if B is not None and np.size(B) else (None, 0)
    c_elems = 0 if M == 0 or N == 0 else (M - 1) * ldc + N
    tC = torch.full((c_elems + c_off + 4,), c_fill, dtype=torch.float32, device="cuda")
    pC = tC.data_ptr() + 4 * c_off
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    st = sg.sgemm_f32(M, N, K, pA, lda, pB, ldb, pC, ldc, s)
    torch.cuda.synchronize()
    raw = tC.cpu().numpy()[c_off:c_off + c_elems]
    if M == 0 or N == 0:
        return st, np.zeros((M, N), np.float32), raw
    C = np.stack([raw[i * ldc:i * ldc + N] for i in range(M)]) if ldc != N else raw.reshape(M, N)
    return st, C, raw
