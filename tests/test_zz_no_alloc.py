"""The allocation-free entry point, sgemm_f32_static_scratch (needs a GB300).

Some callers cannot call cudaMalloc: their device memory belongs to another
allocator, or they must not risk the device-wide synchronisation a cudaFree
can bring.  For them the library offers one entry point whose scratch (the
per-tile flags of the balanced schedule) is a fixed array inside the library
instead of a caller-provided workspace.  Here its result is compared, through
the C ABI, with the FP64 oracle on the same inputs (the FP32 acceptance bound
of every other parity test), and with the workspace entry point sgemm_f32_ws,
on two calls in a row: the array keeps the previous call's contents, so the
second call checks that each call clears what it needs.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
from tests import _tolerance as tol

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = -8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("M,N,K", [(2500, 2100, 333), (1000, 1030, 777)])
def test_static_scratch_matches_oracle(oracle_lib, M, N, K):
    # 2500 x 2100 has 340 output tiles (more than two per SM, not a multiple of
    # the resident CTAs: the balanced schedule and its flags are used);
    # 1000 x 1030 has 72 (one CTA per tile: the scratch is not needed)
    A = synth.matrix(M, K, 41, 0)
    B = synth.matrix(K, N, 41, 1)
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    Cr, Sr = oracle_lib.gemm(A, B)
    C_ws = torch.empty(M, N, device="cuda")
    ws = torch.zeros(sg.workspace_size(M, N, K) // 4, dtype=torch.int32, device="cuda")
    assert sg.sgemm_f32_ws(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, C_ws.data_ptr(), N,
                           ws.data_ptr(), ws.numel() * 4, _stream()) == 0
    for call in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        st = sg.sgemm_f32_static_scratch(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, C.data_ptr(), N,
                                         _stream())
        torch.cuda.synchronize()
        assert st == 0, sg.status_string(st)
        Ch = C.cpu().numpy()
        tol.assert_close(Ch, Cr, Sr, K, f"static scratch vs oracle, call {call + 1}")
        # the same product as the workspace entry point, within the same bound
        tol.assert_close(Ch, C_ws.cpu().numpy().astype(np.float64), Sr, K,
                         f"static scratch vs sgemm_f32_ws, call {call + 1}")


def test_static_scratch_integer_inputs_bit_exact(oracle_lib):
    # integer-valued inputs: every partial sum is exact in FP32, so the result
    # must equal the oracle bit for bit whatever the split of K
    M, N, K = 2500, 2100, 333
    A = synth.matrix(M, K, 42, 0, "int5")
    B = synth.matrix(K, N, 42, 1, "int5")
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    Cr, _ = oracle_lib.gemm(A, B)
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        assert sg.sgemm_f32_static_scratch(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, C.data_ptr(), N,
                                           _stream()) == 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), Cr)


def test_static_scratch_rejects_problems_beyond_its_limit():
    # 129 x 129 = 16641 output tiles > 16383: rejected on the host, nothing launched
    M = N = 129 * 128
    FAKE = 1 << 20  # never dereferenced
    st = sg.sgemm_f32_static_scratch(M, N, 8, FAKE, 8, FAKE * 64, N, FAKE * 4096, N, 0)
    assert st == SCRATCH_LIMIT
    assert "16383" in sg.status_string(st)
