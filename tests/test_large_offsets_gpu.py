"""Element offsets past 2**31 in A, B and C (needs a GB300 and about 27 GB of
free device memory).

A, B and C are narrow views into buffers with very wide rows, so that the
last rows of each start more than 2**31 floats into their buffer: every
address computation on the path (copies, tensor maps, stores, the split
pass of the 3xTF32 variant) must be 64-bit.  The padding is NaN, so a read of
it would show in the result.  Rows on both sides of the 2**31 boundary are
checked against the FP64 oracle; the CUDA-core result must equal the oracle
exactly for integer inputs, with and without the k-major copy of A.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from tests import _tolerance as tol

pytestmark = pytest.mark.gpu

M, N, K = 33000, 384, 256
LDA = LDC = 1 << 16          # row 32768 of A and C starts at 2**31
LDB = (1 << 23) + (1 << 16)  # row 255 of B starts past 2**31


@pytest.fixture(scope="module")
def big():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()
    free, _ = torch.cuda.mem_get_info()
    need = 4 * (M * LDA + K * LDB + M * LDC) + (2 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.1f} GiB free on the device")
    g = torch.Generator(device="cuda")
    g.manual_seed(71)
    A_buf = torch.full((M, LDA), float("nan"), device="cuda")
    B_buf = torch.full((K, LDB), float("nan"), device="cuda")
    A = A_buf[:, :K]
    B = B_buf[:, :N]
    A.copy_(torch.randint(-2, 3, (M, K), generator=g, device="cuda").float())
    B.copy_(torch.randint(-2, 3, (K, N), generator=g, device="cuda").float())
    assert A.stride(0) * (M - 1) >= 2 ** 31 and B.stride(0) * (K - 1) >= 2 ** 31
    yield A, B
    del A_buf, B_buf


def _rows():
    return np.array([0, 1, 127, 128, 16383, 32767, 32768, 32769, 32895, 32896, M - 2, M - 1])


def _check_rows(oracle_lib, A, B, C, exact, what):
    rows = _rows()
    Ah = A[torch.from_numpy(rows).cuda()].cpu().numpy()
    Bh = B.cpu().numpy()
    Cr, Sr = oracle_lib.gemm(np.ascontiguousarray(Ah), np.ascontiguousarray(Bh))
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    if exact:
        np.testing.assert_array_equal(got.astype(np.float64), Cr)
    else:
        tol.assert_close(got, Cr, Sr, K, what)


def test_cuda_core_path_past_2_31(oracle_lib, big):
    A, B = big
    C_buf = torch.full((M, LDC), -3.0, device="cuda")
    C = C_buf[:, :N]
    sg.sgemm(A, B, out=C)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, A, B, C, True, "cuda-core")
    assert torch.all(C_buf[M - 1, N:N + 64] == -3.0)  # the padding of the last row is left alone
    del C_buf


def test_kmajor_copy_past_2_31(oracle_lib, big):
    """The same A placed 4 bytes off 16-byte alignment, so that sgemm_f32_ws
    transposes it into its k-major copy first; its last rows still start past
    2**31 floats into their buffer."""
    A, B = big
    free, _ = torch.cuda.mem_get_info()
    if free < 8 * M * LDA + (2 << 30):
        pytest.skip("needs room for a second A buffer and C")
    A2_buf = torch.full((M, LDA), float("nan"), device="cuda")
    A2 = A2_buf[:, 1:K + 1]
    A2.copy_(A)
    C_buf = torch.full((M, LDC), -3.0, device="cuda")
    C = C_buf[:, :N]
    nbytes = sg.workspace_size_for(M, N, K, A2.data_ptr(), LDA, B.data_ptr(), LDB)
    sst, kind, _ = sg.ws_schedule(M, N, K, A2.data_ptr(), LDA, B.data_ptr(), LDB, C.data_ptr(), LDC, nbytes)
    assert sst == 0 and kind & 16, kind
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert sg.sgemm_f32_ws(M, N, K, A2.data_ptr(), LDA, B.data_ptr(), LDB, C.data_ptr(), LDC, ws.data_ptr(), nbytes,
                           torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    _check_rows(oracle_lib, A, B, C, True, "k-major copy")
    assert torch.all(C_buf[M - 1, N:N + 64] == -3.0)
    del A2_buf, C_buf, ws


def test_tensor_core_path_past_2_31(oracle_lib, big):
    A, B = big
    C_buf = torch.full((M, LDC), -3.0, device="cuda")
    C = C_buf[:, :N]
    sg.sgemm_tc(A, B, out=C)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, A, B, C, True, "3xTF32")  # integer inputs split exactly
    assert torch.all(C_buf[M - 1, N:N + 64] == -3.0)
    del C_buf
