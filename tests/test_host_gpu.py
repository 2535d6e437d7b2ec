"""sgemm_f32_host: operands in host memory (copies overlapped with the
product in row panels) vs the FP64 oracle (needs a GB300)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
from tests import _tolerance as tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


def test_pageable_strided_ragged(oracle_lib):
    """Pageable host views with row strides wider than the rows."""
    base_a = synth.matrix(1000, 800, 91, 0)
    base_b = synth.matrix(777, 1100, 91, 1)
    A = torch.from_numpy(base_a)[:, :777]
    B = torch.from_numpy(base_b)[:, 3:1033]
    out = torch.full((1000, 1040), -5.0)
    sg.sgemm_host(A, B, out=out[:, 4:1034])
    Cr, Sr = oracle_lib.gemm(A.numpy(), B.numpy())
    tol.assert_close(out[:, 4:1034].numpy(), Cr, Sr, 777, "host strided")
    assert torch.all(out[:, :4] == -5.0) and torch.all(out[:, 1034:] == -5.0)


@pytest.mark.parametrize("M,N,K", [(4100, 300, 200), (2048, 512, 1024), (129, 7, 3), (2500, 1030, 333),
                                   (3000, 700, 64), (3200, 2100, 96)])
def test_pinned_integer_exact(oracle_lib, M, N, K):
    """Pinned buffers across one to four row panels; integer inputs make every
    partial sum exact, so C must equal the oracle bit for bit.  With several
    panels and N >= 512 the first panel is computed in column blocks of B
    (2048x512: 256 + 256; 2500x1030: 256 + 256 + 256 + 262, rows not 16-byte
    aligned; 3000x700: 256 + 444).  3200x2100 is wide: panels of 1024, 1664
    and 512 rows, the first in column blocks of 512 + 512 + 512 + 564."""
    A = torch.from_numpy(synth.matrix(M, K, 93, 0, "int5")).pin_memory()
    B = torch.from_numpy(synth.matrix(K, N, 93, 1, "int5")).pin_memory()
    C = sg.sgemm_host(A, B)
    Cr, _ = oracle_lib.gemm(A.numpy(), B.numpy())
    np.testing.assert_array_equal(C.numpy().astype(np.float64), Cr)


def test_back_to_back_calls_share_a_workspace(oracle_lib):
    """Two products queued on one stream with one workspace and no sync in
    between: the second call's copies wait for the first call's product."""
    M, N, K = 2100, 260, 300
    dev = torch.device("cuda:0")
    ws = torch.empty(sg.host_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    As = [torch.from_numpy(synth.matrix(M, K, 95 + i, 0)).pin_memory() for i in range(2)]
    Bs = [torch.from_numpy(synth.matrix(K, N, 95 + i, 1)).pin_memory() for i in range(2)]
    Cs = [torch.empty(M, N).pin_memory() for _ in range(2)]
    for i in range(2):
        st = sg.sgemm_f32_host(M, N, K, As[i].data_ptr(), K, Bs[i].data_ptr(), N, Cs[i].data_ptr(), N,
                               ws.data_ptr(), ws.numel(), s.cuda_stream)
        assert st == 0
    s.synchronize()
    for i in range(2):
        Cr, Sr = oracle_lib.gemm(As[i].numpy(), Bs[i].numpy())
        tol.assert_close(Cs[i].numpy(), Cr, Sr, K, f"call {i}")


def test_empty_and_k_zero():
    C = torch.full((5, 6), 7.0)
    A = torch.empty(5, 0)
    B = torch.empty(0, 6)
    sg.sgemm_host(A, B, out=C)
    assert torch.all(C == 0.0)
    # several panels, first one split in column halves, nothing to copy in
    C = torch.full((2100, 600), 7.0).pin_memory()
    sg.sgemm_host(torch.empty(2100, 0), torch.empty(0, 600), out=C)
    assert torch.all(C == 0.0)
    assert sg.sgemm_f32_host(0, 6, 3, 0, 3, 0, 6, 0, 6, 0, 0, 0) == 0


def test_workspace_checks():
    A = torch.zeros(64, 64)
    need = sg.host_workspace_size(64, 64, 64)
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    C = torch.zeros(64, 64)
    p = A.data_ptr()
    assert sg.sgemm_f32_host(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, 0, 0, 0) == -3
    assert sg.sgemm_f32_host(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, ws.data_ptr() + 16, need, 0) == -7
    assert sg.sgemm_f32_host(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, ws.data_ptr(), need - 4, 0) == -7
    assert sg.sgemm_f32_host(64, 64, 64, p, 64, p, 64, p, 64, ws.data_ptr(), need, 0) == -4
