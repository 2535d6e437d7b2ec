"""Tensor-core 3xTF32 variant (sgemm_f32_3xtf32) vs the FP64 oracle (needs a GB300).

Same acceptance as the CUDA-core path: |C - C_ref| <= 4*K*2**-24*(|A|.|B|)_ij
and relative Frobenius error <= 1e-5.  Integer-valued inputs in {-2..2} are
split exactly (lo = 0) and every partial sum is exact, so there the result
must equal the oracle bit for bit.
"""
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


def _tc(A, B):
    C = sg.sgemm_tc(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("M,N,K", [(128, 128, 32), (256, 256, 256), (1000, 1030, 777), (129, 255, 4097),
                                   (1, 1, 1), (5, 7, 3)])
def test_integer_inputs_exact(oracle_lib, M, N, K):
    A = synth.matrix(M, K, 71, 0, "int5")
    B = synth.matrix(K, N, 71, 1, "int5")
    C = _tc(A, B).cpu().numpy()
    Cr, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(C.astype(np.float64), Cr)
    assert sg.tc_timeouts() == 0


@pytest.mark.parametrize("M,N,K,kind", [(256, 256, 256, "uniform"), (1024, 1024, 1024, "normal"),
                                        (1000, 1030, 777, "uniform"), (300, 500, 2048, "normal")])
def test_float_inputs_within_tolerance(oracle_lib, M, N, K, kind):
    A = synth.matrix(M, K, 73, 0, kind)
    B = synth.matrix(K, N, 73, 1, kind)
    C = _tc(A, B).cpu().numpy()
    Cr, Sr = oracle_lib.gemm(A, B)
    tol.assert_close(C, Cr, Sr, K, f"3xtf32 {M}x{N}x{K}")


@pytest.mark.parametrize("name", ["sgemm_4096x4096x4096_uniform", "sgemm_8192x8192x8192_normal",
                                  "sgemm_16384x256x4096_normal"])
def test_workloads_sampled(oracle_lib, name):
    w = synth.WORKLOADS[name]
    A, B = w.inputs()
    C = _tc(A, B)
    rows, cols = synth.sample_indices(w.M, w.N, 4096, w.seed)
    Cs = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    ref, S = oracle_lib.gemm_sampled(A, B, rows, cols)
    rep = tol.assert_close(Cs, ref, S, w.K, name)
    assert rep["frob_rel"] < 1e-5


def test_strided_misaligned_views(oracle_lib):
    base = torch.from_numpy(synth.matrix(300, 402, 75, 0)).cuda()
    A = base[3:280, 1:390]              # row stride 402, base misaligned by 4 bytes
    B = torch.from_numpy(synth.matrix(389, 131, 75, 1)).cuda()
    out = torch.full((277, 140), -9.0, device="cuda")
    sg.sgemm_tc(A, B, out=out[:, 2:133])
    torch.cuda.synchronize()
    Cr, Sr = oracle_lib.gemm(A.cpu().numpy(), B.cpu().numpy())
    tol.assert_close(out[:, 2:133].cpu().numpy(), Cr, Sr, 389, "views")
    assert torch.all(out[:, :2] == -9.0) and torch.all(out[:, 133:] == -9.0)


def test_k_zero_and_empty():
    t = torch.full((64,), 3.0, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    assert sg.sgemm_f32_3xtf32(4, 4, 0, 0, 1, 0, 4, t.data_ptr(), 4, ws.data_ptr(), 256, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(t[:16] == 0.0) and torch.all(t[16:] == 3.0)
    assert sg.sgemm_f32_3xtf32(0, 4, 4, 0, 4, 0, 4, 0, 4, 0, 0, 0) == 0


def test_workspace_checks():
    A = torch.zeros(64, 64, device="cuda")
    need = sg.tc_workspace_size(64, 64, 64)
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    p = A.data_ptr()
    C = torch.zeros(64, 64, device="cuda")
    assert sg.sgemm_f32_3xtf32(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, 0, 0, 0) == -3
    assert sg.sgemm_f32_3xtf32(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, ws.data_ptr() + 16, need, 0) == -7
    assert sg.sgemm_f32_3xtf32(64, 64, 64, p, 64, p, 64, C.data_ptr(), 64, ws.data_ptr(), need - 4, 0) == -7
    assert sg.sgemm_f32_3xtf32(64, 64, 64, p, 64, p, 64, p, 64, ws.data_ptr(), need, 0) == -4
    # the workspace may not overlap an operand
    big = torch.empty(need // 4 + 64 * 64 + 64, device="cuda")
    wsp = (big.data_ptr() + 255) // 256 * 256
    assert sg.sgemm_f32_3xtf32(64, 64, 64, wsp + need - 256, 64, p, 64, C.data_ptr(), 64, wsp, need, 0) == -4


@pytest.mark.parametrize("M,N,K", [(300, 500, 2048), (129, 255, 4097), (1024, 1024, 1024), (2048, 2048, 2048)])
def test_split_tiles_deterministic(oracle_lib, M, N, K):
    """Shapes whose tiles are cut between CTA pairs (2 to 17 parts per tile):
    the parts are added in part order, so repeated calls are bit-identical,
    and the result meets the FP32 acceptance bound."""
    A = synth.matrix(M, K, 77, 0, "normal")
    B = synth.matrix(K, N, 77, 1, "normal")
    C1 = _tc(A, B).clone()
    C2 = _tc(A, B)
    assert torch.equal(C1, C2)
    if M * N * K <= 2048 ** 3 // 4:
        Cr, Sr = oracle_lib.gemm(A, B)
        tol.assert_close(C1.cpu().numpy(), Cr, Sr, K, f"split {M}x{N}x{K}")
    else:
        rows, cols = synth.sample_indices(M, N, 2048, 77)
        Cs = C1[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
        ref, S = oracle_lib.gemm_sampled(A, B, rows, cols)
        tol.assert_close(Cs, ref, S, K, f"split {M}x{N}x{K} sampled")
    assert sg.tc_timeouts() == 0


def test_dirty_workspace(oracle_lib):
    """A reused workspace full of stale bytes (counts and partial sums
    included) does not leak into C."""
    M, N, K = 1000, 1030, 777
    A = synth.matrix(M, K, 79, 0)
    B = synth.matrix(K, N, 79, 1)
    need = sg.tc_workspace_size(M, N, K)
    ws = torch.full(((need + 3) // 4,), float("nan"), device="cuda")
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.empty(M, N, device="cuda")
    st = sg.sgemm_f32_3xtf32(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, C.data_ptr(), N, ws.data_ptr(),
                             ws.numel() * 4, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    Cr, Sr = oracle_lib.gemm(A, B)
    tol.assert_close(C.cpu().numpy(), Cr, Sr, K, "dirty workspace")
    assert sg.tc_timeouts() == 0


def test_short_split_region(oracle_lib):
    """One full wave of CTA pairs plus two tiles: the split region holds fewer
    K blocks than there are pairs, so only some pairs share it."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    M, N, K = 256 * (pairs + 2), 200, 4096
    A = synth.matrix(M, K, 81, 0, "normal")
    B = synth.matrix(K, N, 81, 1, "normal")
    C1 = _tc(A, B).clone()
    C2 = _tc(A, B)
    assert torch.equal(C1, C2)
    rows, cols = synth.sample_indices(M, N, 2048, 81)
    rows = np.concatenate([rows, np.arange(M - 256, M, dtype=rows.dtype)])  # every row of the last tile
    cols = np.concatenate([cols, np.full(256, N - 1, dtype=cols.dtype)])
    Cs = C1[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    ref, S = oracle_lib.gemm_sampled(A, B, rows, cols)
    tol.assert_close(Cs, ref, S, K, "short split region")
    assert sg.tc_timeouts() == 0
