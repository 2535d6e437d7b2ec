"""CUDA path vs the FP64 oracle, element by element (needs a GB300).

Acceptance (tests/_tolerance.py): |C - C_ref| <= 4*K*2**-24*(|A|.|B|)_ij and
relative Frobenius error <= 1e-5; integer-valued inputs must match exactly.
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


def _gpu():
    from tests import _gpu
    return _gpu


@pytest.mark.parametrize("name", ["sgemm_256x256x256_uniform", "sgemm_1024x1024x1024_normal",
                                  "sgemm_1000x1030x777_ragged_uniform"])
def test_workloads_full(oracle_lib, name):
    w = synth.WORKLOADS[name]
    A, B = w.inputs(ld_buffers=True)
    st, C, _ = _gpu().run(w.M, w.N, w.K, A, w.lda, B, w.ldb, w.ldc)
    assert st == 0
    Cr, Sr = oracle_lib.gemm(A, B, M=w.M, N=w.N, K=w.K, lda=w.lda, ldb=w.ldb)
    rep = tol.assert_close(C, Cr, Sr, w.K, name)
    assert rep["n"] == w.M * w.N


@pytest.mark.parametrize("name", ["sgemm_4096x4096x4096_uniform", "sgemm_16384x256x4096_normal",
                                  "sgemm_8192x8192x8192_normal"])
def test_workloads_sampled(oracle_lib, name):
    w = synth.WORKLOADS[name]
    A, B = w.inputs()
    tA = torch.from_numpy(A).cuda()
    tB = torch.from_numpy(B).cuda()
    C = sg.sgemm(tA, tB)
    torch.cuda.synchronize()
    rows, cols = synth.sample_indices(w.M, w.N, 4096, w.seed)
    Cs = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    ref, S = oracle_lib.gemm_sampled(A, B, rows, cols)
    rep = tol.assert_close(Cs, ref, S, w.K, name)
    assert rep["n"] == rows.size >= 4096


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1000, 1030, 777), (300, 200, 8192), (129, 257, 4095)])
def test_integer_inputs_bit_exact(oracle_lib, M, N, K):
    A = synth.matrix(M, K, 13, 0, "int5")
    B = synth.matrix(K, N, 13, 1, "int5")
    st, C, _ = _gpu().run(M, N, K, A, K, B, N)
    assert st == 0
    Cr, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(C.astype(np.float64), Cr)


@pytest.mark.parametrize("name", ["sgemm_4096x4096x4096_uniform", "sgemm_16384x256x4096_normal"])
def test_workloads_full_large(oracle_lib, name):
    # every output of the product, on the entry point and workspace the
    # benchmark times (sgemm_f32_ws with the workspace it asks for)
    w = synth.WORKLOADS[name]
    A, B = w.inputs()
    C = sg.sgemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    Cr, Sr = oracle_lib.gemm(A, B)
    rep = tol.assert_close(C.cpu().numpy(), Cr, Sr, w.K, name)
    assert rep["n"] == w.M * w.N


def test_integer_inputs_bit_exact_4096_full(oracle_lib):
    # integer inputs in {-2..2}: every partial sum is exact in FP32, so all
    # 4096 x 4096 outputs must equal the oracle bit for bit
    M = N = K = 4096
    A = synth.matrix(M, K, 3, 0, "int5")
    B = synth.matrix(K, N, 3, 1, "int5")
    C = sg.sgemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    Cr, _ = oracle_lib.gemm(A, B, with_abs=False)
    np.testing.assert_array_equal(C.cpu().numpy().astype(np.float64), Cr)


SIZES = [1, 2, 3, 4, 5, 7, 8, 15, 16, 17, 31, 33, 127, 128, 129]


def _edge_shapes():
    rng = np.random.default_rng(1234)
    shapes = {(m, 17, 33) for m in SIZES} | {(33, n, 17) for n in SIZES} | {(17, 33, k) for k in SIZES}
    while len(shapes) < 160:
        shapes.add(tuple(int(x) for x in rng.choice(SIZES, 3)))
    return sorted(shapes)


def test_edge_shape_sweep(oracle_lib):
    for (M, N, K) in _edge_shapes():
        A = synth.matrix(M, K, 99, 0)
        B = synth.matrix(K, N, 99, 1)
        st, C, _ = _gpu().run(M, N, K, A, K, B, N)
        assert st == 0, (M, N, K)
        Cr, Sr = oracle_lib.gemm(A, B)
        tol.assert_close(C, Cr, Sr, K, f"{M}x{N}x{K}")


@pytest.mark.parametrize("a_off,b_off,c_off", [(0, 0, 0), (1, 0, 0), (0, 1, 0), (0, 2, 0), (0, 0, 1),
                                               (0, 0, 2), (3, 3, 3), (1, 2, 3)])
@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad", [(0, 0, 0), (1, 2, 3), (4, 4, 4), (5, 6, 7)])
def test_leading_dims_offsets_and_poisoned_padding(oracle_lib, a_off, b_off, c_off, lda_pad, ldb_pad, ldc_pad):
    M, N, K = 133, 150, 70
    lda, ldb, ldc = K + lda_pad, N + ldb_pad, N + ldc_pad
    A = synth.matrix(M, K, 31, 0, ld=lda, pad_value=np.nan)
    B = synth.matrix(K, N, 31, 1, ld=ldb, pad_value=np.nan)
    st, C, raw = _gpu().run(M, N, K, A, lda, B, ldb, ldc, a_off, b_off, c_off, c_fill=-7.0)
    assert st == 0
    Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
    tol.assert_close(C, Cr, Sr, K, "strided")
    # elements between N and ldc in each row are left alone
    for i in range(M - 1):
        assert np.all(raw[i * ldc + N:(i + 1) * ldc] == -7.0)


def test_k_zero_gives_zeros():
    st, C, _ = _gpu().run(37, 45, 0, None, 1, None, 45, c_fill=123.0)
    assert st == 0 and np.all(C == 0.0) and not np.signbit(C).any()


def test_empty_m_or_n_is_noop():
    t = torch.full((16,), 5.0, device="cuda")
    assert sg.sgemm_f32(0, 4, 4, t.data_ptr(), 4, t.data_ptr(), 4, t.data_ptr(), 4, 0) == 0
    assert sg.sgemm_f32(4, 0, 4, t.data_ptr(), 4, t.data_ptr(), 1, t.data_ptr(), 1, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(t == 5.0)


def test_nan_and_inf_propagate(oracle_lib):
    M, N, K = 70, 90, 50
    A = synth.matrix(M, K, 5, 0)
    B = synth.matrix(K, N, 5, 1)
    A[3, 7] = np.nan
    B[11, 20] = np.inf
    st, C, _ = _gpu().run(M, N, K, A, K, B, N)
    assert st == 0
    Cr, Sr = oracle_lib.gemm(A, B)
    assert np.array_equal(np.isnan(C), np.isnan(Cr))
    assert np.array_equal(np.isinf(C), np.isinf(Cr))
    ok = np.isfinite(Cr)
    tol.assert_close(C[ok], Cr[ok], Sr[ok], K, "finite part")


def test_alias_rejected_with_device_pointers():
    t = torch.zeros(64 * 64 * 3, device="cuda")
    p = t.data_ptr()
    assert sg.sgemm_f32(64, 64, 64, p, 64, p + 4 * 4096, 64, p + 4 * 100, 64, 0) == -4
    assert sg.sgemm_f32(64, 64, 64, p, 64, p + 4 * 4096, 64, p + 4 * 4096, 64, 0) == -4


def test_transpose_identity(oracle_lib):
    # (A.B)^T = B^T.A^T.  Without a workspace every output's FMAs run in k
    # order within K parts whose cut points depend only on the tile and K-tile
    # counts (one part, or one per CTA of a cluster), the same for both
    # products here (6 tiles each), so the two agree bit for bit; the balanced
    # schedule cuts K at points that depend on the tile's position, so there
    # they agree to FP32 rounding.
    An = synth.matrix(300, 200, 8, 0, "normal")
    Bn = synth.matrix(200, 170, 8, 1, "normal")
    A, B = torch.from_numpy(An).cuda(), torch.from_numpy(Bn).cuda()
    C = sg.sgemm(A, B, balanced=False)
    Ct = sg.sgemm(B.t().contiguous(), A.t().contiguous(), balanced=False)
    Cb = sg.sgemm(A, B)
    Cbt = sg.sgemm(B.t().contiguous(), A.t().contiguous())
    torch.cuda.synchronize()
    assert torch.equal(C, Ct.t())
    _, S = oracle_lib.gemm(An, Bn)
    tol.assert_close(Cb.cpu().numpy(), Cbt.t().cpu().numpy().astype(np.float64), S, 200, "balanced transpose")


def test_deterministic_and_stream_ordered(oracle_lib):
    s = torch.cuda.Stream()
    A = torch.from_numpy(synth.matrix(513, 385, 4, 0)).cuda()
    B = torch.from_numpy(synth.matrix(385, 257, 4, 1)).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C1 = sg.sgemm(A, B)
        C2 = sg.sgemm(A, B, stream=s)
    s.synchronize()
    assert torch.equal(C1, C2)
    Cr, Sr = oracle_lib.gemm(A.cpu().numpy(), B.cpu().numpy())
    tol.assert_close(C1.cpu().numpy(), Cr, Sr, 385, "side stream")


def test_torch_wrapper_strided_views(oracle_lib):
    base = torch.from_numpy(synth.matrix(200, 300, 6, 0)).cuda()
    A = base[10:150, 20:250]          # row stride 300, offset pointer
    B = torch.from_numpy(synth.matrix(230, 90, 6, 1)).cuda()
    out = torch.full((140, 96), -1.0, device="cuda")
    sg.sgemm(A, B, out=out[:, :90])
    torch.cuda.synchronize()
    Cr, Sr = oracle_lib.gemm(A.cpu().numpy(), B.cpu().numpy())
    tol.assert_close(out[:, :90].cpu().numpy(), Cr, Sr, 230, "views")
    assert torch.all(out[:, 90:] == -1.0)
