"""sgemm_f32_ws (balanced schedules) vs the FP64 oracle and vs sgemm_f32 (needs a GB300).

Shapes have more 128 x 128 output tiles than the GPU holds CTAs at once (2 per
SM) and a count that does not divide evenly, so tiles are cut into K parts:
between two CTAs through C (schedule 1, rows not 16-byte aligned) or into 4 to
8 parts of a split tail (schedule 3, aligned rows).
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


def _tiles(M, N):
    return ((M + 127) // 128) * ((N + 127) // 128)


def _run_ws(M, N, K, A, lda, B, ldb, ldc, a_off=0, b_off=0, c_off=0, ws_fill=0):
    from tests._gpu import dev_buffer
    tA, pA = dev_buffer(A, a_off)
    tB, pB = dev_buffer(B, b_off)
    c_elems = (M - 1) * ldc + N
    tC = torch.full((c_elems + c_off + 4,), float("nan"), device="cuda")
    nbytes = sg.workspace_size(M, N, K)
    ws = torch.full((nbytes // 4,), ws_fill, dtype=torch.int32, device="cuda")
    pC = tC.data_ptr() + 4 * c_off
    sst, kind, words = sg.ws_schedule(M, N, K, pA, lda, pB, ldb, pC, ldc, nbytes)
    assert sst == 0 and 0 < words <= nbytes // 4
    st = sg.sgemm_f32_ws(M, N, K, pA, lda, pB, ldb, pC, ldc, ws.data_ptr(), nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    raw = tC.cpu().numpy()[c_off:c_off + c_elems]
    C = np.stack([raw[i * ldc:i * ldc + N] for i in range(M)])
    # the call zero-fills the first `words` words (flags and error word, or
    # tile counts) and leaves them zero
    return st, C, ws.cpu().numpy()[:words], kind


@pytest.mark.parametrize("M,N,K,kind", [(2500, 2100, 333, "uniform"), (2432, 2560, 300, "normal"),
                                        (4096, 1408, 129, "uniform")])
def test_streamk_full_check(oracle_lib, M, N, K, kind):
    assert _tiles(M, N) > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    A = synth.matrix(M, K, 17, 0, kind)
    B = synth.matrix(K, N, 17, 1, kind)
    st, C, ws, kind = _run_ws(M, N, K, A, K, B, N, N, ws_fill=7)
    assert st == 0
    assert kind == (3 if K % 4 == 0 and N % 4 == 0 else 1)
    assert not ws.any(), "flags and error word (or tile counts) must be zero after a successful call"
    Cr, Sr = oracle_lib.gemm(A, B)
    tol.assert_close(C, Cr, Sr, K, f"stream-K {M}x{N}x{K}")


def test_streamk_misaligned_strides_and_offsets(oracle_lib):
    M, N, K = 2401, 2333, 257
    lda, ldb, ldc = 259, 2335, 2337
    A = synth.matrix(M, K, 23, 0, ld=lda, pad_value=np.nan)
    B = synth.matrix(K, N, 23, 1, ld=ldb, pad_value=np.nan)
    st, C, ws, kind = _run_ws(M, N, K, A, lda, B, ldb, ldc, a_off=1, b_off=3, c_off=2)
    assert st == 0 and kind == 1 and not ws.any()
    Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
    tol.assert_close(C, Cr, Sr, K, "stream-K misaligned")


def test_streamk_integer_inputs_exact_and_equal_to_data_parallel(oracle_lib):
    M, N, K = 2500, 2100, 1000
    A = synth.matrix(M, K, 29, 0, "int5")
    B = synth.matrix(K, N, 29, 1, "int5")
    st, C, _, kind = _run_ws(M, N, K, A, K, B, N, N)
    assert st == 0 and kind == 3
    Cr, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(C.astype(np.float64), Cr)
    from tests._gpu import run
    st2, C2, _ = run(M, N, K, A, K, B, N)
    assert st2 == 0
    np.testing.assert_array_equal(C, C2)


def test_streamk_deterministic_4096():
    A = torch.from_numpy(synth.matrix(4096, 4096, 3, 0)).cuda()
    B = torch.from_numpy(synth.matrix(4096, 4096, 3, 1)).cuda()
    C1 = sg.sgemm(A, B)
    C2 = sg.sgemm(A, B)
    C3 = sg.sgemm(A, B, balanced=False)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    # same products, different split of the K sum on cut tiles: FP32 rounding only
    rel = ((C1.double() - C3.double()).norm() / C3.double().norm()).item()
    assert rel < 1e-6


def test_words_past_the_used_ones_are_untouched():
    """Schedule 1 (rows not 16-byte aligned) uses only its flag words."""
    M, N, K = 2500, 2100, 41
    A = synth.matrix(M, K, 37, 0)
    B = synth.matrix(K, N, 37, 1)
    from tests._gpu import dev_buffer
    tA, pA = dev_buffer(A)
    tB, pB = dev_buffer(B)
    C = torch.empty(M, N, device="cuda")
    nbytes = (_tiles(M, N) + 1) * 4  # schedule 1's flags only: no room to copy A
    sst, kind, used = sg.ws_schedule(M, N, K, pA, K, pB, N, C.data_ptr(), N, nbytes)
    assert sst == 0 and kind == 1 and used == _tiles(M, N) + 1
    ws = torch.full((nbytes // 4 + 8,), 7, dtype=torch.int32, device="cuda")
    st = sg.sgemm_f32_ws(M, N, K, pA, K, pB, N, C.data_ptr(), N, ws.data_ptr(), nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and not ws[:used].any() and torch.all(ws[used:] == 7)


@pytest.mark.parametrize("extra_rows,extra_cols,K,n_cut", [(0, 23, 512, 0), (5, 0, 1024, 0), (5, 0, 1024, 12)])
def test_split_tail_parts(oracle_lib, extra_rows, extra_cols, K, n_cut):
    """Schedule 3 with more leftover tiles than SMs (fewer than 8 parts each)
    and with a handful of leftover tiles (4 parts), ragged last tile row and
    column: full check against the oracle, deterministic, tile counts left
    zero."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # one whole wave of 2 * sms tiles plus the leftover: rows of 128 x (cols) tiles
    cols = 20 + extra_cols
    rows = (2 * sms + (sms + 4 if extra_cols else 5)) // cols + 1 + extra_rows
    M, N = 128 * rows - 37, 128 * cols - n_cut  # ragged last tile row; n_cut keeps rows 16-byte aligned
    T = _tiles(M, N)
    assert T > 2 * sms and T % (2 * sms) != 0
    A = synth.matrix(M, K, 53, 0, "normal")
    B = synth.matrix(K, N, 53, 1, "normal")
    st, C, ws, kind = _run_ws(M, N, K, A, K, B, N, N, ws_fill=9)
    assert st == 0 and kind == 3 and not ws.any()
    Cr, Sr = oracle_lib.gemm(A, B)
    tol.assert_close(C, Cr, Sr, K, f"split tail {M}x{N}x{K}")
    st2, C2, _, _ = _run_ws(M, N, K, A, K, B, N, N)
    assert st2 == 0 and np.array_equal(C, C2)


def test_small_workspace_falls_back_to_one_cta_per_tile(oracle_lib):
    M, N, K = 2500, 2100, 64
    A = synth.matrix(M, K, 31, 0)
    B = synth.matrix(K, N, 31, 1)
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.empty(M, N, device="cuda")
    ws = torch.zeros(16, dtype=torch.int32, device="cuda")  # too small: ignored
    st = sg.sgemm_f32_ws(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, C.data_ptr(), N, ws.data_ptr(), 64,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and not ws.any()
    Cr, Sr = oracle_lib.gemm(A, B)
    tol.assert_close(C.cpu().numpy(), Cr, Sr, K, "fallback")


def _plan_words(M, N, K, pA, lda, pB, ldb, pC, ldc):
    """Flag words (with the error word) of the multi-part schedule (kind 2,
    fewer tiles than resident CTAs) the library plans for these operands, or
    None if it plans another schedule."""
    sst, kind, words = sg.ws_schedule(M, N, K, pA, lda, pB, ldb, pC, ldc, sg.workspace_size(M, N, K))
    assert sst == 0
    if kind != 2:
        return None
    assert words > _tiles(M, N) + 1, "more parts than tiles"
    return words


# Products with at most G / 2 tiles take the cluster split of K instead where
# it is expected to be faster (test_clusterk_gpu.py); these shapes keep the
# multi-part split.
@pytest.mark.parametrize("M,N,K,lds,kind", [
    (2048, 1024, 1024, None, "normal"),          # 128 tiles
    (1000, 2470, 333, (333, 2470, 2470), "uniform"),  # 160 tiles, misaligned rows: cp.async path
    (1024, 256, 8192, None, "normal"),           # 16 tiles, deep K
])
def test_multipart_split_full_check(oracle_lib, M, N, K, lds, kind):
    lda, ldb, ldc = lds or (K, N, N)
    A = synth.matrix(M, K, 43, 0, kind, ld=lda)
    B = synth.matrix(K, N, 43, 1, kind, ld=ldb)
    from tests._gpu import dev_buffer
    tA, pA = dev_buffer(A)
    tB, pB = dev_buffer(B)
    c_elems = (M - 1) * ldc + N
    tC = torch.full((c_elems + 4,), float("nan"), device="cuda")
    words = _plan_words(M, N, K, pA, lda, pB, ldb, tC.data_ptr(), ldc)
    assert words is not None, "shape must use the multi-part schedule"
    nbytes = sg.workspace_size(M, N, K)
    assert nbytes >= words * 4 + (words - 1) * 128 * 128 * 4
    ws = torch.full((nbytes // 4,), 5, dtype=torch.int32, device="cuda")
    st = sg.sgemm_f32_ws(M, N, K, pA, lda, pB, ldb, tC.data_ptr(), ldc, ws.data_ptr(), nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    assert not ws[:words].any(), "flags and error word must be zero after a successful call"
    raw = tC.cpu().numpy()[:c_elems]
    C = np.stack([raw[i * ldc:i * ldc + N] for i in range(M)])
    Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
    tol.assert_close(C, Cr, Sr, K, f"multi-part {M}x{N}x{K}")


def test_multipart_integer_exact_and_deterministic(oracle_lib):
    M, N, K = 2048, 1024, 1024
    A = synth.matrix(M, K, 47, 0, "int5")
    B = synth.matrix(K, N, 47, 1, "int5")
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    probe = torch.empty(M, N, device="cuda")
    assert _plan_words(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, probe.data_ptr(), N) is not None
    C1 = sg.sgemm(tA, tB)
    C2 = sg.sgemm(tA, tB)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    Cr, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(C1.cpu().numpy().astype(np.float64), Cr)
