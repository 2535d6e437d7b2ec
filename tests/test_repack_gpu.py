"""Operands whose rows are not 16-byte aligned, copied into the workspace
(sgemm_f32_ws with room for the copies) vs the FP64 oracle (needs a GB300).

An unaligned A is transposed into its k-major copy (K rows of M rounded up to
4 floats) when the workspace has room for it, else repacked into rows of K
rounded up to 4; an unaligned B is repacked into rows of N rounded up to 4.
The 16-byte-aligned kernels and schedules then run on the copies.  Checked:
the reported plan (schedule bits and copy bits), the result against the
oracle (exactly, for integer inputs), that the schedule's leading words are
zero again afterwards, that nothing past the requested size is written, and
that the smaller workspace of sgemm_f32_workspace_size keeps the uncopied
path.
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


def _r256(b):
    return (b + 255) // 256 * 256


def _a_repack(M, K):
    return _r256(M * ((K + 3) // 4 * 4) * 4)


def _a_kmajor(M, K):
    return _r256(K * ((M + 3) // 4 * 4) * 4)


def _b_repack(K, N):
    return _r256(K * ((N + 3) // 4 * 4) * 4)


def _room(M, N, K):
    """Workspace bytes with room for either copy of A and the repacked B,
    whatever the size of the product (sgemm_f32_ws copies whenever the
    workspace has room)."""
    return sg.workspace_size(M, N, K) + max(_a_repack(M, K), _a_kmajor(M, K)) + _b_repack(K, N)


def _run(M, N, K, A, lda, B, ldb, ldc, a_off=0, b_off=0, nbytes=None, guard=64):
    from tests._gpu import dev_buffer
    tA, pA = dev_buffer(A, a_off)
    tB, pB = dev_buffer(B, b_off)
    c_elems = (M - 1) * ldc + N
    tC = torch.full((c_elems + 4,), float("nan"), device="cuda")
    if nbytes is None:
        nbytes = _room(M, N, K)
    ws = torch.full((nbytes // 4 + guard,), 9, dtype=torch.int32, device="cuda")
    sst, kind, words = sg.ws_schedule(M, N, K, pA, lda, pB, ldb, tC.data_ptr(), ldc, nbytes)
    assert sst == 0
    st = sg.sgemm_f32_ws(M, N, K, pA, lda, pB, ldb, tC.data_ptr(), ldc, ws.data_ptr(), nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    raw = tC.cpu().numpy()[:c_elems]
    C = np.stack([raw[i * ldc:i * ldc + N] for i in range(M)])
    w = ws.cpu().numpy()
    assert not w[:words].any(), "schedule words must be zero after the call"
    assert np.all(w[nbytes // 4:] == 9), "nothing past the requested workspace is written"
    return C, kind


# Products of at least 2 GFLOP (smaller ones copy nothing; the copy kernels
# on tiny shapes are covered by test_forced_copies_on_small_shapes).
@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,a_off,b_off,bits", [
    (1300, 1030, 777, 777, 1030, 1030, 0, 0, 16 | 8),   # ragged: A k-major, B repacked
    (2500, 2100, 333, 333, 2100, 2100, 0, 0, 16),       # A only (K odd), 380 tiles: split tail after
    (2500, 2100, 336, 336, 2102, 2100, 0, 0, 8),        # B only (ldb not a multiple of 4)
    (2300, 900, 512, 512, 900, 901, 1, 0, 16),          # A base off by 4 bytes, C misaligned too
    (512, 1030, 2049, 2049, 1030, 1030, 0, 0, 16 | 8),  # deep odd K
    (3001, 700, 515, 515, 700, 700, 0, 0, 16),          # M not a multiple of 4: padded k-major rows
])
def test_copied_operands_match_the_oracle(oracle_lib, M, N, K, lda, ldb, ldc, a_off, b_off, bits):
    A = synth.matrix(M, K, 351, 0, ld=lda, pad_value=np.nan)
    B = synth.matrix(K, N, 351, 1, ld=ldb, pad_value=np.nan)
    C, kind = _run(M, N, K, A, lda, B, ldb, ldc, a_off, b_off)
    assert kind & 28 == bits
    Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
    tol.assert_close(C, Cr, Sr, K, f"copied {M}x{N}x{K}")


@pytest.mark.parametrize("tiles_m,K", [(8, 1023), (4, 511)])
def test_room_for_the_row_repack_only(oracle_lib, tiles_m, K):
    """A workspace with room for the row repack of A but not for its k-major
    copy takes the row repack.  The tiles are exactly one wave of the CTAs the
    GPU holds at once (2 per SM), so both kernel families run one CTA per
    tile and the schedule needs no workspace; M = 1 and K = 3 (mod 4) with
    3K > M make the k-major copy (K rows of M rounded up to 4) larger than the
    row repack (M rows of K rounded up to 4)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if (2 * sms) % tiles_m:
        pytest.skip("the SM count does not split into whole tile columns")
    M, N = 128 * tiles_m - 3, 128 * (2 * sms // tiles_m)
    assert M % 4 == 1 and K % 4 == 3 and 3 * K > M
    assert _a_kmajor(M, K) > _a_repack(M, K)
    nbytes = _a_repack(M, K)
    A = synth.matrix(M, K, 352, 0, ld=K, pad_value=np.nan)
    B = synth.matrix(K, N, 352, 1, ld=N, pad_value=np.nan)
    C, kind = _run(M, N, K, A, K, B, N, N, nbytes=nbytes)
    assert kind == 4, kind  # one CTA per tile, A row-repacked
    Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=K, ldb=N)
    tol.assert_close(C, Cr, Sr, K, f"row-repacked {M}x{N}x{K}")
    # with room for the k-major copy as well, that copy is taken instead
    C2, kind2 = _run(M, N, K, A, K, B, N, N, nbytes=_a_kmajor(M, K))
    assert kind2 == 16, kind2
    tol.assert_close(C2, Cr, Sr, K, f"k-major {M}x{N}x{K}")


def test_repacked_integer_exact_and_same_as_aligned_copy(oracle_lib):
    """Integer inputs: exact.  And the repacked run equals the same product on
    operands the caller laid out with aligned rows (same kernels, same
    schedule, so bit for bit)."""
    M, N, K = 2432, 2560, 301
    A = synth.matrix(M, K, 353, 0, "int5")
    B = synth.matrix(K, N, 353, 1, "int5")
    C, kind = _run(M, N, K, A, K, B, N, N)
    assert kind == 3 | 16  # split tail, A in its k-major copy
    Cr, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(C.astype(np.float64), Cr)
    K4 = (K + 3) // 4 * 4
    A4 = np.zeros((M, K4), np.float32)
    A4[:, :K] = A
    Ca, kind_a = _run(M, N, K, A4, K4, B, N, N)
    assert kind_a == 3
    np.testing.assert_array_equal(C, Ca)


_FORCED_CHILD = r"""
import sys, json
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
import oracle
from tests import _tolerance as tol
from tests._gpu import dev_buffer
sg.load_library()
oracle.build()
out = []
for (M, N, K, lda, ldb) in json.loads(sys.argv[2]):
    A = synth.matrix(M, K, 358, 0, ld=lda, pad_value=np.nan)
    B = synth.matrix(K, N, 358, 1, ld=ldb, pad_value=np.nan)
    tA, pA = dev_buffer(A)
    tB, pB = dev_buffer(B)
    tC = torch.full((M * N + 4,), float("nan"), device="cuda")
    nbytes = sg.workspace_size(M, N, K) + (M + 4) * (K + 4) * 4 + (K + 4) * (M + 4) * 4 + (K + 4) * (N + 4) * 4 + 4096
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    _, kind, _ = sg.ws_schedule(M, N, K, pA, lda, pB, ldb, tC.data_ptr(), N, nbytes)
    st = sg.sgemm_f32_ws(M, N, K, pA, lda, pB, ldb, tC.data_ptr(), N, ws.data_ptr(), nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, st
    C = tC.cpu().numpy()[:M * N].reshape(M, N)
    Cr, Sr = oracle.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
    tol.assert_close(C, Cr, Sr, K, f"forced copies {M}x{N}x{K}")
    out.append(kind)
print(json.dumps(out))
"""


@pytest.mark.parametrize("tune,bits", [("kernels=kmajor16", 16 | 8), ("kernels=rowmajor8", 4 | 8)])
def test_forced_copies_on_small_shapes(tune, bits):
    """Below 2 GFLOP nothing is copied by default; with the kernel family
    forced by SGEMM_F32_TUNE (read once per process, so in a child process)
    the copies run on tiny and ragged shapes: N < 4, K < 16, M not a
    multiple of 4, a deep odd K."""
    import json, os, subprocess, sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    shapes = [(300, 5, 7, 7, 5), (129, 1030, 2049, 2049, 1030), (1001, 700, 515, 515, 702), (1000, 1030, 777, 777, 1030)]
    r = subprocess.run([sys.executable, "-c", _FORCED_CHILD, root, json.dumps(shapes)], cwd=root,
                       env=dict(os.environ, SGEMM_F32_TUNE=tune), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    kinds = json.loads(r.stdout.strip().splitlines()[-1])
    assert all(k & 28 == bits for k in kinds), kinds


def test_smaller_workspace_keeps_the_unrepacked_path(oracle_lib):
    M, N, K = 1000, 1030, 777
    A = synth.matrix(M, K, 355, 0)
    B = synth.matrix(K, N, 355, 1)
    C, kind = _run(M, N, K, A, K, B, N, N, nbytes=sg.workspace_size(M, N, K))
    assert kind & 28 == 0
    Cr, Sr = oracle_lib.gemm(A, B)
    tol.assert_close(C, Cr, Sr, K, "unrepacked")


def test_size_query_asks_for_repack_room_only_for_large_products():
    # unaligned rows: room for the copies from 2 GFLOP on; aligned rows: room
    # only where the k-major copy pays on its own (2048 x 2048 x 2049 does,
    # 1536^3 and the ragged product do not)
    from tests._gpu import dev_buffer
    for (M, N, K), large, pays in (((1000, 1030, 777), False, False), ((2048, 2048, 2049), True, True),
                                   ((1536, 1536, 1537), True, False)):
        tA, pA = dev_buffer(np.zeros(4, np.float32))
        base = sg.workspace_size(M, N, K)
        got = sg.workspace_size_for(M, N, K, pA, K, pA, N)
        assert (got > base) == large, (M, N, K)
        aligned = sg.workspace_size_for(M, N, K, pA, (K + 3) // 4 * 4, pA, (N + 3) // 4 * 4)
        assert (aligned > base) == pays, (M, N, K)


def test_torch_wrapper_uses_the_repack(oracle_lib):
    M, N, K = 2100, 2060, 513  # 4.4 GFLOP: the size query asks for repack room
    base = torch.from_numpy(synth.matrix(M, K + 3, 357, 0)).cuda()
    A = base[:, 1:K + 1]  # row stride K + 3, base off by 4 bytes
    B = torch.from_numpy(synth.matrix(K, N, 357, 1)).cuda()
    C = torch.empty(M, N, device="cuda")
    _, kind, _ = sg.ws_schedule(M, N, K, A.data_ptr(), K + 3, B.data_ptr(), N, C.data_ptr(), N)
    assert kind & 16
    sg.sgemm(A, B, out=C)
    torch.cuda.synchronize()
    Cr, Sr = oracle_lib.gemm(A.cpu().numpy(), B.cpu().numpy())
    tol.assert_close(C.cpu().numpy(), Cr, Sr, K, "wrapper")
