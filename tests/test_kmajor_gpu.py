"""The k-major copy of A (sgemm_f32_ws transposes A into its workspace first
and runs the kernels that load k-major A tiles) vs the FP64 oracle, and vs
the same call without the copy (needs a GB300).

With one CTA per tile the copy changes where A's tiles come from, not the
order of any sum, so the two calls agree bit for bit.  The split schedules
cut K into parts of whole K tiles, which are 32 deep on the k-major kernels
and 16 deep on the row-major ones, so there a part boundary can fall
elsewhere and the two calls agree within the FP32 bound, each checked
against the oracle.  Shapes are chosen where the size query asks for the
copy (large N) and cover the three schedules it runs with: one CTA per tile
over whole waves, the split tail, and the multi-part split of fewer tiles
than resident CTAs.
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


def _call(M, N, K, tA, tB, nbytes, guard=64):
    tC = torch.full((M, N), float("nan"), device="cuda")
    ws = torch.full((nbytes // 4 + guard,), 7, dtype=torch.int32, device="cuda")
    sst, kind, words = sg.ws_schedule(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, nbytes)
    assert sst == 0
    st = sg.sgemm_f32_ws(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, ws.data_ptr(), nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, sg.status_string(st)
    w = ws.cpu().numpy()
    assert not w[:words].any(), "schedule words must be zero after the call"
    assert np.all(w[nbytes // 4:] == 7), "nothing past the workspace is written"
    return tC.cpu().numpy(), kind


@pytest.mark.parametrize("M,N,K,sched,dist", [
    (2432, 4096, 4096, 0, "uniform"),   # 608 tiles = 2 whole waves of 304: one CTA per tile
    (4096, 8192, 1024, 3, "normal"),    # 2048 tiles: split tail
    (512, 8192, 8192, 2, "uniform"),    # 256 tiles < 304: multi-part split
    (4001, 4100, 3000, 3, "uniform"),   # ragged M, N and K tiles (M not a multiple of 4: padded k-major rows)
])
def test_kmajor_copy_matches_oracle_and_the_direct_call(oracle_lib, M, N, K, sched, dist):
    A = synth.matrix(M, K, 610, 0, dist)
    B = synth.matrix(K, N, 610, 1, dist)
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    nbytes = sg.workspace_size_for(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N)
    C, kind = _call(M, N, K, tA, tB, nbytes)
    assert kind == sched | 16, kind
    rows, cols = synth.sample_indices(M, N, 4096, 610)
    ref, S = oracle_lib.gemm_sampled(A, B, rows, cols)
    tol.assert_close(C[rows, cols], ref, S, K, f"k-major {M}x{N}x{K}")
    # without room for the copy: the row-major kernels
    C0, kind0 = _call(M, N, K, tA, tB, sg.workspace_size(M, N, K))
    assert kind0 & 16 == 0
    tol.assert_close(C0[rows, cols], ref, S, K, f"row-major {M}x{N}x{K}")
    if sched == 0:  # one CTA per tile on both: the same sums in the same order
        np.testing.assert_array_equal(C, C0)


def test_kmajor_copy_integer_inputs_exact(oracle_lib):
    """Integers in [-2, 2]: every partial sum is exact in FP32, so the sampled
    outputs equal the oracle exactly."""
    M, N, K = 4096, 8192, 1024
    A = synth.matrix(M, K, 611, 0, "int5")
    B = synth.matrix(K, N, 611, 1, "int5")
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C, kind = _call(M, N, K, tA, tB, sg.workspace_size_for(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N))
    assert kind & 16
    rows, cols = synth.sample_indices(M, N, 4096, 611)
    ref, _ = oracle_lib.gemm_sampled(A, B, rows, cols)
    np.testing.assert_array_equal(C[rows, cols].astype(np.float64), ref)


def test_size_query_asks_for_the_copy_only_where_it_pays():
    from tests._gpu import dev_buffer
    tA, pA = dev_buffer(np.zeros(4, np.float32))
    for (M, N, K), pays in (((4096, 4096, 4096), True), ((8192, 8192, 8192), True), ((2432, 4096, 4096), True),
                            ((16384, 256, 4096), False), ((2048, 2048, 2048), True), ((16384, 512, 4096), False),
                            ((2500, 2100, 4096), True), ((3072, 3072, 3072), True), ((4096, 1024, 4096), False),
                            ((1024, 1024, 1024), False)):
        base = sg.workspace_size(M, N, K)
        got = sg.workspace_size_for(M, N, K, pA, K, pA, N)
        assert (got > base) == pays, (M, N, K)
        if pays:
            assert got >= K * ((M + 3) // 4 * 4) * 4  # the k-major copy follows the schedule's words
