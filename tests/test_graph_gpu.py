"""sgemm_f32, sgemm_f32_ws, sgemm_f32_host and sgemm_f32_3xtf32 captured in a
CUDA graph and replayed (needs a GB300).

Each of them only enqueues work on the caller's stream (kernel launches,
memsets, and for the host-buffer path copies on two internal streams joined by
events), so a stream capture records the whole call.  After a first call
outside the capture (the per-device set-up runs once), a replayed graph must
give exactly the result of a direct call: the schedules are deterministic, so
bit for bit.  Each graph is replayed with new operand values in the same
buffers, to show that it reads them at replay time.
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


def _capture(call):
    """Graph of one call(stream) -> status; the call must succeed in capture."""
    g = torch.cuda.CUDAGraph()
    status = []
    with torch.cuda.graph(g):
        status.append(call(torch.cuda.current_stream().cuda_stream))
    assert status == [0]
    return g


def _replay_matches_direct(oracle_lib, M, N, K, call, tA, tB, tC, seed, check_tol=True):
    """Direct call, then graph replays on fresh inputs copied into the same
    buffers; each replay must equal a direct call on those inputs."""
    s = torch.cuda.current_stream().cuda_stream
    assert call(s) == 0  # set-up outside the capture
    torch.cuda.synchronize()
    g = _capture(call)
    for r in range(2):
        A = synth.matrix(M, K, seed + r, 0)
        B = synth.matrix(K, N, seed + r, 1)
        tA.copy_(torch.from_numpy(A))
        tB.copy_(torch.from_numpy(B))
        tC.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        from_graph = tC.clone()
        tC.fill_(float("nan"))
        assert call(torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(from_graph.cpu(), tC.cpu()), f"replay {r} differs from a direct call"
        if check_tol:
            Cr, Sr = oracle_lib.gemm(A, B)
            tol.assert_close(from_graph.cpu().numpy(), Cr, Sr, K, f"graph replay {r} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,kind", [
    (2432, 2560, 300, 3),   # 380 tiles: whole waves plus the split-tail grid (programmatic launch)
    (2048, 1024, 1024, 2),  # 128 tiles: cooperative stream-K grid with partial-sum slots
    (1024, 1024, 1024, 32),  # 64 tiles: cluster split of K through distributed shared memory
])
def test_balanced_schedules_in_a_graph(oracle_lib, M, N, K, kind):
    tA = torch.empty(M, K, device="cuda")
    tB = torch.empty(K, N, device="cuda")
    tC = torch.empty(M, N, device="cuda")
    nbytes = sg.workspace_size(M, N, K)
    sst, got, _ = sg.ws_schedule(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, nbytes)
    assert sst == 0 and got & 255 == kind  # (bits 8 and up: the cluster size)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def call(s):
        return sg.sgemm_f32_ws(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, ws.data_ptr(), nbytes,
                               s)
    _replay_matches_direct(oracle_lib, M, N, K, call, tA, tB, tC, 301)


def test_kmajor_copy_in_a_graph(oracle_lib):
    """A whose rows are not 16-byte aligned (lda = K + 1) with room for its
    k-major copy (a product of at least 2 GFLOP): the transpose kernel, then
    the k-major kernels."""
    M, N, K = 1300, 1032, 777
    lda = K + 1
    tA = torch.empty(M, lda, device="cuda")[:, :K]
    tB = torch.empty(K, N, device="cuda")
    tC = torch.empty(M, N, device="cuda")
    nbytes = sg.workspace_size(M, N, K) + (K * ((M + 3) // 4 * 4) * 4 + 255) // 256 * 256
    sst, got, _ = sg.ws_schedule(M, N, K, tA.data_ptr(), lda, tB.data_ptr(), N, tC.data_ptr(), N, nbytes)
    assert sst == 0 and got & 16
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def call(s):
        return sg.sgemm_f32_ws(M, N, K, tA.data_ptr(), lda, tB.data_ptr(), N, tC.data_ptr(), N, ws.data_ptr(),
                               nbytes, s)
    _replay_matches_direct(oracle_lib, M, N, K, call, tA, tB, tC, 321)


def test_no_workspace_entry_in_a_graph(oracle_lib):
    M, N, K = 300, 262, 190
    tA = torch.empty(M, K, device="cuda")
    tB = torch.empty(K, N, device="cuda")
    tC = torch.empty(M, N, device="cuda")

    def call(s):
        return sg.sgemm_f32(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, s)
    _replay_matches_direct(oracle_lib, M, N, K, call, tA, tB, tC, 311)


def test_tensor_core_variant_in_a_graph(oracle_lib):
    M, N, K = 1000, 1030, 777
    tA = torch.empty(M, K, device="cuda")
    tB = torch.empty(K, N, device="cuda")
    tC = torch.empty(M, N, device="cuda")
    nbytes = sg.tc_workspace_size(M, N, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def call(s):
        return sg.sgemm_f32_3xtf32(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, ws.data_ptr(),
                                   nbytes, s)
    _replay_matches_direct(oracle_lib, M, N, K, call, tA, tB, tC, 321)


def test_host_buffer_entry_in_a_graph(oracle_lib):
    """Copies in on one internal stream, products on the captured stream,
    copies back on another: the events fork and join them inside the graph."""
    M, N, K = 2100, 600, 256
    hA = torch.empty(M, K).pin_memory()
    hB = torch.empty(K, N).pin_memory()
    hC = torch.empty(M, N).pin_memory()
    nbytes = sg.host_workspace_size(M, N, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def call(s):
        return sg.sgemm_f32_host(M, N, K, hA.data_ptr(), K, hB.data_ptr(), N, hC.data_ptr(), N, ws.data_ptr(),
                                 nbytes, s)
    hA.copy_(torch.from_numpy(synth.matrix(M, K, 330, 0, "int5")))
    hB.copy_(torch.from_numpy(synth.matrix(K, N, 330, 1, "int5")))
    assert call(torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    g = _capture(call)
    for r in range(2):
        A = synth.matrix(M, K, 331 + r, 0, "int5")
        B = synth.matrix(K, N, 331 + r, 1, "int5")
        hA.copy_(torch.from_numpy(A))
        hB.copy_(torch.from_numpy(B))
        hC.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        Cr, _ = oracle_lib.gemm(A, B)
        np.testing.assert_array_equal(hC.numpy().astype(np.float64), Cr)
