"""Several host threads calling the C ABI at once, each on its own stream with
its own workspace (needs a GB300).

The library's per-device set-up and caches are guarded by mutexes and the
calls only enqueue work, so concurrent callers must get exactly the results
of the same calls made one after another: every schedule is deterministic.
Each thread runs one shape of each schedule (one CTA per tile, the stream-K
split, the split tail, a repacked operand) and the tensor-core variant.
"""
import ctypes
import threading

import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth

pytestmark = pytest.mark.gpu

SHAPES = [(300, 262, 190), (1024, 1024, 1024), (2432, 2560, 300), (2100, 2060, 513)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


def _jobs(seed):
    jobs = []
    for i, (M, N, K) in enumerate(SHAPES):
        lda = K + (3 if i == 3 else 0)  # the last one has rows that are not 16-byte aligned
        A = torch.from_numpy(synth.matrix(M, K, seed + i, 0, ld=lda)).cuda()
        B = torch.from_numpy(synth.matrix(K, N, seed + i, 1)).cuda()
        jobs.append((M, N, K, A, lda, B))
    return jobs


def _run_all(jobs, stream):
    """Every job through sgemm_f32_ws (own workspace) and sgemm_f32_3xtf32."""
    out = []
    s = stream.cuda_stream
    with torch.cuda.stream(stream):
        for M, N, K, A, lda, B in jobs:
            C = torch.empty(M, N, device="cuda")
            nbytes = sg.workspace_size_for(M, N, K, A.data_ptr(), lda, B.data_ptr(), N)
            ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
            assert sg.sgemm_f32_ws(M, N, K, A.data_ptr(), lda, B.data_ptr(), N, C.data_ptr(), N, ws.data_ptr(),
                                   nbytes, s) == 0
            Ct = torch.empty(M, N, device="cuda")
            tbytes = sg.tc_workspace_size(M, N, K)
            tws = torch.empty(tbytes, dtype=torch.uint8, device="cuda")
            assert sg.sgemm_f32_3xtf32(M, N, K, A.data_ptr(), lda, B.data_ptr(), N, Ct.data_ptr(), N,
                                       tws.data_ptr(), tbytes, s) == 0
            out.append((C, Ct, ws, tws))  # keep the workspaces alive until the stream is done
    stream.synchronize()
    return [(C, Ct) for C, Ct, _, _ in out]


def test_concurrent_callers_match_serial_calls():
    n_threads = 4
    jobs = [_jobs(400 + 10 * t) for t in range(n_threads)]
    serial = [_run_all(j, torch.cuda.Stream()) for j in jobs]
    results = [None] * n_threads
    errors = []
    start = threading.Barrier(n_threads)

    def work(t):
        try:
            torch.cuda.set_device(0)
            start.wait()
            for _ in range(3):
                results[t] = _run_all(jobs[t], torch.cuda.Stream())
        except Exception as e:  # reported below, on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(n_threads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(n_threads):
        for (C, Ct), (Cs, Cts) in zip(results[t], serial[t]):
            assert torch.equal(C, Cs)
            assert torch.equal(Ct, Cts)
    assert sg.copy_timeouts() == 0 and sg.tc_timeouts() == 0


def test_torch_wrappers_on_two_streams_do_not_share_a_workspace():
    """sgemm / sgemm_tc cache their workspaces per device and stream, so
    products queued on two streams at once cannot overwrite each other's
    partial sums."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    jobs = _jobs(470)
    want = []
    for M, N, K, A, lda, B in jobs:
        Av = A.view(-1)[: (M - 1) * lda + K].as_strided((M, K), (lda, 1))
        want.append((sg.sgemm(Av, B), sg.sgemm_tc(Av, B)))
    torch.cuda.synchronize()
    for rep in range(3):
        got = []
        for i, (M, N, K, A, lda, B) in enumerate(jobs):
            Av = A.view(-1)[: (M - 1) * lda + K].as_strided((M, K), (lda, 1))
            s = s1 if (i + rep) % 2 == 0 else s2
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                got.append((sg.sgemm(Av, B, stream=s), sg.sgemm_tc(Av, B, stream=s)))
        torch.cuda.synchronize()
        for (C, Ct), (Cw, Ctw) in zip(got, want):
            assert torch.equal(C, Cw)
            assert torch.equal(Ct, Ctw)
