"""Seeded random shapes, leading dimensions and base offsets through every
schedule of sgemm_f32_ws (every other case with room to copy unaligned
operands: an unaligned A into its k-major copy, an unaligned B into aligned
rows), through sgemm_f32 and sgemm_f32_static_scratch, and through the 3xTF32
variant, against the FP64 oracle (needs a GB300).

Shapes are drawn log-uniformly so that small products (one CTA per tile,
multi-part split, cluster split of K), products with a partial last wave
(split tail or two-part split) and copied operands all occur; the test
asserts that each of them did.  Large products are checked on seeded
sampled outputs, the rest in full.
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


def _cases(n=36):
    rng = np.random.default_rng(2024)
    cases = []
    for i in range(n):
        M = int(np.exp(rng.uniform(0, np.log(2700))))
        N = int(np.exp(rng.uniform(0, np.log(2700))))
        K = int(np.exp(rng.uniform(0, np.log(1500))))
        if i % 3 == 0:  # force a partial last wave, with K deep enough to split
            M, N, K = int(rng.integers(2200, 2700)), int(rng.integers(2200, 2700)), int(rng.integers(17, 600))
        elif i % 6 == 1:  # 180 .. 210 tiles, between half and all of the resident CTAs: multi-part split
            M, N, K = 1800 + 3 * i, 1600 + 5 * i, 200 + 7 * i
        pads = [0, 0, 0, 1, 2, 3, 4]
        lda, ldb, ldc = K + int(rng.choice(pads)), N + int(rng.choice(pads)), N + int(rng.choice(pads))
        offs = [int(rng.choice([0, 0, 0, 1, 2])) for _ in range(3)]
        cases.append((M, N, K, lda, ldb, ldc, offs))
    return cases


def _check(oracle_lib, A, B, C, M, N, K, lda, ldb, what, seed):
    if M * N * K <= 2.5e8:
        Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
        tol.assert_close(C, Cr, Sr, K, what)
    else:
        rows, cols = synth.sample_indices(M, N, 2048, seed)
        A2 = np.stack([A[r * lda:r * lda + K] for r in range(M)])
        B2 = np.stack([B[k * ldb:k * ldb + N] for k in range(K)])
        ref, S = oracle_lib.gemm_sampled(A2, B2, rows, cols)
        tol.assert_close(C[rows, cols], ref, S, K, what)


def test_random_shapes_every_schedule(oracle_lib):
    from tests._gpu import dev_buffer
    seen = set()
    s = torch.cuda.current_stream().cuda_stream
    for i, (M, N, K, lda, ldb, ldc, (oa, ob, oc)) in enumerate(_cases()):
        A = synth.matrix(M, K, 500 + i, 0, ld=lda, pad_value=np.nan)
        B = synth.matrix(K, N, 500 + i, 1, ld=ldb, pad_value=np.nan)
        tA, pA = dev_buffer(A, oa)
        tB, pB = dev_buffer(B, ob)
        c_elems = (M - 1) * ldc + N
        tC = torch.full((c_elems + oc + 4,), float("nan"), device="cuda")
        pC = tC.data_ptr() + 4 * oc
        nbytes = sg.workspace_size(M, N, K)
        if i % 2 == 0:  # room for the copies (any size), else the narrow-copy kernels on unaligned rows
            nbytes += max(_r256(M * ((K + 3) // 4 * 4) * 4), _r256(K * ((M + 3) // 4 * 4) * 4))
            nbytes += _r256(K * ((N + 3) // 4 * 4) * 4)
        ws = torch.full((nbytes // 4,), 3, dtype=torch.int32, device="cuda")
        sst, kind, words = sg.ws_schedule(M, N, K, pA, lda, pB, ldb, pC, ldc, nbytes)
        assert sst == 0
        seen.add(kind & 3)
        seen |= {b for b in (4, 8, 16, 32) if kind & b}
        what = f"case {i}: {M}x{N}x{K} ld {lda},{ldb},{ldc} off {oa},{ob},{oc} kind {kind}"
        assert sg.sgemm_f32_ws(M, N, K, pA, lda, pB, ldb, pC, ldc, ws.data_ptr(), nbytes, s) == 0, what
        torch.cuda.synchronize()
        assert not ws[:words].any(), what
        raw = tC.cpu().numpy()[oc:oc + c_elems]
        C = np.stack([raw[r * ldc:r * ldc + N] for r in range(M)])
        _check(oracle_lib, A, B, C, M, N, K, lda, ldb, what, 500 + i)
        # the entry points without a workspace on the same operands: sgemm_f32
        # (one CTA per tile or the cluster split of K) and, every other case,
        # sgemm_f32_static_scratch (its fixed scratch for the flags)
        for name, fn in (("sgemm_f32", sg.sgemm_f32), ("static scratch", sg.sgemm_f32_static_scratch)):
            if name == "static scratch" and i % 2:
                continue
            tC.fill_(float("nan"))
            assert fn(M, N, K, pA, lda, pB, ldb, pC, ldc, s) == 0, what
            torch.cuda.synchronize()
            raw = tC.cpu().numpy()[oc:oc + c_elems]
            C = np.stack([raw[r * ldc:r * ldc + N] for r in range(M)])
            _check(oracle_lib, A, B, C, M, N, K, lda, ldb, f"{name} " + what, 500 + i)
        if i % 3 == 0:  # the tensor-core variant on the same operands
            tbytes = sg.tc_workspace_size(M, N, K)
            tws = torch.empty(max(tbytes, 256) + 256, dtype=torch.uint8, device="cuda")
            tw = (tws.data_ptr() + 255) // 256 * 256
            tC.fill_(float("nan"))
            assert sg.sgemm_f32_3xtf32(M, N, K, pA, lda, pB, ldb, pC, ldc, tw, tbytes, s) == 0, what
            torch.cuda.synchronize()
            raw = tC.cpu().numpy()[oc:oc + c_elems]
            C = np.stack([raw[r * ldc:r * ldc + N] for r in range(M)])
            _check(oracle_lib, A, B, C, M, N, K, lda, ldb, "3xTF32 " + what, 500 + i)
    assert {0, 1, 2, 3, 8, 16, 32} <= seen, f"schedules and copies seen: {sorted(seen)}"
    assert sg.copy_timeouts() == 0 and sg.tc_timeouts() == 0
