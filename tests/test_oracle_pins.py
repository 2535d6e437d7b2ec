"""Pins for the FP64 oracle's matrix product (CPU only).

Each check fixes the oracle against something other than itself: values
worked by hand, closed forms (ones, identities), numpy's float64 matmul,
exact rational brute force, structural identities, and planted mistakes that
the acceptance test must reject.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from dense_fp32_tiled_gb300 import synth
from tests import _tolerance as tol

HERE = os.path.dirname(os.path.abspath(__file__))


def _read_small_golden():
    blocks, cur, name, rows = [], {}, None, []
    with open(os.path.join(HERE, "golden", "gemm_small.txt")) as f:
        lines = [l.strip() for l in f if l.strip() and not l.startswith("#")]
    i = 0
    while i < len(lines):
        tag, r, c = lines[i].split()
        r, c = int(r), int(c)
        mat = np.array([[float(x) for x in lines[i + 1 + q].split()] for q in range(r)])
        assert mat.shape == (r, c)
        cur[tag] = mat
        i += 1 + r
        if tag == "C":
            blocks.append(cur)
            cur = {}
    return blocks


def test_golden_small_products(oracle_lib):
    blocks = _read_small_golden()
    assert len(blocks) == 4
    for b in blocks:
        C, S = oracle_lib.gemm(b["A"].astype(np.float32), b["B"].astype(np.float32))
        np.testing.assert_array_equal(C, b["C"])
        np.testing.assert_array_equal(S, np.abs(b["A"]) @ np.abs(b["B"]))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (64, 33, 129), (17, 1, 300), (5, 6, 0)])
def test_ones_give_K(oracle_lib, M, N, K):
    C, S = oracle_lib.gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
    assert np.all(C == K) and np.all(S == K)


def test_identity(oracle_lib):
    B = synth.matrix(37, 53, seed=11, matrix_id=1)
    C, _ = oracle_lib.gemm(np.eye(37, dtype=np.float32), B)
    np.testing.assert_array_equal(C, B.astype(np.float64))
    A = synth.matrix(29, 37, seed=11, matrix_id=0)
    C, _ = oracle_lib.gemm(A, np.eye(37, dtype=np.float32))
    np.testing.assert_array_equal(C, A.astype(np.float64))


@pytest.mark.parametrize("M,N,K,kind", [(1, 1, 1, "uniform"), (7, 9, 11, "normal"),
                                        (130, 67, 258, "uniform"), (64, 128, 1000, "normal")])
def test_matches_numpy_float64(oracle_lib, M, N, K, kind):
    A = synth.matrix(M, K, 5, 0, kind)
    B = synth.matrix(K, N, 5, 1, kind)
    C, S = oracle_lib.gemm(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    sref = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    # different summation order: FP64 rounding only
    assert np.all(np.abs(C - ref) <= 64 * K * 2.0 ** -53 * sref + 1e-300)
    np.testing.assert_allclose(S, sref, rtol=64 * K * 2.0 ** -53)


def test_exact_rational_brute_force(oracle_lib):
    # dyadic inputs with few significant bits: every partial sum is exact in FP64
    rng = np.random.default_rng(7)
    A = (rng.integers(-64, 64, size=(4, 6)) / 16.0).astype(np.float32)
    B = (rng.integers(-64, 64, size=(6, 5)) / 8.0).astype(np.float32)
    C, _ = oracle_lib.gemm(A, B)
    for i in range(4):
        for j in range(5):
            exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(6))
            assert Fraction(C[i, j]) == exact


def test_transpose_identity(oracle_lib):
    A = synth.matrix(23, 41, 9, 0, "normal")
    B = synth.matrix(41, 17, 9, 1, "normal")
    C, _ = oracle_lib.gemm(A, B)
    Ct, _ = oracle_lib.gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))
    np.testing.assert_array_equal(C, Ct.T)


def test_column_locality(oracle_lib):
    # column j of C depends only on column j of B
    A = synth.matrix(19, 31, 3, 0)
    B = synth.matrix(31, 12, 3, 1)
    C, _ = oracle_lib.gemm(A, B)
    B2 = B.copy()
    B2[:, 5] += 1.0
    C2, _ = oracle_lib.gemm(A, B2)
    changed = np.any(C != C2, axis=0)
    assert changed[5] and changed.sum() == 1


def test_leading_dimensions_and_poisoned_padding(oracle_lib):
    M, N, K, lda, ldb = 13, 10, 9, 12, 15
    Ad = synth.matrix(M, K, 21, 0)
    Bd = synth.matrix(K, N, 21, 1)
    Af = synth.matrix(M, K, 21, 0, ld=lda, pad_value=np.nan)
    Bf = synth.matrix(K, N, 21, 1, ld=ldb, pad_value=np.nan)
    C1, S1 = oracle_lib.gemm(Ad, Bd)
    C2, S2 = oracle_lib.gemm(Af, Bf, M=M, N=N, K=K, lda=lda, ldb=ldb)
    assert not np.isnan(C2).any()
    np.testing.assert_array_equal(C1, C2)
    np.testing.assert_array_equal(S1, S2)


def test_sampled_matches_full(oracle_lib):
    M, N, K = 70, 90, 33
    A = synth.matrix(M, K, 2, 0)
    B = synth.matrix(K, N, 2, 1)
    C, S = oracle_lib.gemm(A, B)
    r, c = synth.sample_indices(M, N, 200, seed=2, tile_m=32, tile_n=32)
    v, s = oracle_lib.gemm_sampled(A, B, r, c)
    np.testing.assert_array_equal(v, C[r, c])
    np.testing.assert_array_equal(s, S[r, c])


def test_nan_propagates_along_its_row(oracle_lib):
    A = synth.matrix(6, 5, 1, 0)
    B = synth.matrix(5, 4, 1, 1)
    A[2, 3] = np.nan
    C, _ = oracle_lib.gemm(A, B)
    assert np.isnan(C[2]).all() and not np.isnan(np.delete(C, 2, axis=0)).any()


def test_rejects_bad_arguments(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm(np.zeros(10, np.float32), np.zeros(10, np.float32), M=2, N=2, K=3, lda=2, ldb=2)


# ---- the acceptance test itself: honest FP32 passes, planted mistakes fail ----

def _fp32_sequential(A, B):
    acc = np.zeros((A.shape[0], B.shape[1]), np.float32)
    for k in range(A.shape[1]):
        acc = (acc + A[:, k:k + 1] * B[k:k + 1, :]).astype(np.float32)
    return acc


@pytest.mark.parametrize("kind", ["uniform", "normal"])
def test_fp32_sequential_and_blas_pass(oracle_lib, kind):
    M, N, K = 48, 40, 777
    A = synth.matrix(M, K, 8, 0, kind)
    B = synth.matrix(K, N, 8, 1, kind)
    C, S = oracle_lib.gemm(A, B)
    tol.assert_close(_fp32_sequential(A, B), C, S, K, "fp32 sequential sum")
    tol.assert_close(A @ B, C, S, K, "numpy float32 matmul")


def test_planted_mistakes_are_rejected(oracle_lib):
    M, N, K = 40, 36, 300
    A = synth.matrix(M, K, 4, 0)
    B = synth.matrix(K, N, 4, 1)
    C, S = oracle_lib.gemm(A, B)
    # dropped last k term
    A_drop = A.copy()
    A_drop[:, -1] = 0
    bad, _ = oracle_lib.gemm(A_drop, B)
    assert not tol.check(bad.astype(np.float32), C, S, K)[0]
    # wrong sign of one term
    A_sign = A.copy()
    A_sign[:, 17] *= -1
    bad, _ = oracle_lib.gemm(A_sign, B)
    assert not tol.check(bad.astype(np.float32), C, S, K)[0]
    # transposed operand (square case)
    Asq = synth.matrix(64, 64, 4, 2)
    Bsq = synth.matrix(64, 64, 4, 3)
    Csq, Ssq = oracle_lib.gemm(Asq, Bsq)
    bad, _ = oracle_lib.gemm(np.ascontiguousarray(Asq.T), Bsq)
    assert not tol.check(bad.astype(np.float32), Csq, Ssq, 64)[0]
    # off-by-one row shift
    bad = np.roll(C, 1, axis=0)
    assert not tol.check(bad.astype(np.float32), C, S, K)[0]
    # K == 0: only exact zeros pass
    Z, SZ = oracle_lib.gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert tol.check(np.zeros((3, 4), np.float32), Z, SZ, 0)[0]
    assert not tol.check(np.full((3, 4), 1e-30, np.float32), Z, SZ, 0)[0]


def test_bit_exact_integer_inputs_any_order(oracle_lib):
    # entries in {-2..2}: every FP32 partial sum stays below 2**24 for K <= 8192,
    # so any summation order reproduces the FP64 value exactly
    M, N, K = 20, 24, 2048
    A = synth.matrix(M, K, 6, 0, "int5")
    B = synth.matrix(K, N, 6, 1, "int5")
    C, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(_fp32_sequential(A, B).astype(np.float64), C)
    np.testing.assert_array_equal((A @ B).astype(np.float64), C)
