"""Pins for the oracle's transpose (CPU only): a hand-worked case, numpy's
transpose, bit preservation (NaN payloads, signed zeros), strided buffers."""
import os

import numpy as np
import pytest

from dense_fp32_tiled_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_golden_small(oracle_lib):
    lines = [l.split() for l in open(os.path.join(HERE, "golden", "transpose_small.txt"))
             if l.strip() and not l.startswith("#")]
    assert lines[0][:1] == ["IN"] and lines[3][:1] == ["OUT"]
    X = np.array([[float(v) for v in r] for r in lines[1:3]], np.float32)
    Y = np.array([[float(v) for v in r] for r in lines[4:7]], np.float32)
    np.testing.assert_array_equal(oracle_lib.transpose(X), Y)


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 7), (7, 1), (33, 65), (128, 96)])
def test_matches_numpy(oracle_lib, rows, cols):
    X = synth.matrix(rows, cols, 3, 0, "normal")
    np.testing.assert_array_equal(oracle_lib.transpose(X), X.T)


def test_bits_are_preserved(oracle_lib):
    X = synth.matrix(5, 6, 1, 0).copy()
    bits = X.view(np.uint32)
    bits[1, 2] = 0x7FC01234  # NaN with a payload
    bits[3, 4] = 0x80000000  # -0.0
    bits[0, 5] = 0x00000001  # smallest denormal
    Y = oracle_lib.transpose(X)
    np.testing.assert_array_equal(Y.view(np.uint32), X.view(np.uint32).T)


def test_strided_buffers(oracle_lib):
    rows, cols, ld_in, ld_out = 9, 13, 17, 11
    flat = synth.matrix(rows, cols, 2, 0, ld=ld_in, pad_value=-5.0)
    out = np.full((cols - 1) * ld_out + rows, 7.0, dtype=np.float32)
    oracle_lib.transpose(flat, rows=rows, cols=cols, ld_in=ld_in, ld_out=ld_out, out=out)
    dense = synth.matrix(rows, cols, 2, 0)
    for j in range(cols):
        np.testing.assert_array_equal(out[j * ld_out:j * ld_out + rows], dense[:, j])
        if j < cols - 1:
            assert np.all(out[j * ld_out + rows:(j + 1) * ld_out] == 7.0)


def test_rejects_bad_arguments(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.transpose(np.zeros(10, np.float32), rows=2, cols=5, ld_in=4, ld_out=2)
