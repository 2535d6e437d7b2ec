"""Seeded synthetic inputs for the FP32 matrix multiply (no GEMM arithmetic here).

Both the CUDA path's tests/benchmark and the FP64 oracle receive matrices made
by this module, so the two sides see identical bits.  Random numbers come from
a counter-based SplitMix64 stream (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014: the 64-bit finaliser with
increment 0x9E3779B97F4A7C15), one stream per (seed, matrix id):

    key       = mix64((seed << 16) ^ matrix_id)
    draw(i)   = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)      (mod 2**64)

Matrices are filled in row-major order of their logical elements.

* uniform[-1, 1):  ((draw >> 40) - 2**23) / 2**23, exact in FP32.
* normal(0, sigma): Box-Muller on draws 2i and 2i+1 in FP64,
  u1 = ((d0 >> 11) + 1) / 2**53, u2 = (d1 >> 11) / 2**53,
  z = sqrt(-2 ln u1) cos(2 pi u2), then sigma * z rounded to FP32.
* integers in {-2, ..., 2}: ((draw >> 32) % 5) - 2, exact in FP32.

The named workloads below are the shapes and value distributions the tiled
matrix multiply is tested and measured on.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, matrix_id: int) -> np.uint64:
    x = np.array([((int(seed) << 16) ^ int(matrix_id)) & (2**64 - 1)], dtype=np.uint64)
    return _mix64(x)[0]


def draws(key: np.uint64, start: int, count: int) -> np.ndarray:
    """draw(start), ..., draw(start + count - 1) of the stream with ``key``."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + i * _GAMMA)


def _fill(n: int, key: np.uint64, kind: str, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        if kind == "uniform":
            d = draws(key, s, c)
            out[s:s + c] = ((d >> np.uint64(40)).astype(np.int64) - (1 << 23)).astype(np.float32) \
                * np.float32(2.0 ** -23)
        elif kind == "normal":
            d = draws(key, 2 * s, 2 * c)
            u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
            u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
            z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
            out[s:s + c] = (sigma * z).astype(np.float32)
        elif kind == "int5":
            d = draws(key, s, c)
            out[s:s + c] = (((d >> np.uint64(32)) % np.uint64(5)).astype(np.int64) - 2).astype(np.float32)
        else:
            raise ValueError(f"unknown distribution {kind!r}")
    return out


def matrix(rows: int, cols: int, seed: int, matrix_id: int, kind: str = "uniform",
           sigma: float = 1.0, ld: int | None = None, pad_value: float = 0.0) -> np.ndarray:
    """A rows x cols float32 matrix from stream (seed, matrix_id).

    With ``ld`` (>= cols) the result is a flat buffer of (rows-1)*ld + cols
    elements in which row r starts at r*ld; the gaps hold ``pad_value``.
    Without it the result is a dense 2-D array.
    """
    key = stream_key(seed, matrix_id)
    vals = _fill(rows * cols, key, kind, sigma)
    if ld is None:
        return vals.reshape(rows, cols)
    assert ld >= max(1, cols)
    n = 0 if rows == 0 or cols == 0 else (rows - 1) * ld + cols
    buf = np.full(n, pad_value, dtype=np.float32)
    for r in range(rows):
        buf[r * ld:r * ld + cols] = vals[r * cols:(r + 1) * cols]
    return buf


def sample_indices(M: int, N: int, count: int, seed: int, tile_m: int = 128, tile_n: int = 128):
    """Seeded output positions for sampled checks of large products.

    ``count`` positions drawn uniformly over M x N from stream (seed ^ 0xC0FFEE, 0),
    followed by the four corners and the last row and column of the final
    (bottom-right) output tile.
    """
    key = stream_key(seed ^ 0xC0FFEE, 0)
    d = draws(key, 0, count) % np.uint64(M * N)
    flat = d.astype(np.int64)
    rows, cols = list(flat // N), list(flat % N)
    forced = [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]
    r0 = ((M - 1) // tile_m) * tile_m
    c0 = ((N - 1) // tile_n) * tile_n
    forced += [(M - 1, j) for j in range(c0, N)] + [(i, N - 1) for i in range(r0, M)]
    for i, j in forced:
        rows.append(i)
        cols.append(j)
    return np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64)


@dataclass(frozen=True)
class Workload:
    """One FP32 matrix-multiply case: shapes, strides, input recipe, check mode."""
    name: str
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    kind: str
    sigma: float
    seed: int
    ids: tuple  # stream ids of (A, B)
    check: str  # "full" or "sampled"

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def inputs(self, ld_buffers: bool = False):
        """(A, B) as float32 arrays: dense 2-D, or flat buffers with the workload's
        leading dimensions when ``ld_buffers``."""
        A = matrix(self.M, self.K, self.seed, self.ids[0], self.kind, self.sigma,
                   ld=self.lda if ld_buffers else None)
        B = matrix(self.K, self.N, self.seed, self.ids[1], self.kind, self.sigma,
                   ld=self.ldb if ld_buffers else None)
        return A, B


def _w(name, M, N, K, kind, sigma, seed, ids=(0, 1), check="full", lda=None, ldb=None, ldc=None):
    return Workload(name, M, N, K, lda or K, ldb or N, ldc or N, kind, sigma, seed, ids, check)


WORKLOADS = {
    w.name: w for w in [
        _w("sgemm_256x256x256_uniform", 256, 256, 256, "uniform", 1.0, 0),
        _w("sgemm_1024x1024x1024_normal", 1024, 1024, 1024, "normal", 1.0, 1),
        _w("sgemm_1000x1030x777_ragged_uniform", 1000, 1030, 777, "uniform", 1.0, 2),
        _w("sgemm_4096x4096x4096_uniform", 4096, 4096, 4096, "uniform", 1.0, 3, check="sampled"),
        _w("sgemm_16384x256x4096_normal", 16384, 256, 4096, "normal", 0.5, 4, check="sampled"),
        _w("sgemm_8192x8192x8192_normal", 8192, 8192, 8192, "normal", 0.5, 4, ids=(2, 3), check="sampled"),
    ]
}

HEADLINE = "sgemm_4096x4096x4096_uniform"
