"""The shared-memory stride sweep on the GPU (needs a GB300).

The bank page ("Memory Bank 机制与加速计算", "四种访问，四种结果") derives that
a warp whose lane l touches 32-bit word l * stride needs gcd(stride, 32)
passes, and its section "把推导变成测量" asks for that to be measured.
smem_bank_stride_probe runs the access pattern on one SM and times it with
the SM's cycle counter.  Checked here, for loads and stores and strides
1 .. 33:
  * every access touched the word it should (the checksum follows from the
    index formula alone, computed here independently of the kernel);
  * the cycles per warp-wide access follow the law: strides with the same
    gcd cost about the same, and the cost grows in proportion to gcd(stride,
    32) once the pipe, not instruction issue, is the bottleneck.
The ncu wavefront counts of the same pattern (one wavefront per pass) are
the golden fixture tests/golden/lds32_stride_sm103.txt.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg

pytestmark = pytest.mark.gpu

WARPS, ITERS = 8, 8192
STRIDES = list(range(1, 34))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


def _words(stride):
    lane = np.arange(32, dtype=np.int64)[:, None]
    u = np.arange(64, dtype=np.int64)[None, :]
    return lane * stride + 32 * u  # (lane, access u of a group of 64)


def _expected_checksum(stride, op):
    w = _words(stride)
    assert w.max() < 4096
    if op == "load":  # s[i] = i; every thread adds the words it reads, ITERS / 64 groups
        return int(WARPS * (ITERS // 64) * w.sum())
    written = np.unique(w)  # stores write each word's own index; the rest stay -1
    return int(written.sum() - (4096 - written.size))


@pytest.fixture(scope="module")
def sweep():
    out = {}
    for op in ("load", "store"):
        for s in STRIDES:
            out[op, s] = sg.bank_stride_probe(s, op, WARPS, ITERS)
    # the measured table (shown with pytest -s)
    print("\nstride gcd(stride,32) load_cycles_per_access store_cycles_per_access")
    for s in STRIDES:
        print(f"{s} {math.gcd(s, 32)} {out['load', s][0]:.3f} {out['store', s][0]:.3f}")
    return out


@pytest.mark.parametrize("op", ["load", "store"])
def test_every_access_touches_its_word(sweep, op):
    for s in STRIDES:
        _, chk = sweep[op, s]
        assert chk == _expected_checksum(s, op), (op, s)


@pytest.mark.parametrize("op", ["load", "store"])
def test_cycles_follow_the_gcd_law(sweep, op):
    cyc = {s: sweep[op, s][0] for s in STRIDES}
    by_g = {}
    for s in STRIDES:
        by_g.setdefault(math.gcd(s, 32), []).append(cyc[s])
    report = {g: [round(c, 2) for c in v] for g, v in sorted(by_g.items())}
    # strides with the same gcd cost the same, within 15 %
    for g, v in by_g.items():
        assert max(v) <= 1.15 * min(v), (op, g, report)
    mean = {g: sum(v) / len(v) for g, v in by_g.items()}
    gs = sorted(mean)
    # the cost rises with the conflict degree ...
    for a, b in zip(gs, gs[1:]):
        assert mean[b] > mean[a], (op, report)
    # ... in proportion to it where the shared-memory pipe is the bottleneck:
    # from degree 4 on, doubling the degree doubles the cycles (within 20 %)
    for a, b in zip(gs, gs[1:]):
        if a >= 4:
            assert 1.6 <= mean[b] / mean[a] <= 2.4, (op, a, b, report)
    # and a 32-way conflict costs 32 passes where one access costs about one
    assert mean[32] / mean[1] >= 16, (op, report)
