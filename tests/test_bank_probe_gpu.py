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
the golden fixture tests/golden/lds32_stride_sm103.txt.  The pattern probe
does the same for any 32-lane load pattern of 4, 8 or 16 bytes: its cycles
per load must equal the passes the oracle's bank model predicts, for every
pattern measured with ncu (the fitted and the held-out golden sets).
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
    # one pass per SM clock: a warp-wide access with lane stride s costs
    # gcd(s, 32) cycles when the shared-memory pipe is the bottleneck, which
    # the probe's volatile accesses (one instruction each, no merging) make it
    cyc = {s: sweep[op, s][0] for s in STRIDES}
    for s in STRIDES:
        g = math.gcd(s, 32)
        assert 0.9 * g <= cyc[s] <= 1.1 * g, (op, s, g, round(cyc[s], 3))
    # and strides with the same gcd cost the same, within 5 %
    by_g = {}
    for s in STRIDES:
        by_g.setdefault(math.gcd(s, 32), []).append(cyc[s])
    for g, v in by_g.items():
        assert max(v) <= 1.05 * min(v), (op, g, v)


def _patterns():
    """(name, width, lane words) of every measured pattern: the held-out set
    and the set the oracle's wide-access rule was fitted to."""
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import lds_heldout_patterns as P
    out = list(P.patterns())
    with open(os.path.join(here, "lds_wavefronts_sm103.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                w, expr = line.split("=")[0].split(None, 1)
                w = int(w)
                out.append((f"fitted {w} {expr.strip()}", w, P.lane_words_expr(w, expr.strip())))
    return out


def test_pattern_cycles_equal_the_bank_model(oracle_lib):
    # the SM clock counts one cycle per pass for any width (measured), so the
    # oracle's bank model, which predicts the passes of a warp-wide access
    # from its lane addresses alone, must predict the cycles of every pattern;
    # the checksum shows that every lane read the words it should
    pats = _patterns()
    assert len(pats) >= 80
    bad = []
    for name, width, words in pats:
        cyc, chk = sg.bank_pattern_probe(width, words, WARPS, ITERS)
        expect_chk = WARPS * (ITERS // 64) * sum(64 * w + 32 * 2016 for w in words)
        assert chk == expect_chk, name
        model = oracle_lib.shared_request([4 * w for w in words], width)["wavefronts"]
        if not 0.9 * model <= cyc <= 1.1 * model:
            bad.append((name, model, round(cyc, 3)))
    assert not bad, bad
