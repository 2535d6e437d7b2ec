"""Pins for the oracle's shared-memory bank model (CPU only).

Against the examples the pages print (tests/golden/bank_examples.txt), the
gcd law stated on the bank page ("四种访问，四种结果": a full-warp scalar read
with stride s touches 32/gcd(s,32) banks with conflict degree gcd(s,32)),
the +1-padding and XOR-swizzle layouts of "多一列" / "Padding 之外的选择",
and the footprint example of "放进矩阵转置里看".
"""
import math
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    out = []
    with open(os.path.join(HERE, "golden", "bank_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("=")
            tag, kind, *args = lhs.split()
            out.append((tag, kind, " ".join(args), [int(x) for x in rhs.split()]))
    return out


def _eval_index(expr, lane):
    return eval(expr, {"__builtins__": {}}, {"lane": lane})


def test_golden_bank_examples(oracle_lib):
    cases = _golden()
    assert len(cases) >= 25
    for tag, kind, arg, expect in cases:
        if kind == "bank":
            assert oracle_lib.bank_of(int(arg)) == expect[0], (tag, arg)
        else:
            addrs = [4 * _eval_index(arg, l) for l in range(32)]
            r = oracle_lib.shared_request(addrs, 4)
            banks = {oracle_lib.bank_of(a) for a in addrs}
            assert (r["degree"], len(banks)) == tuple(expect), (tag, arg, r)


@pytest.mark.parametrize("stride", range(1, 65))
def test_gcd_law(oracle_lib, stride):
    for base in (0, 5):
        addrs = [4 * (base + l * stride) for l in range(32)]
        r = oracle_lib.shared_request(addrs, 4)
        g = math.gcd(stride, 32)
        assert r["degree"] == g
        assert len({oracle_lib.bank_of(a) for a in addrs}) == 32 // g


def test_padded_tile_rows_and_columns(oracle_lib):
    # tile[32][33]: bank = (row + col) % 32, row and column reads conflict-free
    for c in range(32):
        col = [4 * (r * 33 + c) for r in range(32)]
        assert oracle_lib.shared_request(col, 4)["degree"] == 1
        assert [oracle_lib.bank_of(a) for a in col] == [(r + c) % 32 for r in range(32)]
    for r in range(32):
        row = [4 * (r * 33 + c) for c in range(32)]
        assert oracle_lib.shared_request(row, 4)["degree"] == 1
    # tile[32][32]: column reads are 32-way
    assert oracle_lib.shared_request([4 * (r * 32 + 3) for r in range(32)], 4)["degree"] == 32
    # footprint: 32*32*4 = 4096 B vs 32*33*4 = 4224 B (+128 B)
    assert 32 * 32 * 4 == 4096 and 32 * 33 * 4 == 4224


def test_xor_swizzle_is_conflict_free_both_ways(oracle_lib):
    phys = lambda r, c: 4 * (r * 32 + (c ^ r))
    for r in range(32):
        assert sorted((c ^ r) for c in range(32)) == list(range(32))
        assert oracle_lib.shared_request([phys(r, c) for c in range(32)], 4)["degree"] == 1
    for c in range(32):
        assert oracle_lib.shared_request([phys(r, c) for r in range(32)], 4)["degree"] == 1


def test_measured_wide_load_wavefronts(oracle_lib):
    """The lane grouping of 8- and 16-byte loads, against ncu counts on sm_103."""
    n = 0
    with open(os.path.join(HERE, "golden", "lds_wavefronts_sm103.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("=")
            width, expr = lhs.split(None, 1)
            width = int(width)
            addrs = [width * _eval_index(expr.strip(), l) for l in range(32)]
            r = oracle_lib.shared_request(addrs, width)
            assert r["wavefronts"] == int(rhs.split()[0]), (width, expr, r)
            n += 1
    assert n == 52


def test_wide_accesses(oracle_lib):
    # 32 lanes reading consecutive float4: 512 distinct bytes -> 4 passes, all needed
    r = oracle_lib.shared_request([16 * l for l in range(32)], 16)
    assert (r["wavefronts"], r["ideal"], r["distinct"]) == (4, 4, 128)
    # every lane reading the same float4: one pass per half-warp
    r = oracle_lib.shared_request([48] * 32, 16)
    assert (r["wavefronts"], r["ideal"]) == (2, 2)
    # 8 distinct float4 covering 128 contiguous bytes, each quad of lanes
    # reading 4 of them: two passes per half
    r = oracle_lib.shared_request([16 * (l % 8) for l in range(32)], 16)
    assert (r["wavefronts"], r["ideal"]) == (4, 2)
    # the same 8 float4 with lanes paired inside each quad: one pass per half
    r = oracle_lib.shared_request([16 * (l >> 1) for l in range(16)] * 2, 16)
    assert (r["wavefronts"], r["ideal"]) == (2, 2)
    # float4 reads 512 B apart: same 4 banks, 8 distinct words per bank per quarter
    r = oracle_lib.shared_request([512 * l for l in range(32)], 16)
    assert r["wavefronts"] == 32 and r["ideal"] == 4 and r["degree"] == 8
    # doubles (8 B): consecutive -> 2 passes, no excess
    r = oracle_lib.shared_request([8 * l for l in range(32)], 8)
    assert (r["wavefronts"], r["ideal"]) == (2, 2)
    # inactive lanes do not count
    r = oracle_lib.shared_request([4 * 32 * l for l in range(32)], 4, active=[1] + [0] * 31)
    assert r["degree"] == 1 and r["wavefronts"] == 1
    with pytest.raises(ValueError):
        oracle_lib.shared_request([2], 4)


def test_measured_stride_sweep_matches_gcd_law_and_model(oracle_lib):
    """ncu on GB300: 32-bit loads and stores s[lane*stride], stride 1..33."""
    seen = set()
    with open(os.path.join(HERE, "golden", "lds32_stride_sm103.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("=")
            op, stride = lhs.split()
            stride = int(stride)
            wavefronts, conflicts = (int(x) for x in rhs.split())
            g = math.gcd(stride, 32)
            assert wavefronts == g and conflicts == g - 1, (op, stride)
            r = oracle_lib.shared_request([4 * (l * stride) for l in range(32)], 4)
            assert r["wavefronts"] == wavefronts
            seen.add((op, stride))
    assert seen == {(op, s) for op in ("lds32", "sts32") for s in range(1, 34)}


def _heldout():
    import sys
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import lds_heldout_patterns as P
    measured = {}
    with open(os.path.join(HERE, "golden", "lds_wavefronts_heldout_sm103.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, val = line.rsplit("=", 1)
                measured[name.strip()] = int(val)
    return P, measured


def test_heldout_wide_load_wavefronts(oracle_lib):
    # patterns chosen after the wide-access rule was fitted (new permutations,
    # strided and broadcast mixes, and the product kernels' own fragment
    # reads, as the library reports them); the unchanged rule must predict
    # every measured count
    pytest.importorskip("ctypes")
    from dense_fp32_tiled_gb300 import build as sg_build
    import dense_fp32_tiled_gb300 as sg
    sg_build.build()
    sg.load_library()
    P, measured = _heldout()
    pats = P.patterns()
    assert len(pats) == len(measured) >= 30
    widths = {w for _, w, _ in pats}
    assert widths == {4, 8, 16}
    for name, width, words in pats:
        r = oracle_lib.shared_request([4 * x for x in words], width)
        assert r["wavefronts"] == measured[name], (name, r, measured[name])


def test_heldout_patterns_are_new():
    # none of the held-out expressions is one of the fitted ones
    P, _ = _heldout()
    fitted = set()
    with open(os.path.join(HERE, "golden", "lds_wavefronts_sm103.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                w, expr = line.split("=")[0].split(None, 1)
                fitted.add((int(w), expr.strip().replace(" ", "")))
    for w, e in P.WIDE + P.NARROW:
        assert (w, e.replace(" ", "")) not in fitted, (w, e)
