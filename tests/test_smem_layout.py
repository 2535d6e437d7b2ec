"""The kernel's shared-memory layout against the bank rule (CPU only).

The library reports, for every shared-memory instruction of its main loop,
the byte offset each lane touches -- computed by the same index functions the
kernel uses.  The oracle's bank model (bank = (byte_address / 4) % 32; a
conflict is the same bank at a different word, the same word is broadcast;
bank page, "地址怎样落到 bank", "四种访问，四种结果" and "为什么 double 和
float4 要另算") must find every one of them conflict-free: the passes it
needs equal the least its distinct words require.
"""
import pytest

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import build as sg_build

KINDS = {0: "A copy (16 B)", 1: "B copy (16 B)", 2: "A fragment read", 3: "B fragment read",
         4: "B copy (8 B)", 5: "B copy (4 B)", 6: "A copy (4 B)", 7: "A transpose read",
         8: "A transpose store", 11: "A fragment read (k-major copy of A, 8 x 16 tiles)",
         12: "B fragment read (k-major copy of A, 8 x 16 tiles)",
         13: "partial tile store (cluster split of K)", 14: "partial tile row read (cluster split of K)"}


@pytest.fixture(scope="module")
def lib():
    sg_build.build()
    return sg.load_library()


@pytest.mark.parametrize("kind", sorted(KINDS))
def test_every_access_conflict_free(lib, oracle_lib, kind):
    n_warps, n_steps, n_stages = sg.smem_shape(kind)
    for stage in range(n_stages):
        for warp in range(n_warps):
            for step in range(n_steps):
                offs, width = sg.smem_request(kind, warp, step, stage)
                r = oracle_lib.shared_request(offs, width)
                assert r["wavefronts"] == r["ideal"], (KINDS[kind], stage, warp, step, r)


TILE = 16 * 128


@pytest.mark.parametrize("kind", [0, 1, 4, 5, 6, 8])
def test_copies_and_stores_fill_each_tile_word_once(lib, kind):
    n_warps, n_steps, _ = sg.smem_shape(kind)
    words = []
    for warp in range(n_warps):
        for step in range(n_steps):
            offs, width = sg.smem_request(kind, warp, step, 0)
            for o in offs:
                words += [o // 4 + w for w in range(width // 4)]
    assert len(words) == TILE and len(set(words)) == TILE
    lo = min(words)
    assert max(words) - lo == TILE - 1  # one contiguous tile region


def test_transpose_reads_what_the_copies_wrote(lib):
    # the transpose reads every word of the raw A tile exactly once
    def region(kind):
        n_warps, n_steps, _ = sg.smem_shape(kind)
        out = []
        for warp in range(n_warps):
            for step in range(n_steps):
                offs, width = sg.smem_request(kind, warp, step, 0)
                out += [o // 4 + w for o in offs for w in range(width // 4)]
        return out
    copied = region(0)
    read = region(7)
    assert sorted(copied) == sorted(read) and len(set(read)) == TILE
    assert sorted(region(6)) == sorted(copied)


def test_fragment_reads_stay_inside_their_tile(lib):
    # A reads land in the As buffer the transpose stores fill, B reads in B's region
    def region(kind):
        n_warps, n_steps, _ = sg.smem_shape(kind)
        out = set()
        for warp in range(n_warps):
            for step in range(n_steps):
                offs, width = sg.smem_request(kind, warp, step, 0)
                out |= {o // 4 + w for o in offs for w in range(width // 4)}
        return out
    assert region(2) == region(8)
    assert region(3) == region(1)
    for kind in (2, 3):
        n_warps, n_steps, _ = sg.smem_shape(kind)
        for warp in range(n_warps):
            for step in range(n_steps):
                offs, _ = sg.smem_request(kind, warp, step, 0)
                assert all(o % 16 == 0 for o in offs)


def test_cluster_partial_tile_written_and_read_once(lib):
    # the stores of a CTA's 8 x 8 accumulators cover the 128 x 128 partial
    # tile word for word, and the row reads of the sum (all 128 rows) read
    # back exactly those words, 16 bytes at a time
    def words(kind):
        n_warps, n_steps, n_stages = sg.smem_shape(kind)
        assert n_stages == 1
        out = []
        for warp in range(n_warps):
            for step in range(n_steps):
                offs, width = sg.smem_request(kind, warp, step, 0)
                assert width == 16 and all(o % 16 == 0 for o in offs)
                out += [o // 4 + w for o in offs for w in range(4)]
        return out
    stored, read = words(13), words(14)
    assert len(stored) == 128 * 128 and sorted(stored) == list(range(128 * 128))
    assert sorted(read) == sorted(stored)
    # a row read covers exactly its row (words 128 r .. 128 r + 127)
    for warp in range(8):
        for step in range(16):
            offs, _ = sg.smem_request(14, warp, step, 0)
            row = 8 * step + warp
            assert sorted(o // 4 for o in offs) == list(range(128 * row, 128 * row + 128, 4))


def test_bad_query_rejected(lib):
    with pytest.raises(sg.SgemmError):
        sg.smem_request(9, 0, 0, 0)
    with pytest.raises(sg.SgemmError):
        sg.smem_request(15, 0, 0, 0)
    with pytest.raises(sg.SgemmError):
        sg.smem_request(0, 8, 0, 0)
