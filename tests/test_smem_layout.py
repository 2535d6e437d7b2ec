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

KINDS = {0: "A copy (4 B)", 1: "B copy (16 B)", 2: "A fragment read", 3: "B fragment read",
         4: "B copy (8 B)", 5: "B copy (4 B)"}


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


@pytest.mark.parametrize("kind,tile_words", [(0, 16 * 128), (1, 16 * 128), (4, 16 * 128), (5, 16 * 128)])
def test_copies_fill_each_tile_word_once(lib, kind, tile_words):
    n_warps, n_steps, _ = sg.smem_shape(kind)
    words = []
    for warp in range(n_warps):
        for step in range(n_steps):
            offs, width = sg.smem_request(kind, warp, step, 0)
            for o in offs:
                words += [o // 4 + w for w in range(width // 4)]
    assert len(words) == tile_words and len(set(words)) == tile_words


def test_fragment_reads_stay_inside_their_tile(lib):
    # A reads land in the A part of a stage, B reads in the B part
    a_words = set(range(0, 16 * 128))
    b_words = set(range(16 * 128, 2 * 16 * 128))
    for kind, region in ((2, a_words), (3, b_words)):
        n_warps, n_steps, _ = sg.smem_shape(kind)
        for warp in range(n_warps):
            for step in range(n_steps):
                offs, width = sg.smem_request(kind, warp, step, 0)
                assert all(o % 16 == 0 for o in offs)
                assert all(o // 4 + w in region for o in offs for w in range(4))


def test_bad_query_rejected(lib):
    with pytest.raises(sg.SgemmError):
        sg.smem_request(9, 0, 0, 0)
    with pytest.raises(sg.SgemmError):
        sg.smem_request(0, 8, 0, 0)
