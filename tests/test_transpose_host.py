"""Transpose C ABI on the host (CPU only): argument checks, and the kernels'
shared-memory layouts against the bank model, including the pages' claim that
an unpadded 32 x 32 tile read down a column is a 32-way conflict while
[32][33] padding or the col ^ row swizzle removes it (bank page, "多一列" and
"Padding 之外的选择")."""
import pytest

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import build as sg_build

FAKE = 0x10000


@pytest.fixture(scope="module")
def lib():
    sg_build.build()
    return sg.load_library()


@pytest.mark.parametrize("args,code", [
    ((-1, 4, FAKE, 4, FAKE * 2, 4), -1),
    ((4, 5, FAKE, 4, FAKE * 2, 4), -2),        # ld_in < cols
    ((4, 5, FAKE, 5, FAKE * 2, 3), -2),        # ld_out < rows
    ((4, 5, 0, 5, FAKE * 2, 4), -3),
    ((4, 5, FAKE, 5, 0, 4), -3),
    ((4, 5, FAKE + 2, 5, FAKE * 2, 4), -7),
    ((4, 5, FAKE, 5, FAKE + 40, 4), -4),       # output overlaps the input's last row
    ((0, 5, 0, 5, 0, 1), 0),
])
def test_invalid_calls_rejected(lib, args, code):
    assert sg.transpose_f32(*args, 0) == code
    assert sg.transpose_f32(*args, 0, layout="padded") == code


def test_unknown_layout_rejected(lib):
    assert lib.transpose_f32_layout(4, 4, None, 4, None, 4, 9, None) == -7
    assert sg.transpose_status_string(-4) == "input and output overlap"


def _requests(layout, kind):
    n_steps = 16 if layout == "fast" or (layout == "fast_vec" and kind == 1) else 4
    for warp in range(8):
        for step in range(n_steps):
            yield sg.transpose_smem_request(layout, kind, warp, step)


@pytest.mark.parametrize("layout", ["padded", "swizzled", "fast", "fast_vec"])
@pytest.mark.parametrize("kind", [0, 1])
def test_conflict_free_layouts(lib, oracle_lib, layout, kind):
    for offs, width in _requests(layout, kind):
        r = oracle_lib.shared_request(offs, width)
        assert r["wavefronts"] == r["ideal"], (layout, kind, r)


def test_unpadded_column_reads_are_32_way(lib, oracle_lib):
    for offs, width in _requests("unpadded", 0):      # row writes: fine
        assert oracle_lib.shared_request(offs, width)["degree"] == 1
    for offs, width in _requests("unpadded", 1):      # column reads: 32 rows, one bank
        assert oracle_lib.shared_request(offs, width)["degree"] == 32


def test_tiles_are_bijections(lib):
    for layout, words in (("padded", 32 * 32), ("unpadded", 32 * 32), ("swizzled", 32 * 32), ("fast", 64 * 64),
                          ("fast_vec", 64 * 64)):
        for kind in (0, 1):
            seen = []
            for offs, width in _requests(layout, kind):
                seen += [o // 4 + w for o in offs for w in range(width // 4)]
            assert len(seen) == words and len(set(seen)) == words, (layout, kind)


def test_vector_tile_writes_are_128_bit(lib):
    for warp in range(8):
        for step in range(4):
            offs, width = sg.transpose_smem_request("fast_vec", 0, warp, step)
            assert width == 16 and all(o % 16 == 0 for o in offs)
