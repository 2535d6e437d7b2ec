"""transpose_f32 and transpose_f32_layout vs the oracle's transpose: bit-exact
(needs a GB300)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth

pytestmark = pytest.mark.gpu

LAYOUTS = [None, "padded", "unpadded", "swizzled"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


def _run(x_flat, rows, cols, ld_in, ld_out, layout, in_off=0, out_off=0, fill=-3.0):
    from tests._gpu import dev_buffer
    t_in, p_in = dev_buffer(x_flat, in_off)
    n_out = (cols - 1) * ld_out + rows
    t_out = torch.full((n_out + out_off + 4,), fill, dtype=torch.float32, device="cuda")
    st = sg.transpose_f32(rows, cols, p_in, ld_in, t_out.data_ptr() + 4 * out_off, ld_out,
                          torch.cuda.current_stream().cuda_stream, layout=layout)
    torch.cuda.synchronize()
    return st, t_out.cpu().numpy()[out_off:out_off + n_out]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 7), (7, 1), (33, 65), (64, 64), (1000, 1030), (4097, 129),
                                       (129, 4097)])
def test_bit_exact(oracle_lib, layout, rows, cols):
    x = synth.matrix(rows, cols, 51, 0, "normal", ld=cols)
    st, got = _run(x, rows, cols, cols, rows, layout)
    assert st == 0
    ref = oracle_lib.transpose(x.reshape(rows, cols))
    np.testing.assert_array_equal(got.view(np.uint32), ref.reshape(-1).view(np.uint32))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("in_off,out_off,pad_in,pad_out", [(0, 0, 4, 8), (1, 0, 3, 0), (0, 2, 0, 5), (3, 1, 7, 9)])
def test_strides_offsets_padding_untouched(oracle_lib, layout, in_off, out_off, pad_in, pad_out):
    rows, cols = 301, 257
    ld_in, ld_out = cols + pad_in, rows + pad_out
    x = synth.matrix(rows, cols, 53, 0, ld=ld_in, pad_value=np.nan)
    st, got = _run(x, rows, cols, ld_in, ld_out, layout, in_off, out_off, fill=-3.0)
    assert st == 0
    ref = np.full((cols - 1) * ld_out + rows, -3.0, dtype=np.float32)
    oracle_lib.transpose(x, rows=rows, cols=cols, ld_in=ld_in, ld_out=ld_out, out=ref)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_special_values_keep_their_bits(oracle_lib):
    rows, cols = 70, 90
    x = synth.matrix(rows, cols, 55, 0).copy()
    b = x.view(np.uint32)
    b[3, 4], b[5, 6], b[7, 8], b[9, 10] = 0x7FC0ABCD, 0xFF800000, 0x80000000, 0x00000003
    for layout in LAYOUTS:
        st, got = _run(x.reshape(-1), rows, cols, cols, rows, layout)
        assert st == 0
        np.testing.assert_array_equal(got.view(np.uint32), oracle_lib.transpose(x).reshape(-1).view(np.uint32))


def test_large_full_check(oracle_lib):
    rows, cols = 8192, 6144
    x = synth.matrix(rows, cols, 57, 0)
    tx = torch.from_numpy(x).cuda()
    y = sg.transpose(tx)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y.cpu().numpy().view(np.uint32), oracle_lib.transpose(x).view(np.uint32))


def test_alias_rejected_with_device_pointers():
    t = torch.zeros(64 * 64 * 2, device="cuda")
    p = t.data_ptr()
    assert sg.transpose_f32(64, 64, p, 64, p + 4 * 100, 64, 0) == -4


@pytest.mark.parametrize("rows,cols,ld_in,ld_out,in_off,out_off", [
    (4, 4, 4, 4, 0, 0), (64, 64, 64, 64, 0, 0), (68, 132, 132, 68, 0, 0), (1000, 1032, 1036, 1004, 4, 8),
    (4096, 260, 264, 4100, 0, 4), (260, 4096, 4096, 260, 8, 0)])
def test_vector_path_bit_exact(oracle_lib, rows, cols, ld_in, ld_out, in_off, out_off):
    """16-byte aligned rows, sizes multiples of 4: transpose_f32 takes the
    16-byte vector kernel (swizzled tile), ragged edge tiles included, and
    leaves the padding of both matrices untouched."""
    x = synth.matrix(rows, cols, 59, 0, "normal", ld=ld_in, pad_value=np.nan)
    st, got = _run(x, rows, cols, ld_in, ld_out, None, in_off, out_off, fill=-3.0)
    assert st == 0
    ref = np.full((cols - 1) * ld_out + rows, -3.0, dtype=np.float32)
    oracle_lib.transpose(x, rows=rows, cols=cols, ld_in=ld_in, ld_out=ld_out, out=ref)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
