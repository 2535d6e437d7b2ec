"""C-ABI library: loads, exports what include/sgemm_f32.h declares, and
rejects invalid calls on the host before touching any GPU (CPU only)."""
import ctypes

import pytest

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import build as sg_build


@pytest.fixture(scope="module")
def lib():
    sg_build.build()
    return sg.load_library()


def test_exports_every_declared_symbol(lib):
    names = sg.declared_functions()
    assert {"sgemm_f32", "sgemm_f32_status_string", "sgemm_f32_smem_shape",
            "sgemm_f32_smem_request"} <= set(names)
    raw = ctypes.CDLL(sg_build.LIB)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = sg.status_string(code)
        assert s and s != "unknown status"
    assert sg.status_string(12345) == "unknown status"


# Every call below fails argument checks, which run before any CUDA call.
FAKE = 0x10000  # never dereferenced: the call returns before any launch


@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4), -1),
    ((4, -1, 4, FAKE, 4, FAKE, 4, FAKE, 4), -1),
    ((4, 4, -1, FAKE, 4, FAKE, 4, FAKE, 4), -1),
    ((4, 4, 8, FAKE, 7, FAKE, 4, FAKE, 4), -2),          # lda < K
    ((4, 5, 8, FAKE, 8, FAKE, 4, FAKE, 5), -2),          # ldb < N
    ((4, 5, 8, FAKE, 8, FAKE, 5, FAKE, 4), -2),          # ldc < N
    ((4, 4, 0, 0, 1, 0, 4, FAKE, 0), -2),                # ldc 0
    ((4, 4, 4, 0, 4, FAKE, 4, FAKE * 2, 4), -3),         # A null, K > 0
    ((4, 4, 4, FAKE, 4, 0, 4, FAKE * 2, 4), -3),         # B null, K > 0
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, 0, 4), -3),         # C null
    ((4, 4, 4, FAKE + 2, 4, FAKE * 2, 4, FAKE * 3, 4), -7),  # A not 4-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3 + 1, 4), -7),  # C not 4-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE + 16, 4), -4),     # C overlaps A
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 2 + 60, 4), -4), # C overlaps B's last element
])
def test_invalid_calls_rejected_on_host(lib, args, code):
    assert sg.sgemm_f32(*args, 0) == code


def test_adjacent_buffers_are_not_aliases(lib):
    # C starts right after B ends: not an overlap, so the call proceeds past the
    # alias check; with M=0 it then returns OK without launching.
    assert sg.sgemm_f32(0, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 2 + 64, 4, 0) == 0


def test_empty_outputs_are_noops(lib):
    assert sg.sgemm_f32(0, 5, 5, 0, 5, 0, 5, 0, 5, 0) == 0
    assert sg.sgemm_f32(5, 0, 5, 0, 5, 0, 1, 0, 1, 0) == 0


def test_torch_wrapper_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    with pytest.raises(TypeError):
        sg.sgemm(torch.ones(2, 2), torch.ones(2, 2))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from dense_fp32_tiled_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load_library()


def test_workspace_size(lib):
    assert sg.workspace_size(0, 5, 5) == 0 and sg.workspace_size(5, -1, 5) == 0
    # one flag per 128 x 128 tile plus an error word, rounded up to 256 bytes
    assert sg.workspace_size(4096, 4096, 4096) == ((32 * 32 + 1) * 4 + 255) // 256 * 256
    assert sg.workspace_size(129, 1, 7) == 256


@pytest.mark.parametrize("args,code", [
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 64), -3),           # NULL workspace, bytes > 0
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, FAKE * 4 + 8, 64), -7),  # workspace not 16-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, FAKE * 3 + 16, 64), -4),  # workspace overlaps C
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, FAKE + 48, 16), -4),     # workspace overlaps A
    ((4, 4, 4, FAKE, 3, FAKE * 2, 4, FAKE * 3, 4, FAKE * 4, 64), -2),      # usual checks still apply
    ((0, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 0), 0),               # empty: no-op
])
def test_workspace_call_rejected_on_host(lib, args, code):
    assert sg.sgemm_f32_ws(*args, 0) == code


# sgemm_f32_3xtf32: the same host checks, plus the workspace rules; all run
# before any CUDA call.  (The workspace-overlap check needs the workspace
# size, which depends on the device: it is tested on the GPU.)  Argument order: M, N, K, A, lda, B, ldb, C, ldc,
# workspace, workspace_bytes, stream.
WS = 0x100000  # 256-byte aligned, far from FAKE .. FAKE * 3


@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 20), -1),
    ((4, 4, 8, FAKE, 7, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 20), -2),      # lda < K
    ((4, 5, 8, FAKE, 8, FAKE * 2, 5, FAKE * 3, 4, WS, 1 << 20), -2),      # ldc < N
    ((4, 4, 4, 0, 4, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 20), -3),         # A null
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, 0, 4, WS, 1 << 20), -3),             # C null
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 1 << 20), -3),       # no workspace
    ((4, 4, 4, FAKE + 2, 4, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 20), -7),  # A not 4-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, WS + 16, 1 << 20), -7), # workspace not 256-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE + 16, 4, WS, 1 << 20), -4),     # C overlaps A
])
def test_tc_invalid_calls_rejected_on_host(lib, args, code):
    assert sg.sgemm_f32_3xtf32(*args, 0) == code


def test_tc_empty_product_is_a_no_op(lib):
    assert sg.sgemm_f32_3xtf32(0, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 0, 0) == 0
    assert sg.sgemm_f32_3xtf32(4, 0, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 0, 0) == 0


# sgemm_f32_host: host-side argument checks (same order as sgemm_f32's, then
# the device workspace); all return before any CUDA call.
@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 30), -1),
    ((4, 4, 8, FAKE, 7, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 30), -2),       # lda < K
    ((4, 4, 4, 0, 4, FAKE * 2, 4, FAKE * 3, 4, WS, 1 << 30), -3),          # A null
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 1 << 30), -3),        # no workspace
    ((4, 4, 4, FAKE, 4, FAKE * 2 + 2, 4, FAKE * 3, 4, WS, 1 << 30), -7),   # B not 4-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, WS + 64, 1 << 30), -7),  # workspace not 256-byte aligned
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 2 + 16, 4, WS, 1 << 30), -4),  # C overlaps B
    ((4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, WS, 16), -7),            # workspace too small
])
def test_host_invalid_calls_rejected_on_host(lib, args, code):
    assert sg.sgemm_f32_host(*args, 0) == code


def test_host_empty_product_is_a_no_op(lib):
    assert sg.sgemm_f32_host(0, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, 0, 0) == 0


def test_schedule_query_checks_arguments_on_host(lib):
    assert sg.ws_schedule(-1, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4) == (-1, 0, 0)
    assert sg.ws_schedule(4, 4, 8, FAKE, 7, FAKE * 2, 4, FAKE * 3, 4) == (-2, 0, 0)
    assert sg.ws_schedule(0, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4) == (0, 0, 0)
    assert lib.sgemm_f32_ws_schedule(4, 4, 4, FAKE, 4, FAKE * 2, 4, FAKE * 3, 4, 0, None, None) == -3


def test_bank_probe_rejects_bad_arguments_on_the_host(lib):
    # the checks come before any CUDA call, so this needs no GPU
    import ctypes
    cyc, chk = ctypes.c_double(), ctypes.c_longlong()
    probe = lib.smem_bank_stride_probe
    for args in [(0, 0, 8, 64), (65, 0, 8, 64), (1, 2, 8, 64), (1, 0, 0, 64), (1, 0, 9, 64), (1, 0, 8, 32),
                 (1, 0, 8, 100), (1, 0, 8, 65536 + 64)]:
        assert probe(*args, ctypes.byref(cyc), ctypes.byref(chk)) == -7, args
    assert probe(1, 0, 8, 64, None, ctypes.byref(chk)) == -3
    assert probe(1, 0, 8, 64, ctypes.byref(cyc), None) == -3
