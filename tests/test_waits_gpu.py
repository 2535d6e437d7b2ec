"""Failure detection without a GPU fault (needs a GB300).

Every wait in the library's kernels is bounded: the copy-ring mbarrier waits
and the stream-K partner-flag waits of the CUDA-core kernels, and the
tensor-core pipeline's mbarrier waits.  A wait that runs out records a flag
and returns; nothing traps or hangs.  The self-test entry points run those
same wait routines, in a one-CTA kernel with a short limit, on a target
nothing completes (an mbarrier phase with no arrival, a flag nobody raises):
the wait must give up and the kernel must return normally.  On a target
already complete the wait must not give up.  Afterwards the context must
still run products correctly, and the production timeout flags stay clear.
"""
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
from tests import _tolerance as tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


@pytest.mark.parametrize("case", ["copy_never", "flag_never", "tc_never"])
def test_wait_on_nothing_gives_up_and_returns(case):
    assert sg.wait_selftest(case, polls=1000) is True


@pytest.mark.parametrize("case", ["copy_done", "flag_done", "tc_done"])
def test_wait_on_completed_target_does_not_give_up(case):
    assert sg.wait_selftest(case, polls=1000) is False


def test_limits_are_checked():
    lib = sg.load_library()
    import ctypes
    n = ctypes.c_uint()
    assert lib.sgemm_f32_wait_selftest(0, 0, ctypes.byref(n)) == -7
    assert lib.sgemm_f32_wait_selftest(0, 1 << 17, ctypes.byref(n)) == -7
    assert lib.sgemm_f32_wait_selftest(4, 10, ctypes.byref(n)) == -7
    assert lib.sgemm_f32_3xtf32_wait_selftest(2, 10, ctypes.byref(n)) == -7
    assert lib.sgemm_f32_wait_selftest(0, 10, None) == -3


def test_context_usable_and_flags_clear_after_timeouts(oracle_lib):
    for case in ("copy_never", "flag_never", "tc_never"):
        assert sg.wait_selftest(case, polls=500)
    M, N, K = 700, 900, 300
    A = synth.matrix(M, K, 341, 0)
    B = synth.matrix(K, N, 341, 1)
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    Cr, Sr = oracle_lib.gemm(A, B)
    for fn in (sg.sgemm, sg.sgemm_tc):
        C = fn(tA, tB)
        torch.cuda.synchronize()
        tol.assert_close(C.cpu().numpy(), Cr, Sr, K, fn.__name__)
    assert sg.copy_timeouts() == 0
    assert sg.tc_timeouts() == 0
