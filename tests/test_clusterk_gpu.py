"""The cluster split of K vs the FP64 oracle (needs a GB300).

Products with at most G / 2 output tiles (G = 2 CTAs per SM) run each tile
on a thread-block cluster of S CTAs (2 <= S <= 16; above 8 where the GPU
schedules such clusters), each CTA summing a slice of K, the slices added in
rank order through distributed shared memory.
sgemm_f32 (no workspace) takes it whenever it applies; sgemm_f32_ws takes it
unless its cost model expects the multi-part split to be faster.
sgemm_f32_ws_schedule reports it as bit 32 with S in bits 8 and up and no
workspace words, and with a workspace of 0 bytes it reports what sgemm_f32
runs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
from tests import _tolerance as tol
from tests._gpu import dev_buffer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()


def _tiles(M, N):
    return ((M + 127) // 128) * ((N + 127) // 128)


_PTRS = (1 << 36, 2 << 36, 3 << 36)  # host-only schedule queries: never dereferenced


def _max_cluster():
    """The largest cluster the library uses on this GPU (16 where the GPU
    schedules clusters of 16 of its CTAs, else 8): the size it reports for a
    single tile with a deep K."""
    sst, kind, _ = sg.ws_schedule(128, 128, 4096, *_PTRS[:1], 4096, _PTRS[1], 128, _PTRS[2], 128, 0)
    assert sst == 0 and kind & 32
    return kind >> 8


def _cluster_bound(M, N, K):
    """The largest S the library may pick without a workspace: the most CTAs
    per tile that fit the resident CTAs, at most half the 16-deep K tiles,
    and at most 8, or the largest cluster when T such clusters take at most
    a quarter of the resident CTAs.  It picks less where the GPU cannot hold
    T clusters of that size at once (each must fit in one GPC)."""
    G = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    T, big = _tiles(M, N), _max_cluster()
    return min(G // T, big if 4 * T * big <= G else 8, (K + 15) // 16 // 2)


def _run(M, N, K, A, lda, B, ldb, ldc, offs=(0, 0, 0), nbytes=0, ws_fill=7):
    """One call (sgemm_f32 when nbytes == 0, else sgemm_f32_ws); returns C
    (M x N), the raw C buffer with its padding, the workspace words and the
    reported schedule."""
    tA, pA = dev_buffer(A, offs[0])
    tB, pB = dev_buffer(B, offs[1])
    c_elems = (M - 1) * ldc + N
    tC = torch.full((c_elems + offs[2] + 4,), float("nan"), device="cuda")
    pC = tC.data_ptr() + 4 * offs[2]
    sst, kind, words = sg.ws_schedule(M, N, K, pA, lda, pB, ldb, pC, ldc, nbytes)
    assert sst == 0
    s = torch.cuda.current_stream().cuda_stream
    ws = None
    if nbytes:
        ws = torch.full((nbytes // 4,), ws_fill, dtype=torch.int32, device="cuda")
        st = sg.sgemm_f32_ws(M, N, K, pA, lda, pB, ldb, pC, ldc, ws.data_ptr(), nbytes, s)
    else:
        st = sg.sgemm_f32(M, N, K, pA, lda, pB, ldb, pC, ldc, s)
    torch.cuda.synchronize()
    assert st == 0, sg.status_string(st)
    raw = tC.cpu().numpy()
    body = raw[offs[2]:offs[2] + c_elems]
    C = np.stack([body[i * ldc:i * ldc + N] for i in range(M)])
    return C, raw, (ws.cpu().numpy() if ws is not None else None), kind, words


def _padding_untouched(raw, M, N, ldc, c_off):
    mask = np.ones(raw.size, bool)
    for i in range(M):
        mask[c_off + i * ldc:c_off + i * ldc + N] = False
    assert np.isnan(raw[mask]).all(), "C written outside its M x N elements"


# Cluster sizes S = 2 .. 16 (the row ranges of the final sum are uneven for
# S not dividing 128; sizes above 8 for at most 4 tiles, where the GPU has
# them, else these shapes run with 8), ragged M, N and K tiles, every
# copy-width class of A, B and C (row strides and base offsets), and products
# smaller than a tile.
@pytest.mark.parametrize("M,N,K,lds,offs,S", [
    (1024, 2432, 64, None, (0, 0, 0), 2),            # 152 tiles, 2 K tiles per CTA
    (100, 12923, 96, None, (0, 0, 0), 3),            # 1 x 101 tiles
    (1024, 1024, 1024, None, (0, 0, 0), 4),          # 64 tiles, tensor copies
    (700, 1250, 160, (161, 1250, 1251), (1, 0, 3), 5),  # A and C 4-byte aligned
    (600, 1280, 200, (202, 1282, 1280), (2, 2, 0), 6),  # A and B 8-byte aligned
    (128, 5504, 224, (224, 5505, 5506), (0, 1, 2), 7),  # B 4-byte, C 8-byte aligned
    (256, 256, 256, None, (0, 0, 0), 8),             # 4 tiles, 16 K tiles
    (1000, 1030, 777, (777, 1030, 1030), (0, 0, 0), 4),  # misaligned rows, ragged K
    (256, 200, 320, None, (0, 0, 0), 10),            # 4 tiles, 20 K tiles
    (128, 500, 384, (385, 500, 500), (0, 0, 0), 12),  # 4 tiles, A 4-byte aligned
    (200, 130, 448, None, (0, 0, 2), 14),            # 4 tiles, C 8-byte aligned
    (256, 256, 1024, None, (0, 0, 0), 16),           # 4 tiles
    (512, 512, 1024, None, (0, 0, 0), 8),            # 16 tiles: at most 8 above 4 tiles
    (77, 250, 999, (1001, 252, 260), (0, 0, 0), 16),  # ragged K tile, padded C rows
    (300, 600, 400, (400, 602, 600), (0, 0, 0), 8),  # A 16-byte, B 8-byte aligned
    (200, 300, 500, (501, 301, 300), (0, 0, 0), 8),  # A and B 4-byte aligned
    (3, 5, 100, (100, 5, 7), (0, 0, 1), 3),          # a few elements
    (1, 100, 512, None, (0, 0, 0), 16),              # one row
])
def test_cluster_split_full_check(oracle_lib, M, N, K, lds, offs, S):
    lda, ldb, ldc = lds or (K, N, N)
    bound = _cluster_bound(M, N, K)
    assert bound == (min(S, _max_cluster()) if S > 8 else S)
    A = synth.matrix(M, K, 71, 0, "normal", ld=lda, pad_value=np.nan)
    B = synth.matrix(K, N, 71, 1, "normal", ld=ldb, pad_value=np.nan)
    C, raw, _, kind, words = _run(M, N, K, A, lda, B, ldb, ldc, offs)
    S = kind >> 8
    assert kind & 255 == 32 and words == 0 and 2 <= S <= bound, kind
    Cr, Sr = oracle_lib.gemm(A, B, M=M, N=N, K=K, lda=lda, ldb=ldb)
    tol.assert_close(C, Cr, Sr, K, f"cluster split S={S} {M}x{N}x{K}")
    _padding_untouched(raw, M, N, ldc, offs[2])
    # through sgemm_f32_ws, where the split is also chosen there: the same
    # kernel and slices, so the same result bit for bit, and the workspace
    # is not touched at all
    nbytes = sg.workspace_size(M, N, K)
    fake = [p + 4 * o for p, o in zip(_PTRS, offs)]  # apart, with the offsets' alignment
    _, wkind, _ = sg.ws_schedule(M, N, K, fake[0], lda, fake[1], ldb, fake[2], ldc, nbytes)
    if wkind & 32:
        C2, raw2, ws, kind2, _ = _run(M, N, K, A, lda, B, ldb, ldc, offs, nbytes=nbytes)
        assert kind2 == kind
        assert np.all(ws == 7), "the cluster split uses no workspace"
        np.testing.assert_array_equal(C2.view(np.uint32), C.view(np.uint32))


def test_cluster_split_integer_exact_and_deterministic(oracle_lib):
    M, N, K = 1024, 1024, 1024
    A = synth.matrix(M, K, 73, 0, "int5")
    B = synth.matrix(K, N, 73, 1, "int5")
    tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.empty(M, N, device="cuda")
    sst, kind, _ = sg.ws_schedule(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, C.data_ptr(), N,
                                  sg.workspace_size_for(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N))
    assert sst == 0 and kind & 255 == 32  # the torch wrapper's balanced call takes it too
    C1 = sg.sgemm(tA, tB)
    C2 = sg.sgemm(tA, tB, balanced=False)
    C3 = sg.sgemm(tA, tB)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2) and torch.equal(C1, C3)
    Cr, _ = oracle_lib.gemm(A, B)
    np.testing.assert_array_equal(C1.cpu().numpy().astype(np.float64), Cr)
    assert sg.copy_timeouts() == 0


def test_not_taken_where_it_does_not_apply():
    """More than G / 2 tiles, fewer than 4 K tiles, an empty K, or a
    workspace for a multi-part split that keeps its CTAs busier: no cluster
    split."""
    G = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    pA, pB, pC = _PTRS
    for M, N, K in [(128 * (G // 2 + 1), 128, 512),  # G / 2 + 1 tiles
                    (1024, 1024, 48),                # 3 K tiles: S would be 1
                    (1024, 1024, 0)]:                # K = 0: C is zeroed
        sst, kind, _ = sg.ws_schedule(M, N, K, pA, max(K, 1), pB, N, pC, N, 0)
        assert sst == 0 and kind & 32 == 0, (M, N, K, kind)
    # 128 tiles: S = 2 would give 32 K tiles per CTA against the multi-part
    # split's 27 on 304 CTAs (plus its fixed costs, 3.5 K tiles here); without
    # the workspace the split still runs
    M, N, K = 2048, 1024, 1024
    _, kind, _ = sg.ws_schedule(M, N, K, pA, K, pB, N, pC, N, sg.workspace_size(M, N, K))
    assert kind == 2
    _, kind, _ = sg.ws_schedule(M, N, K, pA, K, pB, N, pC, N, 0)
    assert kind == 32 | (2 << 8)  # S = 2: 128 clusters of 2


_FORCED_CHILD = r"""
import sys, json
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
import oracle
from tests import _tolerance as tol
from tests._gpu import dev_buffer
sg.load_library()
oracle.build()
out = []
for (M, N, K) in json.loads(sys.argv[2]):
    A = synth.matrix(M, K, 74, 0, "normal")
    B = synth.matrix(K, N, 74, 1, "normal")
    tA, pA = dev_buffer(A)
    tB, pB = dev_buffer(B)
    tC = torch.full((M * N + 4,), float("nan"), device="cuda")
    _, kind, _ = sg.ws_schedule(M, N, K, pA, K, pB, N, tC.data_ptr(), N, 0)
    assert sg.sgemm_f32(M, N, K, pA, K, pB, N, tC.data_ptr(), N, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    Cr, Sr = oracle.gemm(A, B)
    tol.assert_close(tC.cpu().numpy()[:M * N].reshape(M, N), Cr, Sr, K, f"forced cluster {M}x{N}x{K}")
    out.append(kind)
print(json.dumps(out))
"""


@pytest.mark.parametrize("tune", ["cluster=off", "cluster=3", "cluster=9", "cluster=13"])
def test_forced_cluster_size(tune):
    """SGEMM_F32_TUNE (read once per process, so in a child process) forces
    the cluster size, or turns the split off, on shapes where the default
    picks another: 4 and 12 tiles (S 9 and 13 need clusters of more than 8,
    which the GPU may not schedule; then no split runs)."""
    import json, os, subprocess, sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    shapes = [(256, 256, 1024), (384, 512, 768)]
    r = subprocess.run([sys.executable, "-c", _FORCED_CHILD, root, json.dumps(shapes)], cwd=root,
                       env=dict(os.environ, SGEMM_F32_TUNE=tune), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    kinds = json.loads(r.stdout.strip().splitlines()[-1])
    want = tune.split("=")[1]
    for k in kinds:
        if want == "off":
            assert k & 32 == 0, kinds
        elif int(want) <= 8 or _max_cluster() >= int(want):
            assert k & 255 == 32 and k >> 8 == int(want), kinds
        else:
            assert k & 32 == 0, kinds

