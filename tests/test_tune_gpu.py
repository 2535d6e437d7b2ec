"""SGEMM_F32_TUNE overrides against the FP64 oracle (needs a GB300).

The variable is read once per process, so each setting runs in a child
process: the forced kernel family, schedule and split-tail part count, and
the two diagnostics (a drained copy ring, one CTA per SM), each on a product
with more tiles than the GPU holds at once and a ragged last K tile.  Every
forced choice must keep the result within the FP32 bound and be the one
sgemm_f32_ws_schedule reports.
"""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

_CHILD = r"""
import sys, json
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import dense_fp32_tiled_gb300 as sg
from dense_fp32_tiled_gb300 import synth
import oracle
from tests import _tolerance as tol
sg.load_library()
oracle.build()
M, N, K = 2500, 2100, 340  # rows 16-byte aligned, last K tile ragged (16 and 32 deep)
A = synth.matrix(M, K, 76, 0, "normal")
B = synth.matrix(K, N, 76, 1, "normal")
tA, tB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
tC = torch.full((M, N), float("nan"), device="cuda")
nbytes = sg.workspace_size_for(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N)
if sys.argv[2] == "room":  # room for the k-major copy too
    nbytes += (K * ((M + 3) // 4 * 4) * 4 + 255) // 256 * 256
ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
_, kind, _ = sg.ws_schedule(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, nbytes)
st = sg.sgemm_f32_ws(M, N, K, tA.data_ptr(), K, tB.data_ptr(), N, tC.data_ptr(), N, ws.data_ptr(), nbytes,
                     torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
assert st == 0, sg.status_string(st)
Cr, Sr = oracle.gemm(A, B)
tol.assert_close(tC.cpu().numpy(), Cr, Sr, K, "tuned " + sys.argv[3])
assert sg.copy_timeouts() == 0
print(json.dumps({"kind": kind}))
"""

# (setting, workspace, expected schedule bits 0-1, expected k-major copy)
CASES = [
    ("schedule=0", "size", 0, False),
    ("schedule=1", "size", 1, False),
    ("schedule=2", "size", 2, False),
    ("schedule=3", "size", 3, False),
    ("schedule=3,parts=6", "size", 3, False),
    ("kernels=rowmajor8", "room", 3, False),
    ("kernels=kmajor16", "room", 3, True),
    ("kernels=kmajor16,schedule=0,drain=on", "room", 0, True),
    ("kernels=kmajor16,schedule=0,cta_per_sm=1", "room", 0, True),
    ("schedule=0,cta_per_sm=1", "size", 0, False),
]


@pytest.mark.parametrize("setting,room,sched,kmajor", CASES)
def test_forced_setting_matches_the_oracle(setting, room, sched, kmajor):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHILD, root, room, setting], cwd=root,
                       env=dict(os.environ, SGEMM_F32_TUNE=setting), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    kind = json.loads(r.stdout.strip().splitlines()[-1])["kind"]
    assert kind & 3 == sched and bool(kind & 16) == kmajor and kind & 32 == 0, (setting, kind)
