"""The two-stream schedule under a single hardware work queue (CUDA_DEVICE_MAX_CONNECTIONS=1).

The pages' Megatron recipe sets CUDA_DEVICE_MAX_CONNECTIONS=1 so that the communication kernel is
queued ahead of the weight-gradient GEMM ("04 · TP/SP 的通信-计算 overlap 与工程优化", §2).  This
library orders its compute and reduction streams with events instead and must not depend on that
setting: a forward + backward with the INTRA schedule (shard-sums on the second stream, the
input-gradient reduction overlapping the weight-gradient GEMM) and an INTER layer stack run in a
child process with one connection must reproduce, bit for bit, the results of this process (the
default number of connections).  The variable is read when the CUDA context is created, hence the
child process.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs the two workloads and writes their outputs (bf16 bits, fp32) to an .npz file.
CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth

def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)

h = dm.domino_create()
out = {}
M, hid, Fi, t = 1024, 256, 128, 4
s = synth.MlpShape("q", M, hid, Fi * t, synth.ACT_SWIGLU, t, 4, 1, backward=True)
d = synth.make_inputs(s, seed=31)
X, A, B, gY = dev(d["X"]), dev(d["A"][0]), dev(d["B"][0]), dev(d["gY"])
cfg = dm.make_cfg(M, hid, s.F, t, 4, 1, synth.ACT_SWIGLU, sched=dm.SCHED_INTRA)
n = max(dm.domino_workspace_size(cfg, dm.PASS_FWD), dm.domino_workspace_size(cfg, dm.PASS_BWD))
ws = torch.empty(n, dtype=torch.uint8, device="cuda")
Y = torch.empty((M, hid), dtype=torch.bfloat16, device="cuda")
S = torch.empty((M, s.a_rows), dtype=torch.bfloat16, device="cuda")
gX = torch.empty_like(Y)
gA = torch.zeros((s.a_rows, hid), dtype=torch.float32, device="cuda")
gB = torch.zeros((t, hid, Fi), dtype=torch.float32, device="cuda")
dm.domino_mlp_fwd(h, cfg, X, A, B, Y, S, ws, n)
dm.domino_mlp_bwd(h, cfg, X, A, B, S, gY, gX, gA, gB, ws, n)
L = 3
s2 = synth.MlpShape("q2", 512, 256, 512, synth.ACT_GELU, 2, 2, 2, layers=L, layernorm=True)
d2 = synth.make_inputs(s2, seed=32)
cfg2 = dm.make_cfg(512, 256, 512, 2, 2, 2, synth.ACT_GELU, sched=dm.SCHED_INTER, layers=L)
n2 = dm.domino_workspace_size(cfg2, dm.PASS_STACK)
ws2 = torch.empty(n2, dtype=torch.uint8, device="cuda")
Z = torch.empty((512, 256), dtype=torch.bfloat16, device="cuda")
dm.domino_stack_fwd(h, cfg2, dev(d2["X"]), dev(d2["A"]), dev(d2["B"]), Z, ws2, n2)
torch.cuda.synchronize()
st, site = dm.domino_device_status(h)
assert st == 0, site
dm.domino_destroy(h)
np.savez(sys.argv[2], Y=bits(Y), gX=bits(gX), gA=gA.cpu().numpy(), gB=gB.cpu().numpy(), Z=bits(Z))
"""


def run_child(tmp_path, name, connections):
    env = dict(os.environ)
    if connections is None:
        env.pop("CUDA_DEVICE_MAX_CONNECTIONS", None)
    else:
        env["CUDA_DEVICE_MAX_CONNECTIONS"] = str(connections)
    path = str(tmp_path / f"{name}.npz")
    subprocess.run([sys.executable, "-c", CHILD, ROOT, path], env=env, check=True, timeout=600)
    return np.load(path)


def test_single_connection_bit_identical(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from comm_overlap_gb300 import build
    build.build()
    ref = run_child(tmp_path, "default", None)
    one = run_child(tmp_path, "one", 1)
    for k in ("Y", "gX", "gA", "gB", "Z"):
        assert np.array_equal(one[k], ref[k]), k
