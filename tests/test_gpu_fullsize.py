"""Parity at the five workloads' full sizes, in the launch configuration bench.py times.

The oracle evaluates sampled outputs one by one (rows of Y / gX / the stack output, ffn
features of the weight gradients); the GPU computes the whole problem.  The samples always hold
both sides of every row-chunk and tile boundary and the last tile of each chunk (edge_rows), and,
for the weight gradients, the first and last feature of every shard (edge_feats).  Row-split results are
also checked bitwise against the unsplit (p = 1) GPU run at full size.
"""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import Lib, assert_tol, dev_bf16, edge_feats, edge_rows, host_bits, host_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from comm_overlap_gb300 import build
    build.build()
    L = Lib()
    yield L
    st, site = L.status()
    L.close()
    assert st == 0, f"device error word set: site {site:#x}"


def cfg_of(s, p=None, sched=dm.SCHED_INTRA):
    return dm.make_cfg(s.M, s.h, s.F, s.t, s.p if p is None else p, s.q, s.act, sched=sched, layers=s.layers,
                       ln_eps=1e-5)


@pytest.mark.parametrize("name", ["tiny_gelu", "gpt3_2.7b_mlp", "llama2_7b_swiglu"])
def test_forward_full_size(lib, name):
    import torch
    s = synth.SHAPES[name]
    d = synth.make_inputs(s, seed=0)
    X, A, B = dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0])
    Y, _ = lib.fwd(cfg_of(s), X, A, B)
    rows = edge_rows(s.M, s.M // s.p, 10) if s.M > 1024 else np.arange(s.M, dtype=np.int64)
    ref = oracle.mlp_fwd(d["X"], d["A"][0], d["B"][0], s.t, s.act, rows=rows)
    assert_tol(host_f64(Y[torch.from_numpy(rows).cuda()]), ref, f"{name} sampled rows")
    if s.p > 1:
        Y1, _ = lib.fwd(cfg_of(s, p=1), X, A, B)
        assert torch.equal(Y.view(torch.int16), Y1.view(torch.int16)), "row split not bit-identical"


def test_stack_full_size(lib):
    import torch
    s = synth.SHAPES["gpt3_6.7b_stack4"]
    d = synth.make_inputs(s, seed=0)
    X, A, B = dev_bf16(d["X"]), dev_bf16(d["A"]), dev_bf16(d["B"])
    Z = lib.stack(cfg_of(s, sched=dm.SCHED_INTER), X, A, B)
    rows = edge_rows(s.M, s.M // s.p, 11)
    ref = oracle.stack_fwd(d["X"], d["A"], d["B"], s.t, s.act, 1e-5, rows=rows)
    assert_tol(host_f64(Z[torch.from_numpy(rows).cuda()]), ref, "stack sampled rows")
    Z1 = lib.stack(cfg_of(s, p=1, sched=dm.SCHED_INTER), X, A, B)
    assert torch.equal(Z.view(torch.int16), Z1.view(torch.int16)), "row split not bit-identical"


def test_forward_backward_full_size(lib):
    import torch
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    d = synth.make_inputs(s, seed=0)
    X, A, B, gY = dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0]), dev_bf16(d["gY"])
    cfg = cfg_of(s)
    Y, S = lib.fwd(cfg, X, A, B, save=True)
    gA0 = torch.zeros((s.a_rows, s.h), dtype=torch.float32, device="cuda")
    gB0 = torch.zeros((s.t, s.h, s.Fi), dtype=torch.float32, device="cuda")
    gX, gA, gB = lib.bwd(cfg, X, A, B, S, gY, gA0, gB0)
    rows = edge_rows(s.M, s.M // s.p, 12)
    ridx = torch.from_numpy(rows).cuda()
    Yref = oracle.mlp_fwd(d["X"], d["A"][0], d["B"][0], s.t, s.act, rows=rows)
    assert_tol(host_f64(Y[ridx]), Yref, "Y sampled rows")
    dX, _, _ = oracle.mlp_bwd(d["X"], d["A"][0], d["B"][0], d["gY"], s.t, s.act, rows=rows, want_dw=False)
    assert_tol(host_f64(gX[ridx]), dX, "gX sampled rows")
    feats = edge_feats(s.Fi, s.t, 13)
    _, dA, dB = oracle.mlp_bwd(d["X"], d["A"][0], d["B"][0], d["gY"], s.t, s.act, feats=feats, want_dx=False)
    gA_h, gB_h = gA.cpu().numpy().astype(np.float64), gB.cpu().numpy().astype(np.float64)
    for k, f in enumerate(feats):
        i, j = divmod(int(f), s.Fi)
        gate_row, up_row = i * 2 * s.Fi + j, i * 2 * s.Fi + s.Fi + j
        assert_tol(gA_h[gate_row], dA[k, 0], f"gA gate row of feature {f}")
        assert_tol(gA_h[up_row], dA[k, 1], f"gA up row of feature {f}")
        assert_tol(gB_h[i, :, j], dB[k], f"gB column of feature {f}")
    # the input gradient of a row split is bit-identical to the unsplit backward
    gX1, _, _ = lib.bwd(cfg_of(s, p=1), X, A, B, S, gY, gA0, gB0)
    assert torch.equal(gX.view(torch.int16), gX1.view(torch.int16)), "gX row split not bit-identical"
