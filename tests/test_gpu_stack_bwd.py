"""GPU parity of the layer-stack training path (domino_stack_fwd_train + domino_stack_bwd) against
the CPU oracle's stack backward (LayerNorm backward, MLP backward, residual), in double."""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import assert_tol, dev_bf16, edge_rows, host_bits, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from comm_overlap_gb300 import build
    build.build()
    h = dm.domino_create()
    yield h
    st, site = dm.domino_device_status(h)
    dm.domino_destroy(h)
    assert st == 0, f"device error word set: site {site:#x}"


def run_stack_train(h, s, d, sched=dm.SCHED_INTER, p=None, gA0=None, gB0=None):
    import torch
    cfg = dm.make_cfg(s.M, s.h, s.F, s.t, s.p if p is None else p, s.q, s.act, sched=sched, layers=s.layers,
                      ln_eps=1e-5)
    Z, A, B, gZ = dev_bf16(d["X"]), dev_bf16(d["A"]), dev_bf16(d["B"]), dev_bf16(d["gY"])
    out = torch.empty_like(Z)
    save = torch.empty(dm.domino_stack_save_size(cfg), dtype=torch.uint8, device="cuda")
    ws = torch.empty(max(dm.domino_workspace_size(cfg, dm.PASS_STACK), dm.domino_workspace_size(cfg, dm.PASS_STACK_BWD)),
                     dtype=torch.uint8, device="cuda")
    dm.domino_stack_fwd_train(h, cfg, Z, A, B, out, save, ws)
    gZin = torch.empty_like(Z)
    gA = torch.zeros(d["A"].shape, dtype=torch.float32, device="cuda") if gA0 is None else torch.from_numpy(gA0).cuda()
    gB = torch.zeros(d["B"].shape, dtype=torch.float32, device="cuda") if gB0 is None else torch.from_numpy(gB0).cuda()
    dm.domino_stack_bwd(h, cfg, A, B, save, gZ, gZin, gA, gB, ws)
    torch.cuda.synchronize()
    return out, gZin, gA.cpu().numpy().astype(np.float64), gB.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_stack_backward_matches_oracle(handle, act):
    s = synth.MlpShape("sb", 256, 128, 256, act, 2, 2, 2, layers=3, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=41)
    gA0 = synth.normal_f32(d["A"].shape, 0, 0.01, 41, synth.TID_GA0)
    gB0 = synth.normal_f32(d["B"].shape, 0, 0.01, 41, synth.TID_GB0)
    out, gZin, gA, gB = run_stack_train(handle, s, d, gA0=gA0, gB0=gB0)
    assert_tol(host_f64(out), oracle.stack_fwd(d["X"], d["A"], d["B"], s.t, act, 1e-5), "stack output")
    gZ0, dA, dB = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], s.t, act, 1e-5, want_w=True)
    assert_tol(host_f64(gZin), gZ0, "gradient of the stack input")
    for l in range(s.layers):
        assert_tol(gA[l] - gA0[l], dA[l], f"gA increment, layer {l}")
        assert_tol(gB[l] - gB0[l], dB[l], f"gB increment, layer {l}")


def test_stack_backward_splits_and_schedules_bit_identical(handle):
    s = synth.MlpShape("sb", 512, 128, 256, synth.ACT_GELU, 2, 2, 2, layers=2, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=42)
    ref = host_bits(run_stack_train(handle, s, d, p=1)[1])
    for sched in (dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_INTER):
        for p in (2, 4):
            assert np.array_equal(host_bits(run_stack_train(handle, s, d, sched=sched, p=p)[1]), ref), (sched, p)


@pytest.mark.slow
def test_stack_backward_full_size(handle):
    import torch
    base = synth.SHAPES["gpt3_6.7b_stack4"]
    import dataclasses
    s = dataclasses.replace(base, backward=True)
    d = synth.make_inputs(s, seed=0)
    out, gZin, _, _ = run_stack_train(handle, s, d)
    rows = edge_rows(s.M, s.M // s.p, 43, n_random=6)   # every chunk and tile edge, and 6 at random
    gZ0, _, _ = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], s.t, s.act, 1e-5, rows=rows)
    assert_tol(host_f64(gZin[torch.from_numpy(rows).cuda()]), gZ0, "stack input gradient, sampled rows")
