"""The PyTorch module around the library (comm_overlap_gb300.torch_mlp.DominoMLP) against the CPU
oracle: forward output, input gradient through autograd, weight gradients accumulated into fp32
main_grad (twice: accumulation) or returned as bf16 .grad."""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import assert_tol, dev_bf16, host_f64
from test_gpu_bwd import shard_major_dA, shard_major_dB

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from comm_overlap_gb300 import build
    build.build()


def make(act, fuse, sched=dm.SCHED_INTRA):
    import torch
    from comm_overlap_gb300.torch_mlp import DominoMLP
    M, h, Fi, t, p, q = 384, 256, 136, 2, 2, 2
    s = synth.MlpShape("tm", M, h, Fi * t, act, t, p, q, backward=True)
    d = synth.make_inputs(s, seed=51)
    mod = DominoMLP(h, Fi * t, t, p, q, act, sched=sched, fuse_wgrad=fuse)
    with torch.no_grad():
        mod.A.copy_(dev_bf16(d["A"][0]))
        mod.B.copy_(dev_bf16(d["B"][0]))
    return mod, d, s


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_module_fused_main_grad(built, act):
    import torch
    mod, d, s = make(act, True)
    X = dev_bf16(d["X"]).requires_grad_(True)
    gY = dev_bf16(d["gY"])
    Y = mod(X)
    ref_y = oracle.mlp_fwd(d["X"], d["A"][0], d["B"][0], s.t, act)
    assert_tol(host_f64(Y), ref_y, "module forward")
    Y.backward(gY)
    dX, dA, dB = oracle.mlp_bwd(d["X"], d["A"][0], d["B"][0], d["gY"], s.t, act)
    gated = act in synth.GATED
    assert_tol(host_f64(X.grad), dX, "module input gradient")
    assert mod.A.grad is None and mod.B.grad is None
    gA1 = mod.A.main_grad.cpu().numpy().astype(np.float64)
    gB1 = mod.B.main_grad.cpu().numpy().astype(np.float64)
    assert_tol(gA1, shard_major_dA(dA, s.t, s.Fi, gated), "main_grad of A")
    assert_tol(gB1, shard_major_dB(dB, s.t, s.Fi), "main_grad of B")
    # a second micro-batch accumulates into the same fp32 buffers
    X.grad = None
    mod(X).backward(gY)
    torch.cuda.synchronize()
    assert_tol(mod.A.main_grad.cpu().numpy().astype(np.float64), 2 * gA1, "accumulated main_grad of A",
               rel=1e-5, abs_=1e-6)
    assert_tol(mod.B.main_grad.cpu().numpy().astype(np.float64), 2 * gB1, "accumulated main_grad of B",
               rel=1e-5, abs_=1e-6)
    mod.close()


def test_module_plain_grad_and_schedules(built):
    import torch
    act = synth.ACT_SWIGLU
    outs = []
    for sched in (dm.SCHED_INTRA, dm.SCHED_FUSED, dm.SCHED_SERIAL):
        mod, d, s = make(act, False, sched)
        X = dev_bf16(d["X"]).requires_grad_(True)
        Y = mod(X)
        Y.backward(dev_bf16(d["gY"]))
        torch.cuda.synchronize()
        outs.append((Y.detach().clone(), X.grad.clone(), mod.A.grad.clone(), mod.B.grad.clone()))
        if sched == dm.SCHED_INTRA:
            _, dA, dB = oracle.mlp_bwd(d["X"], d["A"][0], d["B"][0], d["gY"], s.t, act, want_dx=False)
            assert mod.A.grad.dtype == torch.bfloat16
            assert_tol(host_f64(mod.A.grad), shard_major_dA(dA, s.t, s.Fi, True), ".grad of A")
            assert_tol(host_f64(mod.B.grad), shard_major_dB(dB, s.t, s.Fi), ".grad of B")
        mod.close()
    for o in outs[1:]:  # every schedule gives the same bits
        for a, b in zip(o, outs[0]):
            assert torch.equal(a, b)


def test_library_call_from_a_fresh_thread(built):
    """A thread that has not used CUDA yet (no current context, like PyTorch's autograd workers)
    can call the library: the entry points bind the device's context before encoding tensor maps."""
    import threading
    import torch
    M, h, Fi, t = 256, 256, 128, 2
    s = synth.MlpShape("th", M, h, Fi * t, synth.ACT_GELU, t, 2, 1)
    d = synth.make_inputs(s, seed=52)
    X, A, B = dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0])
    cfg = dm.make_cfg(M, h, Fi * t, t, 2, 1, synth.ACT_GELU)
    n = dm.domino_workspace_size(cfg, dm.PASS_FWD)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    h_ = dm.domino_create()
    stream = torch.cuda.current_stream().cuda_stream
    errors = []

    def run():
        try:
            dm.domino_mlp_fwd(h_, cfg, X, A, B, Y, None, ws, n, stream)
        except Exception as e:  # reported below
            errors.append(e)

    th = threading.Thread(target=run)
    th.start()
    th.join()
    torch.cuda.synchronize()
    dm.domino_destroy(h_)
    assert not errors, errors
    assert_tol(host_f64(Y), oracle.mlp_fwd(d["X"], d["A"][0], d["B"][0], t, synth.ACT_GELU), "forward from a thread")


def make_stack(act, fuse, L=2, M=256, h=128, F=256, t=2, p=2, q=2, seed=53):
    import torch
    from comm_overlap_gb300.torch_mlp import DominoStack
    s = synth.MlpShape("ts", M, h, F, act, t, p, q, layers=L, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=seed)
    mod = DominoStack(L, h, F, t, p, q, act, fuse_wgrad=fuse)
    with torch.no_grad():
        mod.A.copy_(dev_bf16(d["A"]))
        mod.B.copy_(dev_bf16(d["B"]))
    return mod, d, s


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_stack_module_against_oracle(built, act):
    """DominoStack: output, input gradient through autograd and the fp32 main_grad of every layer
    against the oracle's stack forward and backward; the no-grad forward gives the same bits."""
    import torch
    mod, d, s = make_stack(act, True)
    Z = dev_bf16(d["X"]).requires_grad_(True)
    out = mod(Z)
    assert_tol(host_f64(out), oracle.stack_fwd(d["X"], d["A"], d["B"], s.t, act, 1e-5), "stack module output")
    out.backward(dev_bf16(d["gY"]))
    gZ0, dA, dB = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], s.t, act, 1e-5, want_w=True)
    assert_tol(host_f64(Z.grad), gZ0, "stack module input gradient")
    assert mod.A.grad is None and mod.B.grad is None
    gA = mod.A.main_grad.cpu().numpy().astype(np.float64)
    gB = mod.B.main_grad.cpu().numpy().astype(np.float64)
    for layer in range(s.layers):
        assert_tol(gA[layer], dA[layer], f"main_grad of A, layer {layer}")
        assert_tol(gB[layer], dB[layer], f"main_grad of B, layer {layer}")
    with torch.no_grad():
        inference = mod(Z.detach())
    assert torch.equal(inference, out.detach())
    mod.close()


def test_stack_module_plain_grad(built):
    """fuse_wgrad=False: the weight gradients come back as bf16 .grad, equal to the rounded fp32
    gradients of the fused module."""
    import torch
    fused, d, s = make_stack(synth.ACT_GELU, True)
    plain, _, _ = make_stack(synth.ACT_GELU, False)
    outs = []
    for mod in (fused, plain):
        Z = dev_bf16(d["X"]).requires_grad_(True)
        mod(Z).backward(dev_bf16(d["gY"]))
        torch.cuda.synchronize()
        outs.append(Z.grad.clone())
    assert torch.equal(outs[0], outs[1])
    assert plain.A.grad.dtype == torch.bfloat16
    assert torch.equal(plain.A.grad, fused.A.main_grad.to(torch.bfloat16))
    assert torch.equal(plain.B.grad, fused.B.main_grad.to(torch.bfloat16))
    fused.close()
    plain.close()


def test_stack_module_schedules_and_splits_bit_identical(built):
    """DominoStack under every overlapped schedule and row split gives the same bits for the output,
    the input gradient and the fp32 weight gradients (row splits change only the order in which
    tokens are summed into the weight gradients, so those are compared across schedules at p = 2)."""
    import torch
    from comm_overlap_gb300.torch_mlp import DominoStack
    L, M, h, F, t = 2, 512, 128, 256, 2
    s = synth.MlpShape("tss", M, h, F, synth.ACT_SWIGLU, t, 2, 2, layers=L, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=54)
    results = {}
    for sched in (dm.SCHED_INTER, dm.SCHED_INTRA, dm.SCHED_FUSED, dm.SCHED_SERIAL):
        for p in (1, 2, 4):
            mod = DominoStack(L, h, F, t, p, 2, synth.ACT_SWIGLU, sched=sched)
            with torch.no_grad():
                mod.A.copy_(dev_bf16(d["A"]))
                mod.B.copy_(dev_bf16(d["B"]))
            Z = dev_bf16(d["X"]).requires_grad_(True)
            out = mod(Z)
            out.backward(dev_bf16(d["gY"]))
            torch.cuda.synchronize()
            results[(sched, p)] = (out.detach().clone(), Z.grad.clone(), mod.A.main_grad.clone(),
                                   mod.B.main_grad.clone())
            mod.close()
    ref = results[(dm.SCHED_INTER, 2)]
    for key, r in results.items():
        assert torch.equal(r[0], ref[0]) and torch.equal(r[1], ref[1]), key
        if key[1] == 2:
            assert torch.equal(r[2], ref[2]) and torch.equal(r[3], ref[3]), key
