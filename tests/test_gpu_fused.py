"""GPU parity of the fused schedule (DOMINO_SCHED_FUSED): the second linear and the input-gradient
GEMM reduce their shard partials tile by tile inside one kernel (fp32 running sums in shard order;
a short last round of tiles is shared by several CTA pairs per tile through partial slots).

* Integer-valued inputs: Y and gX equal the oracle's exact result rounded once to bf16.
* Real-valued inputs: within the parity tolerance of the double-precision oracle, and bit-identical
  to the two-stream schedule, which sums the same fp32 partials in the same order.
* Ragged tails in every dimension, t = 1 (the only shard is the last), column and row splits, the
  residual of the layer stack, the stack backward, a whole round followed by a split last round, and
  the full-size forward+backward workload.
"""

import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import Lib, assert_tol, bf16_round, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu


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


def inputs(M, h, Fi, t, act, seed, integer):
    gated = act in synth.GATED
    a_rows = 2 * Fi * t if gated else Fi * t
    if integer:
        # sparse enough that every bf16 intermediate (H, dZ) is an exact small integer
        pz = 0.85 if gated else 0.5
        X = synth.ternary_bf16((M, h), seed, synth.TID_X, p_zero=pz)
        A = synth.ternary_bf16((a_rows, h), seed, synth.TID_A, p_zero=pz)
        B = synth.ternary_bf16((t, h, Fi), seed, synth.TID_B, p_zero=pz)
        gY = synth.ternary_bf16((M, h), seed, synth.TID_GY, p_zero=pz)
    else:
        X = synth.normal_bf16((M, h), 0.0, 1.0, seed, synth.TID_X)
        A = synth.normal_bf16((a_rows, h), 0.0, 0.02, seed, synth.TID_A)
        B = synth.normal_bf16((t, h, Fi), 0.0, 0.02, seed, synth.TID_B)
        gY = synth.normal_bf16((M, h), 0.0, 1.0, seed, synth.TID_GY)
    return X, A, B, gY


def fwd_bwd(lib, M, h, Fi, t, p, q, act, sched, X, A, B, gY):
    import torch
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=sched)
    Xd, Ad, Bd, gYd = dev_bf16(X), dev_bf16(A), dev_bf16(B), dev_bf16(gY)
    Y, S = lib.fwd(cfg, Xd, Ad, Bd, save=True)
    gA0 = torch.zeros(A.shape, dtype=torch.float32, device="cuda")
    gB0 = torch.zeros(B.shape, dtype=torch.float32, device="cuda")
    gX, gA, gB = lib.bwd(cfg, Xd, Ad, Bd, S, gYd, gA0, gB0)
    return Y, gX, gA, gB


# (M, h, F_i, t, p, q): ragged M, N (h/q not a multiple of 32) and K tails, t = 1
SHAPES = [
    (384, 208, 136, 3, 2, 2),
    (520, 136, 264, 2, 1, 1),
    (264, 72, 40, 4, 3, 3),
    (300, 328, 200, 1, 1, 1),
    (256, 256, 64, 8, 1, 1),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_RELU, synth.ACT_BILINEAR])
def test_fused_integer_exact(lib, shape, act):
    M, h, Fi, t, p, q = shape
    X, A, B, gY = inputs(M, h, Fi, t, act, 50, integer=True)
    Y, gX, _, _ = fwd_bwd(lib, M, h, Fi, t, p, q, act, dm.SCHED_FUSED, X, A, B, gY)
    assert np.array_equal(host_f64(Y), bf16_round(oracle.mlp_fwd(X, A, B, t, act))), "Y"
    gX_ref, _, _ = oracle.mlp_bwd(X, A, B, gY, t, act, want_dw=False)
    assert np.array_equal(host_f64(gX), bf16_round(gX_ref)), "gX"


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_fused_matches_oracle_and_stream_schedule(lib, shape, act):
    M, h, Fi, t, p, q = shape
    X, A, B, gY = inputs(M, h, Fi, t, act, 51, integer=False)
    Y, gX, gA, gB = fwd_bwd(lib, M, h, Fi, t, p, q, act, dm.SCHED_FUSED, X, A, B, gY)
    assert_tol(host_f64(Y), oracle.mlp_fwd(X, A, B, t, act), "Y")
    gX_ref, _, _ = oracle.mlp_bwd(X, A, B, gY, t, act, want_dw=False)
    assert_tol(host_f64(gX), gX_ref, "gX")
    Y2, gX2, gA2, gB2 = fwd_bwd(lib, M, h, Fi, t, p, q, act, dm.SCHED_INTRA, X, A, B, gY)
    assert np.array_equal(host_bits(Y), host_bits(Y2)), "Y differs from the two-stream schedule"
    assert np.array_equal(host_bits(gX), host_bits(gX2)), "gX differs from the two-stream schedule"
    # the weight gradients do not go through the shard-sum: same kernels, same order
    assert np.array_equal(gA.cpu().numpy(), gA2.cpu().numpy())
    assert np.array_equal(gB.cpu().numpy(), gB2.cpu().numpy())


def test_fused_repeated_calls_identical(lib):
    """The partial slots and their counters of the split tiles are rewritten and reset by every call:
    no state leaks between calls."""
    M, h, Fi, t, p, q = 512, 256, 128, 4, 2, 1
    X, A, B, gY = inputs(M, h, Fi, t, synth.ACT_GELU, 52, integer=False)
    first = fwd_bwd(lib, M, h, Fi, t, p, q, synth.ACT_GELU, dm.SCHED_FUSED, X, A, B, gY)
    X2, _, _, _ = inputs(M, h, Fi, t, synth.ACT_GELU, 53, integer=False)
    fwd_bwd(lib, M, h, Fi, t, p, q, synth.ACT_GELU, dm.SCHED_FUSED, X2, A, B, gY)
    again = fwd_bwd(lib, M, h, Fi, t, p, q, synth.ACT_GELU, dm.SCHED_FUSED, X, A, B, gY)
    for a, b in zip(first[:2], again[:2]):
        assert np.array_equal(host_bits(a), host_bits(b))


def test_fused_split_last_round(lib):
    """80 output tiles on a GB300's 76 CTA pairs: one whole round, then 4 tiles shared by 8 pairs each
    (one shard per pair, the partials added by each tile's head).  Bit-identical to the two-stream
    schedule, and the rows of the split tiles (rows 4096 - 5119, columns 768 - 1023 in the tile
    order) against the oracle."""
    M, h, Fi, t, p, q = 5120, 1024, 128, 8, 1, 1
    X, A, B, gY = inputs(M, h, Fi, t, synth.ACT_GELU, 56, integer=False)
    Y, gX, _, _ = fwd_bwd(lib, M, h, Fi, t, p, q, synth.ACT_GELU, dm.SCHED_FUSED, X, A, B, gY)
    Y2, gX2, _, _ = fwd_bwd(lib, M, h, Fi, t, p, q, synth.ACT_GELU, dm.SCHED_INTRA, X, A, B, gY)
    assert np.array_equal(host_bits(Y), host_bits(Y2)), "Y differs from the two-stream schedule"
    assert np.array_equal(host_bits(gX), host_bits(gX2)), "gX differs from the two-stream schedule"
    rows = np.unique(np.array([4096, 4097, 4351, 4352, 4607, 4863, 5118, 5119] + list(synth.sample_indices(M, 4, 57))))
    Yr = host_f64(Y)[rows]
    assert_tol(Yr, oracle.mlp_fwd(X, A, B, t, synth.ACT_GELU, rows=rows), "Y rows of the split tiles")


def test_fused_stack_forward_and_backward(lib):
    """Layer stack: the fused epilogue adds the residual (in place for layers after the first)."""
    import torch
    s = synth.MlpShape("fs", 512, 128, 256, synth.ACT_GELU, 2, 2, 2, layers=3, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=54)
    outs = {}
    for sched in (dm.SCHED_FUSED, dm.SCHED_INTER):
        cfg = dm.make_cfg(s.M, s.h, s.F, s.t, s.p, s.q, s.act, sched=sched, layers=s.layers, ln_eps=1e-5)
        Z, A, B, gZ = dev_bf16(d["X"]), dev_bf16(d["A"]), dev_bf16(d["B"]), dev_bf16(d["gY"])
        out = torch.empty_like(Z)
        save = torch.empty(dm.domino_stack_save_size(cfg), dtype=torch.uint8, device="cuda")
        ws = torch.empty(max(dm.domino_workspace_size(cfg, dm.PASS_STACK),
                             dm.domino_workspace_size(cfg, dm.PASS_STACK_BWD)), dtype=torch.uint8, device="cuda")
        dm.domino_stack_fwd_train(lib.h, cfg, Z, A, B, out, save, ws)
        gZin = torch.empty_like(Z)
        gA = torch.zeros(d["A"].shape, dtype=torch.float32, device="cuda")
        gB = torch.zeros(d["B"].shape, dtype=torch.float32, device="cuda")
        dm.domino_stack_bwd(lib.h, cfg, A, B, save, gZ, gZin, gA, gB, ws)
        out_inf = lib.stack(cfg, Z, A, B)
        torch.cuda.synchronize()
        outs[sched] = (out, gZin, out_inf)
    f, r = outs[dm.SCHED_FUSED], outs[dm.SCHED_INTER]
    assert_tol(host_f64(f[0]), oracle.stack_fwd(d["X"], d["A"], d["B"], s.t, s.act, 1e-5), "stack output")
    gZ0, _, _ = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], s.t, s.act, 1e-5)
    assert_tol(host_f64(f[1]), gZ0, "stack input gradient")
    for a, b, what in zip(f, r, ("output", "input gradient", "inference output")):
        assert np.array_equal(host_bits(a), host_bits(b)), what


@pytest.mark.slow
def test_fused_full_size_fwd_bwd(lib):
    """The forward+backward workload at full size: sampled rows against the oracle, and bit-identical
    to the two-stream schedule everywhere."""
    import torch
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    d = synth.make_inputs(s, seed=0)
    res = {}
    for sched in (dm.SCHED_FUSED, dm.SCHED_INTRA):
        Y, gX, _, _ = fwd_bwd(lib, s.M, s.h, s.Fi, s.t, s.p, s.q, s.act, sched, d["X"], d["A"][0], d["B"][0], d["gY"])
        res[sched] = (host_bits(Y), host_bits(gX))
        del Y, gX
        torch.cuda.empty_cache()
    for a, b in zip(res[dm.SCHED_FUSED], res[dm.SCHED_INTRA]):
        assert np.array_equal(a, b)
    rows = synth.sample_indices(s.M, 6, 55)
    Yf = synth.bf16_bits_to_f32(res[dm.SCHED_FUSED][0][rows]).astype(np.float64)
    assert_tol(Yf, oracle.mlp_fwd(d["X"], d["A"][0], d["B"][0], s.t, s.act, rows=rows), "Y sampled rows")
