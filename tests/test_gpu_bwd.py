"""GPU parity of the backward pass (domino_mlp_bwd) and of the layer stack (domino_stack_fwd)
against the CPU oracle."""
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


def shard_major_dA(dA_feat, t, Fi, gated):
    """Oracle dA [f, R, h] -> A storage layout [t * R * F_i, h]."""
    rows = []
    for i in range(t):
        if gated:
            rows.append(dA_feat[i * Fi:(i + 1) * Fi, 0])
            rows.append(dA_feat[i * Fi:(i + 1) * Fi, 1])
        else:
            rows.append(dA_feat[i * Fi:(i + 1) * Fi, 0])
    return np.concatenate(rows, axis=0)


def shard_major_dB(dB_feat, t, Fi):
    """Oracle dB [f, h] -> B storage layout [t, h, F_i]."""
    return np.stack([dB_feat[i * Fi:(i + 1) * Fi].T for i in range(t)])


def run_case(lib, M, h, Fi, t, p, q, act, X, A, B, gY, gA0, gB0, sched=dm.SCHED_INTRA):
    import torch
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=sched)
    dX_, dA_, dB_ = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    _, S = lib.fwd(cfg, dX_, dA_, dB_, save=True)
    gX, gA, gB = lib.bwd(cfg, dX_, dA_, dB_, S, dev_bf16(gY), torch.from_numpy(gA0).cuda(),
                         torch.from_numpy(gB0).cuda())
    return gX, gA.cpu().numpy().astype(np.float64), gB.cpu().numpy().astype(np.float64)


INT_SHAPES = [
    (384, 208, 136, 3, 2, 2),
    (256, 64, 64, 1, 1, 1),
    (264, 72, 40, 4, 3, 3),
    # 8190 tokens in one chunk: weight gradients over a long token range (128 K steps, the last
    # one ragged), still exact in fp32
    (8190, 64, 64, 2, 1, 1),
]


@pytest.mark.parametrize("shape", INT_SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_NONE, synth.ACT_RELU, synth.ACT_BILINEAR])
def test_bwd_integer_bit_exact(lib, shape, act):
    M, h, Fi, t, p, q = shape
    gated = act in synth.GATED
    pz = 0.85 if gated else 0.5
    a_rows = (2 if gated else 1) * Fi * t
    X = synth.ternary_bf16((M, h), 40 + act, synth.TID_X, p_zero=pz)
    A = synth.ternary_bf16((a_rows, h), 40 + act, synth.TID_A, p_zero=pz)
    B = synth.ternary_bf16((t, h, Fi), 40 + act, synth.TID_B, p_zero=pz)
    gY = synth.ternary_bf16((M, h), 40 + act, synth.TID_GY, p_zero=pz)
    # integer initial main_grad values check the += accumulation
    rng = np.random.default_rng(act)
    gA0 = rng.integers(-3, 4, size=(a_rows, h)).astype(np.float32)
    gB0 = rng.integers(-3, 4, size=(t, h, Fi)).astype(np.float32)
    dX, dAf, dBf = oracle.mlp_bwd(X, A, B, gY, t, act)
    # preconditions: the bf16 intermediates (dZ, H) are exact; checked with int64 algebra
    Xi, Ai, Bi, gYi = (synth.bf16_bits_to_f32(v).astype(np.int64) for v in (X, A, B, gY))
    Bfull = np.concatenate(list(Bi), axis=1)
    dH = gYi @ Bfull
    if gated:
        gate = np.concatenate([Ai[i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)])
        up = np.concatenate([Ai[i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)])
        G, U = Xi @ gate.T, Xi @ up.T
        assert max(np.abs(dH * U).max(), np.abs(dH * G).max(), np.abs(G * U).max()) <= 256
    gX, gA, gB = run_case(lib, M, h, Fi, t, p, q, act, X, A, B, gY, gA0, gB0)
    assert np.array_equal(host_f64(gX), bf16_round(dX))
    assert np.array_equal(gA, gA0 + shard_major_dA(dAf, t, Fi, gated))
    assert np.array_equal(gB, gB0 + shard_major_dB(dBf, t, Fi))


REAL_SHAPES = [
    (256, 256, 128, 2, 2, 1),
    (320, 192, 200, 3, 2, 2),
    (16380, 128, 64, 2, 2, 1),  # two row chunks of 8190 tokens: long-K weight gradients
]


@pytest.mark.parametrize("shape", REAL_SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_bwd_matches_oracle(lib, shape, act):
    M, h, Fi, t, p, q = shape
    gated = act in synth.GATED
    a_rows = (2 if gated else 1) * Fi * t
    X = synth.normal_bf16((M, h), 0, 1, 1, synth.TID_X)
    A = synth.normal_bf16((a_rows, h), 0, 0.02, 1, synth.TID_A)
    B = synth.normal_bf16((t, h, Fi), 0, 0.02, 1, synth.TID_B)
    gY = synth.normal_bf16((M, h), 0, 1, 1, synth.TID_GY)
    gA0 = synth.normal_f32((a_rows, h), 0, 0.01, 1, synth.TID_GA0)
    gB0 = synth.normal_f32((t, h, Fi), 0, 0.01, 1, synth.TID_GB0)
    dX, dAf, dBf = oracle.mlp_bwd(X, A, B, gY, t, act)
    gX, gA, gB = run_case(lib, M, h, Fi, t, p, q, act, X, A, B, gY, gA0, gB0)
    assert_tol(host_f64(gX), dX, "gX")
    assert_tol(gA - gA0, shard_major_dA(dAf, t, Fi, gated), "gA increment")
    assert_tol(gB - gB0, shard_major_dB(dBf, t, Fi), "gB increment")


def test_bwd_row_split_gx_bit_identical(lib):
    import torch
    M, h, Fi, t, act = 512, 256, 128, 4, synth.ACT_SWIGLU
    X = synth.normal_bf16((M, h), 0, 1, 2, synth.TID_X)
    A = synth.normal_bf16((2 * Fi * t, h), 0, 0.02, 2, synth.TID_A)
    B = synth.normal_bf16((t, h, Fi), 0, 0.02, 2, synth.TID_B)
    gY = synth.normal_bf16((M, h), 0, 1, 2, synth.TID_GY)
    z = np.zeros((2 * Fi * t, h), np.float32), np.zeros((t, h, Fi), np.float32)
    outs = [run_case(lib, M, h, Fi, t, p, 1, act, X, A, B, gY, *z) for p in (1, 2, 4)]
    base = host_bits(outs[0][0])
    for o in outs[1:]:
        assert np.array_equal(host_bits(o[0]), base)
        # weight gradients sum over tokens, so a row split reorders their fp32 adds
        assert_tol(o[1], outs[0][1], "gA across p")
        assert_tol(o[2], outs[0][2], "gB across p")


def test_stack_matches_oracle(lib):
    L, M, h, F, t, p, q, act = 3, 256, 128, 256, 2, 2, 2, synth.ACT_GELU
    s = synth.MlpShape("s", M, h, F, act, t, p, q, layers=L, layernorm=True)
    d = synth.make_inputs(s, seed=8)
    ref = oracle.stack_fwd(d["X"], d["A"], d["B"], t, act, 1e-5)
    outs = []
    for sched in (dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_INTER):
        cfg = dm.make_cfg(M, h, F, t, p, q, act, sched=sched, layers=L, ln_eps=1e-5)
        Z = lib.stack(cfg, dev_bf16(d["X"]), dev_bf16(d["A"]), dev_bf16(d["B"]))
        outs.append(host_bits(Z))
        assert_tol(host_f64(Z), ref, f"stack sched={sched}")
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_stack_in_place(lib):
    import torch
    L, M, h, F, t, act = 2, 128, 64, 128, 2, synth.ACT_GELU
    s = synth.MlpShape("s", M, h, F, act, t, 2, 1, layers=L, layernorm=True)
    d = synth.make_inputs(s, seed=9)
    cfg = dm.make_cfg(M, h, F, t, 2, 1, act, layers=L, ln_eps=1e-5)
    Z = dev_bf16(d["X"])
    ref = host_bits(lib.stack(cfg, Z, dev_bf16(d["A"]), dev_bf16(d["B"])))
    ws, n = lib.workspace(cfg, dm.PASS_STACK)
    dm.domino_stack_fwd(lib.h, cfg, Z, dev_bf16(d["A"]), dev_bf16(d["B"]), Z, ws, n)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(Z), ref)
