"""Degenerate splits of the chunked MLP, exact on integer inputs: row chunks of a single token
(p = M), column chunks of 8 outputs (the narrowest h / q the 16-byte rows allow), shards of 8 ffn
features (many emulated ranks, each far narrower than one tile), and all of them together.  Every
tile of these launches is a ragged edge tile.  Forward and backward outputs must equal the oracle
exactly (the integer intermediates are exact in bf16 and fp32) under every schedule, and the
row-local outputs (Y, the saved activation, gX) must equal the unsplit run bit for bit."""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import Lib, bf16_round, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu

SCHEDS = [dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_INTER, dm.SCHED_FUSED]

# (M, h, F_i, t, p, q)
SHAPES = [
    (24, 64, 8, 2, 24, 1),     # one-token row chunks
    (64, 64, 8, 16, 1, 8),     # 16 shards of 8 features; 8-column chunks
    (40, 128, 24, 3, 5, 16),   # 8 x 8 chunks of a 40 x 128 output, 3 shards of 24 features
]


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


def int_case(M, h, Fi, t, act, seed):
    gated = act in synth.GATED
    pz = 0.8 if gated else 0.5
    a_rows = (2 if gated else 1) * Fi * t
    X = synth.ternary_bf16((M, h), seed, synth.TID_X, p_zero=pz)
    A = synth.ternary_bf16((a_rows, h), seed, synth.TID_A, p_zero=pz)
    B = synth.ternary_bf16((t, h, Fi), seed, synth.TID_B, p_zero=pz)
    gY = synth.ternary_bf16((M, h), seed, synth.TID_GY, p_zero=pz)
    return X, A, B, gY, a_rows


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_RELU, synth.ACT_BILINEAR])
def test_degenerate_splits_forward_exact(lib, shape, act):
    M, h, Fi, t, p, q = shape
    X, A, B, _, _ = int_case(M, h, Fi, t, act, 60 + act + M)
    Yref, Href = oracle.mlp_fwd(X, A, B, t, act, return_h=True)
    assert np.max(np.abs(Href)) <= 256, "test precondition: H exact in bf16"
    dX, dA, dB = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    base, bsave = lib.fwd(dm.make_cfg(M, h, Fi * t, t, 1, 1, act), dX, dA, dB, save=True)
    assert np.array_equal(host_f64(base), bf16_round(Yref))
    for sched in SCHEDS:
        Y, S = lib.fwd(dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=sched), dX, dA, dB, save=True)
        assert np.array_equal(host_bits(Y), host_bits(base)), sched
        assert np.array_equal(host_bits(S), host_bits(bsave)), sched


@pytest.mark.parametrize("shape", SHAPES)
def test_degenerate_splits_backward_exact(lib, shape):
    import torch
    M, h, Fi, t, p, q = shape
    act = synth.ACT_BILINEAR
    X, A, B, gY, a_rows = int_case(M, h, Fi, t, act, 70 + M)
    # precondition: the bf16 intermediates dG = dH U, dU = dH G and H = G U are exact (int64 algebra)
    Xi, Ai, Bi, gYi = (synth.bf16_bits_to_f32(v).astype(np.int64) for v in (X, A, B, gY))
    dH = gYi @ np.concatenate(list(Bi), axis=1)
    G = Xi @ np.concatenate([Ai[i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)]).T
    U = Xi @ np.concatenate([Ai[i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)]).T
    assert max(np.abs(dH * U).max(), np.abs(dH * G).max(), np.abs(G * U).max()) <= 256
    dXr, dAf, dBf = oracle.mlp_bwd(X, A, B, gY, t, act)
    dA_ref = np.concatenate([np.concatenate([dAf[i * Fi:(i + 1) * Fi, 0], dAf[i * Fi:(i + 1) * Fi, 1]])
                             for i in range(t)])
    dB_ref = np.stack([dBf[i * Fi:(i + 1) * Fi].T for i in range(t)])
    dX, dA, dB, dgY = dev_bf16(X), dev_bf16(A), dev_bf16(B), dev_bf16(gY)
    gA0 = torch.zeros((a_rows, h), dtype=torch.float32, device="cuda")
    gB0 = torch.zeros((t, h, Fi), dtype=torch.float32, device="cuda")
    base = None
    for pp, qq, sched in [(1, 1, dm.SCHED_SERIAL)] + [(p, q, s) for s in SCHEDS]:
        cfg = dm.make_cfg(M, h, Fi * t, t, pp, qq, act, sched=sched)
        _, S = lib.fwd(cfg, dX, dA, dB, save=True)
        gX, gA, gB = lib.bwd(cfg, dX, dA, dB, S, dgY, gA0, gB0)
        assert np.array_equal(host_f64(gX), bf16_round(dXr)), (pp, qq, sched)
        assert np.array_equal(gA.cpu().numpy().astype(np.float64), dA_ref), (pp, qq, sched)
        assert np.array_equal(gB.cpu().numpy().astype(np.float64), dB_ref), (pp, qq, sched)
        if base is None:
            base = host_bits(gX)
        assert np.array_equal(host_bits(gX), base), (pp, qq, sched)
