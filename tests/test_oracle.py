"""Pins for the CPU oracle (no GPU).

The oracle is checked against things fixed independently of it: hand-worked
examples (tests/golden), exact integer brute force with numpy int64 matmul,
float64 library routines (numpy matmul, torch's gelu/silu/layer_norm) on small
inputs, central finite differences for the backward, and invariants the pages
state (shard sum == unsharded product; row subsets are rows of the whole).
"""
import math

import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import synth
from conftest import load_golden

ACTS_PLAIN = [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_GELU]
ACTS_GATED = [oracle.ACT_SWIGLU, oracle.ACT_BILINEAR]


def full_weights(A, B, t, gated):
    """Unsharded weights assembled by slicing/concatenation (independent of the C indexing)."""
    Bfull = np.concatenate([B[i] for i in range(t)], axis=1)  # h x F
    if not gated:
        return A, None, Bfull
    a_rows = A.shape[0]
    Fi = a_rows // (2 * t)
    gate = np.concatenate([A[i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)], axis=0)
    up = np.concatenate([A[i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)], axis=0)
    return gate, up, Bfull


def np_act(act, z):
    import torch
    zt = torch.from_numpy(np.asarray(z, dtype=np.float64))
    if act == oracle.ACT_RELU:
        return torch.relu(zt).numpy()
    if act == oracle.ACT_GELU:
        return torch.nn.functional.gelu(zt, approximate="none").numpy()
    return zt.numpy()


def np_glu(act, g, u):
    import torch
    if act == oracle.ACT_SWIGLU:
        return torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
    return g * u


def small_case(M, h, F, t, act, seed, integer=False):
    s = synth.MlpShape("t", M, h, F, act, t, 1, 1, backward=True)
    d = synth.make_inputs(s, seed=seed, integer=integer)
    return d["X"], d["A"][0], d["B"][0], d["gY"]


# ---------------------------------------------------------------- golden (hand-worked)

def test_golden_relu_worked_example():
    g = load_golden("relu_t2_worked.txt")
    t = int(g["t"])
    X, A = g["X"], g["A"]
    B = g["B"].reshape(t, 2, -1)
    Y = oracle.mlp_fwd(X, A, B, t, oracle.ACT_RELU)
    assert np.array_equal(Y, g["Y"])
    Ys = oracle.mlp_fwd(X, A, B, t, oracle.ACT_RELU, sharded=True)
    assert np.array_equal(Ys, g["P0"] + g["P1"])
    dX, dA, dB = oracle.mlp_bwd(X, A, B, g["gY"], t, oracle.ACT_RELU)
    assert np.array_equal(dX, g["dX"])
    assert np.array_equal(dA[:, 0, :], g["dA"])
    # golden dB is stored shard-wise (t, h, F_i); oracle dB is [f, c] = dL/dBfull[c, f]
    dBfull = dB.T
    assert np.array_equal(np.concatenate(np.split(dBfull, t, axis=1), axis=0), g["dB"])


def test_golden_bilinear_worked_example():
    g = load_golden("bilinear_t2_worked.txt")
    t = int(g["t"])
    B = g["B"].reshape(t, 2, -1)
    Y = oracle.mlp_fwd(g["X"], g["A"], B, t, oracle.ACT_BILINEAR)
    assert np.array_equal(Y, g["Y"])


# ---------------------------------------------------------------- integer brute force

@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_BILINEAR])
@pytest.mark.parametrize("t", [1, 2, 3])
def test_integer_exact_vs_int64_bruteforce(act, t):
    M, h, F = 7, 10, 6 * t
    X, A, B, gY = small_case(M, h, F, t, act, seed=11 + t, integer=True)
    Xi = synth.bf16_bits_to_f32(X).astype(np.int64)
    Ai = synth.bf16_bits_to_f32(A).astype(np.int64)
    Bi = synth.bf16_bits_to_f32(B).astype(np.int64)
    gYi = synth.bf16_bits_to_f32(gY).astype(np.int64)
    gated = act == oracle.ACT_BILINEAR
    gate, up, Bfull = full_weights(Ai, Bi, t, gated)
    if gated:
        G, U = Xi @ gate.T, Xi @ up.T
        H = G * U
    else:
        Z = Xi @ gate.T
        H = np.maximum(Z, 0) if act == oracle.ACT_RELU else Z
    Y = H @ Bfull.T
    assert np.array_equal(oracle.mlp_fwd(X, A, B, t, act), Y.astype(np.float64))
    assert np.array_equal(oracle.mlp_fwd(X, A, B, t, act, sharded=True), Y.astype(np.float64))
    # backward
    dH = gYi @ Bfull
    if gated:
        dG, dU = dH * U, dH * G
        dX = dG @ gate + dU @ up
        dAg, dAu = dG.T @ Xi, dU.T @ Xi
    else:
        dZ = dH * (Z > 0) if act == oracle.ACT_RELU else dH
        dX = dZ @ gate
        dAg = dZ.T @ Xi
    dBfull = gYi.T @ H
    oX, oA, oB = oracle.mlp_bwd(X, A, B, gY, t, act)
    assert np.array_equal(oX, dX.astype(np.float64))
    assert np.array_equal(oA[:, 0, :], dAg.astype(np.float64))
    if gated:
        assert np.array_equal(oA[:, 1, :], dAu.astype(np.float64))
    assert np.array_equal(oB, dBfull.T.astype(np.float64))


# ---------------------------------------------------------------- library fp64 routines

@pytest.mark.parametrize("act", ACTS_PLAIN + ACTS_GATED)
@pytest.mark.parametrize("t", [1, 2, 4])
def test_fwd_matches_float64_library(act, t):
    M, h, F = 9, 24, 8 * t
    X, A, B, _ = small_case(M, h, F, t, act, seed=3)
    Xf, Af, Bf = (synth.bf16_bits_to_f32(a).astype(np.float64) for a in (X, A, B))
    gated = act in ACTS_GATED
    gate, up, Bfull = full_weights(Af, Bf, t, gated)
    H = np_glu(act, Xf @ gate.T, Xf @ up.T) if gated else np_act(act, Xf @ gate.T)
    ref = H @ Bfull.T
    Y = oracle.mlp_fwd(X, A, B, t, act)
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-13)
    # the double-input entry point sees the same values
    Y64 = oracle.mlp_fwd(Xf, Af, Bf, t, act)
    np.testing.assert_allclose(Y64, Y, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("act", [oracle.ACT_GELU, oracle.ACT_SWIGLU])
@pytest.mark.parametrize("t", [1, 2, 3, 8])
def test_shard_sum_equals_unsharded(act, t):
    """Sum over the t shard partials == the unsharded product (row-split distributivity)."""
    M, h, F = 6, 32, 4 * t
    X, A, B, _ = small_case(M, h, F, t, act, seed=5)
    Y = oracle.mlp_fwd(X, A, B, t, act)
    Ys = oracle.mlp_fwd(X, A, B, t, act, sharded=True)
    np.testing.assert_allclose(Ys, Y, rtol=1e-12, atol=1e-14)


def test_row_subset_equals_rows_of_whole():
    M, h, F, t = 16, 16, 32, 4
    X, A, B, gY = small_case(M, h, F, t, oracle.ACT_SWIGLU, seed=9)
    rows = np.array([0, 3, 7, 15])
    assert np.array_equal(oracle.mlp_fwd(X, A, B, t, oracle.ACT_SWIGLU, rows=rows),
                          oracle.mlp_fwd(X, A, B, t, oracle.ACT_SWIGLU)[rows])
    dX, _, _ = oracle.mlp_bwd(X, A, B, gY, t, oracle.ACT_SWIGLU, want_dw=False)
    dXs, _, _ = oracle.mlp_bwd(X, A, B, gY, t, oracle.ACT_SWIGLU, rows=rows, want_dw=False)
    assert np.array_equal(dXs, dX[rows])
    feats = np.array([1, 8, 31])
    _, dA, dB = oracle.mlp_bwd(X, A, B, gY, t, oracle.ACT_SWIGLU, want_dx=False)
    _, dAs, dBs = oracle.mlp_bwd(X, A, B, gY, t, oracle.ACT_SWIGLU, feats=feats, want_dx=False)
    assert np.array_equal(dAs, dA[feats]) and np.array_equal(dBs, dB[feats])


def test_row_chunks_concatenate_to_whole():
    """Row split of X (the batch dimension): chunk results stacked == unsplit result."""
    M, h, F, t, p = 12, 16, 16, 2, 3
    X, A, B, _ = small_case(M, h, F, t, oracle.ACT_GELU, seed=21)
    whole = oracle.mlp_fwd(X, A, B, t, oracle.ACT_GELU)
    m = M // p
    parts = [oracle.mlp_fwd(X[k * m:(k + 1) * m], A, B, t, oracle.ACT_GELU) for k in range(p)]
    assert np.array_equal(np.concatenate(parts, axis=0), whole)


# ---------------------------------------------------------------- elementwise functions

def test_activation_special_values():
    a = oracle
    assert a.act(a.ACT_GELU, 0.0) == 0.0
    assert a.act(a.ACT_GELU, 40.0) == 40.0
    assert a.act(a.ACT_GELU, -40.0) == 0.0
    # x * Phi(x) at x=1 with Phi(1) = 0.841344746068542948585...
    assert abs(a.act(a.ACT_GELU, 1.0) - 0.8413447460685429) < 1e-15
    assert a.act(a.ACT_RELU, -2.0) == 0.0 and a.act(a.ACT_RELU, 2.5) == 2.5
    assert a.act(a.ACT_NONE, -3.25) == -3.25
    assert a.glu(a.ACT_SWIGLU, 0.0, 5.0) == 0.0
    # silu(1) = 1 / (1 + e^-1)
    assert abs(a.glu(a.ACT_SWIGLU, 1.0, 1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(a.glu(a.ACT_SWIGLU, 50.0, 2.0) - 100.0) < 1e-12
    assert a.glu(a.ACT_BILINEAR, -3.0, 4.0) == -12.0


def test_activation_vs_torch_float64():
    import torch
    z = np.linspace(-8, 8, 161)
    np.testing.assert_allclose(oracle.act(oracle.ACT_GELU, z),
                               torch.nn.functional.gelu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-16)
    sil = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    np.testing.assert_allclose([oracle.glu(oracle.ACT_SWIGLU, v, 1.0) for v in z], sil, rtol=1e-14, atol=1e-16)


@pytest.mark.parametrize("act", [oracle.ACT_GELU, oracle.ACT_RELU, oracle.ACT_NONE])
def test_activation_grad_finite_difference(act):
    z = np.linspace(-5, 5, 101) + 0.013  # avoid the relu kink at 0
    eps = 1e-6
    fd = (oracle.act(act, z + eps) - oracle.act(act, z - eps)) / (2 * eps)
    np.testing.assert_allclose(oracle.act_grad(act, z), fd, rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("act", ACTS_GATED)
def test_glu_grad_finite_difference(act):
    eps = 1e-6
    for g in np.linspace(-4, 4, 17):
        for u in (-1.5, 0.25, 2.0):
            fdg = (oracle.glu(act, g + eps, u) - oracle.glu(act, g - eps, u)) / (2 * eps)
            fdu = (oracle.glu(act, g, u + eps) - oracle.glu(act, g, u - eps)) / (2 * eps)
            assert abs(oracle.glu_dg(act, g, u) - fdg) < 1e-7
            assert abs(oracle.glu_du(act, g, u) - fdu) < 1e-7


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_GELU, oracle.ACT_SWIGLU, oracle.ACT_BILINEAR])
@pytest.mark.parametrize("t", [1, 2])
def test_bwd_central_finite_differences(act, t):
    """Loss L = sum(gY * Y); oracle gradients vs central differences in double."""
    rng = np.random.default_rng(7 + act + 10 * t)
    M, h, F = 4, 8, 16
    gated = act in ACTS_GATED
    Fi = F // t
    X = rng.standard_normal((M, h))
    A = rng.standard_normal((2 * F if gated else F, h)) * 0.5
    B = rng.standard_normal((t, h, Fi)) * 0.5
    gY = rng.standard_normal((M, h))

    def loss(X_, A_, B_):
        return float(np.sum(gY * oracle.mlp_fwd(X_, A_, B_, t, act)))

    dX, dA, dB = oracle.mlp_bwd(X, A, B, gY, t, act)
    eps = 1e-6
    for arr, grad_of in ((X, lambda i: dX.flat[i]),):
        for i in range(0, arr.size, 3):
            a1, a2 = arr.copy(), arr.copy()
            a1.flat[i] += eps
            a2.flat[i] -= eps
            fd = (loss(a1, A, B) - loss(a2, A, B)) / (2 * eps)
            assert abs(fd - grad_of(i)) < 1e-6 * max(1.0, abs(fd))
    # A storage gradient from the oracle's per-feature layout
    dA_store = np.zeros_like(A)
    for f in range(F):
        i, j = divmod(f, Fi)
        if gated:
            dA_store[i * 2 * Fi + j] = dA[f, 0]
            dA_store[i * 2 * Fi + Fi + j] = dA[f, 1]
        else:
            dA_store[f] = dA[f, 0]
    for idx in range(0, A.size, 5):
        a1, a2 = A.copy(), A.copy()
        a1.flat[idx] += eps
        a2.flat[idx] -= eps
        fd = (loss(X, a1, B) - loss(X, a2, B)) / (2 * eps)
        assert abs(fd - dA_store.flat[idx]) < 1e-6 * max(1.0, abs(fd))
    dB_store = np.zeros_like(B)
    for f in range(F):
        i, j = divmod(f, Fi)
        dB_store[i, :, j] = dB[f]
    for idx in range(0, B.size, 3):
        b1, b2 = B.copy(), B.copy()
        b1.flat[idx] += eps
        b2.flat[idx] -= eps
        fd = (loss(X, A, b1) - loss(X, A, b2)) / (2 * eps)
        assert abs(fd - dB_store.flat[idx]) < 1e-6 * max(1.0, abs(fd))


def test_bwd_linear_in_output_gradient():
    M, h, F, t = 6, 16, 16, 2
    X, A, B, gY1 = small_case(M, h, F, t, oracle.ACT_SWIGLU, seed=31)
    gY2 = synth.normal_bf16((M, h), 0, 1, 32, 1)
    g1, g2 = (synth.bf16_bits_to_f32(g).astype(np.float64) for g in (gY1, gY2))
    Xf, Af, Bf = (synth.bf16_bits_to_f32(a).astype(np.float64) for a in (X, A, B))
    r1 = oracle.mlp_bwd(Xf, Af, Bf, g1, t, oracle.ACT_SWIGLU)
    r2 = oracle.mlp_bwd(Xf, Af, Bf, g2, t, oracle.ACT_SWIGLU)
    r12 = oracle.mlp_bwd(Xf, Af, Bf, g1 + g2, t, oracle.ACT_SWIGLU)
    for a, b, c in zip(r1, r2, r12):
        np.testing.assert_allclose(a + b, c, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- layernorm and stack

def test_layernorm_moments_and_library():
    import torch
    Z = synth.normal_bf16((8, 64), 0.5, 2.0, 1, 1)
    Zf = synth.bf16_bits_to_f32(Z).astype(np.float64)
    eps = 1e-5
    out = oracle.layernorm(Z, eps)
    np.testing.assert_allclose(out.mean(axis=1), 0.0, atol=1e-13)
    v = Zf.var(axis=1)
    np.testing.assert_allclose(out.var(axis=1), v / (v + eps), rtol=1e-12)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(Zf), (64,), eps=eps).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_stack_matches_float64_composition():
    import torch
    L, M, h, F, t, act = 3, 5, 32, 64, 4, oracle.ACT_GELU
    s = synth.MlpShape("s", M, h, F, act, t, 1, 1, layers=L, layernorm=True)
    d = synth.make_inputs(s, seed=4)
    Z = synth.bf16_bits_to_f32(d["X"]).astype(np.float64)
    for l in range(L):
        Af = synth.bf16_bits_to_f32(d["A"][l]).astype(np.float64)
        Bf = synth.bf16_bits_to_f32(d["B"][l]).astype(np.float64)
        _, _, Bfull = full_weights(Af, Bf, t, False)
        ln = torch.nn.functional.layer_norm(torch.from_numpy(Z), (h,), eps=1e-5).numpy()
        Z = Z + np_act(act, ln @ Af.T) @ Bfull.T
    out = oracle.stack_fwd(d["X"], d["A"], d["B"], t, act, 1e-5)
    np.testing.assert_allclose(out, Z, rtol=1e-11, atol=1e-11)
    # zero layers is the identity
    z0 = oracle.stack_fwd(d["X"], d["A"][:0], d["B"][:0], t, act, 1e-5)
    assert np.array_equal(z0, synth.bf16_bits_to_f32(d["X"]).astype(np.float64))


def test_rejects_bad_sizes():
    X = np.zeros((2, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.mlp_fwd(X, np.zeros((3, 4), np.uint16), np.zeros((2, 4, 2), np.uint16), 2, oracle.ACT_GELU)


def test_seeded_inputs_are_deterministic_bf16():
    a = synth.normal_bf16((3, 5), 0, 1, 0, synth.TID_X)
    b = synth.normal_bf16((3, 5), 0, 1, 0, synth.TID_X)
    assert np.array_equal(a, b)
    f = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3], np.float32)
    # 1+2^-8 is a tie between bf16 neighbours 1 and 1+2^-7: ties go to even (1.0)
    assert np.array_equal(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(f))[:2], [1.0, 1.0])
    assert synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(f))[2] == np.float32(1.0078125)


# ---------------------------------------------------------------- stack backward

def _torch_stack(Z, A, B, t, act, eps):
    """float64 autograd reference of the pre-LN residual stack (library routines)."""
    import torch
    gated = act in ACTS_GATED
    z = Z
    for l in range(A.shape[0]):
        Bfull = torch.cat([B[l][i] for i in range(t)], dim=1)
        if gated:
            Fi = A.shape[1] // (2 * t)
            gate = torch.cat([A[l][i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)], dim=0)
            up = torch.cat([A[l][i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)], dim=0)
        else:
            gate = A[l]
        n = torch.nn.functional.layer_norm(z, (z.shape[1],), eps=eps)
        if gated:
            g, u = n @ gate.T, n @ up.T
            hact = (torch.nn.functional.silu(g) * u) if act == oracle.ACT_SWIGLU else g * u
        else:
            zz = n @ gate.T
            hact = {oracle.ACT_GELU: torch.nn.functional.gelu, oracle.ACT_RELU: torch.relu}.get(act, lambda v: v)(zz)
        z = z + hact @ Bfull.T
    return z


@pytest.mark.parametrize("act", [oracle.ACT_GELU, oracle.ACT_SWIGLU, oracle.ACT_NONE])
def test_stack_bwd_matches_float64_autograd(act):
    import torch
    L, M, h, F, t = 3, 5, 16, 32, 2
    s = synth.MlpShape("sb", M, h, F, act, t, 1, 1, layers=L, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=12)
    d["A"] = synth.normal_bf16(d["A"].shape, 0, 0.3, 12, synth.TID_A)  # larger weights: non-trivial LN paths
    Zf, Af, Bf, gf = (synth.bf16_bits_to_f32(d[k]).astype(np.float64) for k in ("X", "A", "B", "gY"))
    Zt = torch.from_numpy(Zf).requires_grad_(True)
    At = torch.from_numpy(Af).requires_grad_(True)
    Bt = torch.from_numpy(Bf).requires_grad_(True)
    out = _torch_stack(Zt, At, Bt, t, act, 1e-5)
    out.backward(torch.from_numpy(gf))
    gZ0, dA, dB = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], t, act, 1e-5, want_w=True)
    np.testing.assert_allclose(gZ0, Zt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dA, At.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dB, Bt.grad.numpy(), rtol=1e-9, atol=1e-11)
    # the double-input entry point agrees
    gZ0_64, dA64, dB64 = oracle.stack_bwd(Zf, Af, Bf, gf, t, act, 1e-5, want_w=True)
    np.testing.assert_allclose(gZ0_64, gZ0, rtol=1e-13, atol=1e-15)


def test_stack_bwd_rows_and_identity():
    L, M, h, F, t, act = 2, 9, 16, 32, 4, oracle.ACT_GELU
    s = synth.MlpShape("sb", M, h, F, act, t, 1, 1, layers=L, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=13)
    full, _, _ = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], t, act)
    rows = np.array([0, 4, 8])
    part, _, _ = oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], t, act, rows=rows)
    assert np.array_equal(part, full[rows])
    # zero layers: the gradient passes through unchanged
    g0, _, _ = oracle.stack_bwd(d["X"], d["A"][:0], d["B"][:0], d["gY"], t, act)
    assert np.array_equal(g0, synth.bf16_bits_to_f32(d["gY"]).astype(np.float64))
    with pytest.raises(ValueError):
        oracle.stack_bwd(d["X"], d["A"], d["B"], d["gY"], t, act, rows=rows, want_w=True)
