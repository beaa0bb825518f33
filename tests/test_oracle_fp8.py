"""Pins of the FP8 oracle (oracle_fp8.c) against PyTorch's float8_e4m3fn conversions (a library
routine), the E4M3 definition (saturation, NaN), and exact integer arithmetic.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from comm_overlap_gb300 import synth


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got, ref = oracle.e4m3_decode(codes), torch_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(got).sum() == 2  # 0x7F, 0xFF
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_encode_representable_values_and_ties():
    vals = torch_decode(np.arange(256, dtype=np.uint8))
    finite = np.sort(np.unique(vals[~np.isnan(vals)]))
    # every finite value encodes to a code of that value (+0 and -0 both exist)
    assert np.array_equal(oracle.e4m3_decode(oracle.e4m3_encode(finite)), finite)
    # midpoints between neighbours: ties to the even code, as the library rounds
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(mids), torch_encode(mids))


def test_encode_random_values_match_the_library():
    g = np.random.default_rng(0)
    x = np.concatenate([g.normal(0, 1, 4000), g.normal(0, 100, 4000), g.normal(0, 1e-3, 2000),
                        g.uniform(-463.9, 463.9, 2000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_encode_saturates_and_keeps_nan():
    big = np.array([464.0, 470.0, 479.9, 480.0, 1e6, np.inf], dtype=np.float64)
    assert np.all(oracle.e4m3_encode(big) == 0x7E) and np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode([np.nan])[0] == 0x7F


def fp8_inputs(M, h, Fi, t, act, seed):
    gated = act in synth.GATED
    a_rows = (2 if gated else 1) * Fi * t
    X8 = synth.e4m3_codes((M, h), 1.0, 2.0 ** -6, seed, synth.TID_X)
    A8 = synth.e4m3_codes((a_rows, h), 0.02, 2.0 ** -11, seed, synth.TID_A)
    B8 = synth.e4m3_codes((t, h, Fi), 0.02, 2.0 ** -11, seed, synth.TID_B)
    return X8, A8, B8


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU, synth.ACT_RELU])
@pytest.mark.parametrize("t", [1, 2, 4])
def test_fp8_forward_matches_a_library_composition(act, t):
    M, h, Fi = 24, 48, 16
    X8, A8, B8 = fp8_inputs(M, h, Fi, t, act, 10 + t)
    scales = (2.0 ** -6, 2.0 ** -11, 2.0 ** -11, 2.0 ** -7)
    sx, sa, sb, sh = scales
    Y, H8 = oracle.mlp_fwd_fp8(X8, A8, B8, t, act, scales, return_h8=True)
    # the same definition with numpy matmuls and the library's conversions
    X = torch_decode(X8) * sx
    A = torch_decode(A8) * sa
    Bfull = np.concatenate(list(torch_decode(B8) * sb), axis=1)
    if act in synth.GATED:
        gate = np.concatenate([A[i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)])
        up = np.concatenate([A[i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)])
        G, U = X @ gate.T, X @ up.T
        H = torch.nn.functional.silu(torch.from_numpy(G)).numpy() * U
    else:
        Z = torch.from_numpy(X @ A.T)
        H = (torch.nn.functional.gelu(Z) if act == synth.ACT_GELU else torch.relu(Z)).numpy()
    q = np.clip((H / sh).astype(np.float32), -448, 448)
    ref_codes = torch_encode(q)
    # H/sh is formed in double in both; codes may differ only where a double quotient rounds to
    # fp32 differently from numpy's, i.e. never for these sizes
    assert np.array_equal(H8, ref_codes)
    ref = (torch_decode(ref_codes) * sh) @ Bfull.T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [synth.ACT_RELU, synth.ACT_BILINEAR])
def test_fp8_forward_integer_exact(act):
    """Codes of -1, 0, +1 and unit scales: every value is a small integer (|H| <= 16 is exact in E4M3)
    and Y equals the int64 brute force."""
    M, h, Fi, t = 16, 8, 8, 2
    g = np.random.default_rng(act)
    gated = act in synth.GATED
    a_rows = (2 if gated else 1) * Fi * t
    lut = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)  # -1, 0, +1
    pz = 0.7 if gated else 0.34  # sparse enough that |H| stays <= 16
    probs = [(1 - pz) / 2, pz, (1 - pz) / 2]
    Xi = g.choice([-1, 0, 1], size=(M, h), p=probs)
    Ai = g.choice([-1, 0, 1], size=(a_rows, h), p=probs)
    Bi = g.choice([-1, 0, 1], size=(t, h, Fi), p=probs)
    Y = oracle.mlp_fwd_fp8(lut[Xi + 1], lut[Ai + 1], lut[Bi + 1], t, act, (1.0, 1.0, 1.0, 1.0))
    if gated:
        gate = np.concatenate([Ai[i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)])
        up = np.concatenate([Ai[i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)])
        H = (Xi @ gate.T) * (Xi @ up.T)
    else:
        H = np.maximum(Xi @ Ai.T, 0)
    assert np.abs(H).max() <= 16
    ref = H @ np.concatenate(list(Bi), axis=1).T
    assert np.array_equal(Y, ref.astype(np.float64))
