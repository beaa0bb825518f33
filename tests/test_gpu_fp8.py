"""GPU parity of the FP8 forward (domino_mlp_fwd_fp8) against the CPU oracle (oracle_fp8.c).

Integer codes (-1, 0, +1 with unit scales) keep every value a small integer, exactly representable
in E4M3 and fp32, so those cases are compared bit for bit.  Real-valued draws are held to the
parity tolerance of the double-precision oracle, which re-quantises the first-linear output at
the same points; row splits and schedules must be bit-identical.
"""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import assert_tol, bf16_round, edge_rows, host_bits, host_f64

pytestmark = pytest.mark.gpu

SCALES = (2.0 ** -6, 2.0 ** -11, 2.0 ** -11, 2.0 ** -6)


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


def dev_u8(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def run_fp8(handle, X8, A8, B8, t, act, scales, p=1, q=1, sched=dm.SCHED_INTRA):
    import torch
    M, h = X8.shape
    Fi = B8.shape[-1]
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=sched)
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    n = dm.domino_workspace_size(cfg, dm.PASS_FWD_FP8)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    dm.domino_mlp_fwd_fp8(handle, cfg, dev_u8(X8), dev_u8(A8), dev_u8(B8), scales, Y, ws, n)
    torch.cuda.synchronize()
    return Y


# (M, h, F_i, t, p, q): several tiles and ragged tails in M, N (= h / q) and K
SHAPES = [
    (384, 256, 144, 3, 2, 2),
    (520, 144, 272, 2, 1, 1),
    (256, 128, 64, 8, 1, 1),
    (300, 400, 208, 1, 1, 1),
]


def int_codes(shape, rng, p_zero):
    lut = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)  # -1, 0, +1
    return lut[rng.choice([0, 1, 2], size=shape, p=[(1 - p_zero) / 2, p_zero, (1 - p_zero) / 2])]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_RELU, synth.ACT_BILINEAR])
def test_fp8_integer_exact(handle, shape, act):
    M, h, Fi, t, p, q = shape
    gated = act in synth.GATED
    a_rows = (2 if gated else 1) * Fi * t
    rng = np.random.default_rng(70 + act)
    # Z and H are exact integers in fp32 on both sides, so the E4M3 rounding of H (exact up to 16,
    # nearest-even above) is the same decision on both; Y sums integers exactly in fp32
    pz = 0.9 if gated else 0.75
    X8, A8, B8 = int_codes((M, h), rng, pz), int_codes((a_rows, h), rng, pz), int_codes((t, h, Fi), rng, pz)
    ref = oracle.mlp_fwd_fp8(X8, A8, B8, t, act, (1.0, 1.0, 1.0, 1.0))
    Y = run_fp8(handle, X8, A8, B8, t, act, (1.0, 1.0, 1.0, 1.0), p, q)
    assert np.array_equal(host_f64(Y), bf16_round(ref))


def real_codes(M, h, Fi, t, act, seed):
    gated = act in synth.GATED
    a_rows = (2 if gated else 1) * Fi * t
    return (synth.e4m3_codes((M, h), 1.0, SCALES[0], seed, synth.TID_X),
            synth.e4m3_codes((a_rows, h), 0.02, SCALES[1], seed, synth.TID_A),
            synth.e4m3_codes((t, h, Fi), 0.02, SCALES[2], seed, synth.TID_B))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_fp8_matches_oracle(handle, shape, act):
    M, h, Fi, t, p, q = shape
    X8, A8, B8 = real_codes(M, h, Fi, t, act, 71)
    sc = SCALES[:3] + (2.0 ** -7,)  # |H| up to ~3: H / sh stays inside the E4M3 range
    Y = run_fp8(handle, X8, A8, B8, t, act, sc, p, q)
    assert_tol(host_f64(Y), oracle.mlp_fwd_fp8(X8, A8, B8, t, act, sc), "FP8 forward")


def test_fp8_splits_and_schedules_bit_identical(handle):
    M, h, Fi, t, act = 512, 256, 128, 4, synth.ACT_SWIGLU
    X8, A8, B8 = real_codes(M, h, Fi, t, act, 72)
    sc = SCALES[:3] + (2.0 ** -7,)
    base = host_bits(run_fp8(handle, X8, A8, B8, t, act, sc))
    for sched in (dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_FUSED):
        for p, q in ((2, 1), (4, 2)):
            assert np.array_equal(host_bits(run_fp8(handle, X8, A8, B8, t, act, sc, p, q, sched)), base), (sched, p, q)


def test_fp8_validation(handle):
    import torch
    z = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    Y = torch.empty((64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dm.DominoError) as e:  # F_i = 24 is not a multiple of 16
        dm.domino_mlp_fwd_fp8(handle, dm.make_cfg(64, 64, 48, 2), z, z, z, (1, 1, 1, 1), Y, None, 0)
    assert e.value.status == 3
    with pytest.raises(dm.DominoError) as e:
        dm.domino_mlp_fwd_fp8(handle, dm.make_cfg(64, 64, 64, 2), z, z, z, (1, 1, 0, 1), Y, None, 0)
    assert e.value.status == 1


@pytest.mark.slow
@pytest.mark.parametrize("workload", ["llama2_7b_swiglu", "gpt3_2.7b_mlp"])
def test_fp8_full_size_sampled(handle, workload):
    """The FP8 forward at the full size the bench times (its inputs and scales), fused schedule:
    rows at every row-chunk and tile edge plus a few at random against the oracle, and bit-identical
    to the two-stream schedule."""
    import torch

    import bench
    s = synth.SHAPES[workload]
    inp = bench.fp8_inputs(s)
    X8, A8, B8, sc = inp["X"], inp["A"], inp["B"], inp["scales"]
    Yf = run_fp8(handle, X8, A8, B8, s.t, s.act, sc, s.p, s.q, dm.SCHED_FUSED)
    Yi = run_fp8(handle, X8, A8, B8, s.t, s.act, sc, s.p, s.q, dm.SCHED_INTRA)
    assert np.array_equal(host_bits(Yf), host_bits(Yi))
    rows = edge_rows(s.M, s.M // s.p, 73, n_random=6)   # every chunk and tile edge, and 6 at random
    ref = oracle.mlp_fwd_fp8(X8, A8, B8, s.t, s.act, sc, rows=rows)
    assert_tol(host_f64(Yf[torch.from_numpy(rows).cuda()]), ref, "FP8 forward, sampled rows")
