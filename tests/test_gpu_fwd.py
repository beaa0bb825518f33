"""GPU parity of the forward pass (domino_mlp_fwd, domino_shard_sum) against the CPU oracle.

Integer-valued inputs make every intermediate exact, so those cases are compared bit for bit
(the expected value is the oracle's exact result rounded once to bf16).  Real-valued inputs
are held to max|Y - Y_ref| <= 1e-2 * max|Y_ref| + 1e-3.  Row-split results must be
bit-identical to the unsplit run.
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


def int_inputs(M, h, Fi, t, act, seed, p_zero=0.5):
    gated = act in synth.GATED
    a_rows = 2 * Fi * t if gated else Fi * t
    X = synth.ternary_bf16((M, h), seed, synth.TID_X, p_zero=p_zero)
    A = synth.ternary_bf16((a_rows, h), seed, synth.TID_A, p_zero=p_zero)
    B = synth.ternary_bf16((t, h, Fi), seed, synth.TID_B, p_zero=p_zero)
    return X, A, B


def real_inputs(M, h, Fi, t, act, seed):
    gated = act in synth.GATED
    a_rows = 2 * Fi * t if gated else Fi * t
    X = synth.normal_bf16((M, h), 0.0, 1.0, seed, synth.TID_X)
    A = synth.normal_bf16((a_rows, h), 0.0, 0.02, seed, synth.TID_A)
    B = synth.normal_bf16((t, h, Fi), 0.0, 0.02, seed, synth.TID_B)
    return X, A, B


# (M, h, F_i, t, p, q): several M/N/K tiles and ragged tails in each dimension
INT_SHAPES = [
    (384, 208, 136, 3, 2, 2),
    (128, 64, 64, 1, 1, 1),
    (520, 136, 264, 2, 1, 1),
    (264, 72, 40, 4, 3, 3),
]


@pytest.mark.parametrize("shape", INT_SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_NONE, synth.ACT_RELU, synth.ACT_BILINEAR])
def test_fwd_integer_bit_exact(lib, shape, act):
    M, h, Fi, t, p, q = shape
    pz = 0.85 if act == synth.ACT_BILINEAR else 0.5
    X, A, B = int_inputs(M, h, Fi, t, act, seed=17 + M + act, p_zero=pz)
    Yref, Href = oracle.mlp_fwd(X, A, B, t, act, return_h=True)
    assert np.max(np.abs(Href)) <= 256, "test precondition: H exact in bf16"
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, act)
    Y, S = lib.fwd(cfg, dev_bf16(X), dev_bf16(A), dev_bf16(B), save=True)
    assert np.array_equal(host_f64(Y), bf16_round(Yref))
    # the saved first-linear output, pushed through the activation, is the oracle's H
    s = host_f64(S)
    if act == synth.ACT_BILINEAR:
        g = np.concatenate([s[:, i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)], axis=1)
        u = np.concatenate([s[:, i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)], axis=1)
        assert np.array_equal(g * u, Href)
    else:
        assert np.array_equal(np.maximum(s, 0) if act == synth.ACT_RELU else s, Href)


REAL_SHAPES = [
    (256, 256, 512, 2, 2, 1),    # the 4 x 64-token, h=256 tiny GeLU workload
    (320, 256, 200, 2, 2, 2),
    (640, 384, 344, 3, 1, 2),
]


@pytest.mark.parametrize("shape", REAL_SHAPES)
@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_fwd_matches_oracle(lib, shape, act):
    M, h, Fi, t, p, q = shape
    X, A, B = real_inputs(M, h, Fi, t, act, seed=0)
    Yref = oracle.mlp_fwd(X, A, B, t, act)
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, act)
    Y, _ = lib.fwd(cfg, dev_bf16(X), dev_bf16(A), dev_bf16(B))
    assert_tol(host_f64(Y), Yref, f"Y act={act} shape={shape}")


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_row_and_column_splits_bit_identical(lib, act):
    M, h, Fi, t = 512, 256, 192, 4
    X, A, B = real_inputs(M, h, Fi, t, act, seed=3)
    dX, dA, dB = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    base, bsave = lib.fwd(dm.make_cfg(M, h, Fi * t, t, 1, 1, act), dX, dA, dB, save=True)
    base, bsave = host_bits(base), host_bits(bsave)
    for p, q in [(2, 1), (4, 1), (1, 2), (2, 2), (4, 4)]:
        Y, S = lib.fwd(dm.make_cfg(M, h, Fi * t, t, p, q, act), dX, dA, dB, save=True)
        assert np.array_equal(host_bits(Y), base), (p, q)
        assert np.array_equal(host_bits(S), bsave), (p, q)


def test_schedules_bit_identical(lib):
    M, h, Fi, t, act = 512, 256, 256, 2, synth.ACT_GELU
    X, A, B = real_inputs(M, h, Fi, t, act, seed=5)
    dX, dA, dB = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    outs = [host_bits(lib.fwd(dm.make_cfg(M, h, Fi * t, t, 2, 2, act, sched=s), dX, dA, dB)[0])
            for s in (dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_INTER)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_reduction_cta_budget_bit_identical(lib):
    """cfg.reduce_ctas caps the shard-sum grid (grid-stride loop): any budget gives the same Y."""
    M, h, Fi, t, act = 512, 256, 128, 4, synth.ACT_SWIGLU
    X, A, B = real_inputs(M, h, Fi, t, act, seed=8)
    dX, dA, dB = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    base = host_bits(lib.fwd(dm.make_cfg(M, h, Fi * t, t, 2, 2, act), dX, dA, dB)[0])
    for n in (1, 3, 16, 1000):
        Y = lib.fwd(dm.make_cfg(M, h, Fi * t, t, 2, 2, act, reduce_ctas=n), dX, dA, dB)[0]
        assert np.array_equal(host_bits(Y), base), n


def test_repeat_runs_bit_identical(lib):
    M, h, Fi, t, act = 384, 256, 128, 4, synth.ACT_SWIGLU
    X, A, B = real_inputs(M, h, Fi, t, act, seed=6)
    dX, dA, dB = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    cfg = dm.make_cfg(M, h, Fi * t, t, 2, 1, act)
    first = host_bits(lib.fwd(cfg, dX, dA, dB)[0])
    for _ in range(3):
        assert np.array_equal(host_bits(lib.fwd(cfg, dX, dA, dB)[0]), first)


def test_empty_input_is_a_no_op(lib):
    import torch
    cfg = dm.make_cfg(0, 64, 128, 2, 1, 1, synth.ACT_GELU)
    n0 = dm.domino_launch_count(lib.h)
    X = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    dm.domino_mlp_fwd(lib.h, cfg, X.data_ptr() or 256, A, B, Y.data_ptr() or 256, None, None, 0)
    assert dm.domino_launch_count(lib.h) == n0


def test_bad_arguments_launch_nothing(lib):
    import torch
    M, h, F, t = 128, 64, 128, 2
    cfg = dm.make_cfg(M, h, F, t, 1, 1, synth.ACT_GELU)
    X = torch.zeros((M, h), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((F, h), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((t, h, F // t), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    ws, n = lib.workspace(cfg, dm.PASS_FWD)
    n0 = dm.domino_launch_count(lib.h)
    with pytest.raises(dm.DominoError) as e:   # misaligned X
        dm.domino_mlp_fwd(lib.h, cfg, X.data_ptr() + 2, A, B, Y, None, ws, n)
    assert e.value.status == 3
    with pytest.raises(dm.DominoError) as e:   # workspace too small
        dm.domino_mlp_fwd(lib.h, cfg, X, A, B, Y, None, ws, n - 1)
    assert e.value.status == 4
    with pytest.raises(dm.DominoError) as e:   # NULL output
        dm.domino_mlp_fwd(lib.h, cfg, X, A, B, None, None, ws, n)
    assert e.value.status == 1
    assert dm.domino_launch_count(lib.h) == n0


@pytest.mark.parametrize("t", [1, 2, 3, 5, 8])
def test_shard_sum_matches_ordered_fp32_sum(lib, t):
    import torch
    rows, cols, ld = 333, 136, 200
    rng = np.random.default_rng(t)
    P = rng.standard_normal((t, rows, cols)).astype(np.float32)
    res = synth.normal_bf16((rows, ld), 0, 1, 4, 1)
    # expected: fp32 adds in shard order, residual added, one RNE rounding
    acc = P[0].copy()
    for i in range(1, t):
        acc = (acc + P[i]).astype(np.float32)
    with_res = (synth.bf16_bits_to_f32(res)[:, :cols] + acc).astype(np.float32)
    Pd = torch.from_numpy(P).cuda()
    Y = torch.zeros((rows, ld), dtype=torch.bfloat16, device="cuda")
    dm.domino_shard_sum(Pd, t, rows, cols, None, 0, Y, ld)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(Y)[:, :cols], synth.f32_to_bf16_bits(acc))
    assert np.all(host_bits(Y)[:, cols:] == 0)
    R = dev_bf16(res)
    dm.domino_shard_sum(Pd, t, rows, cols, R, ld, Y, ld)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(Y)[:, :cols], synth.f32_to_bf16_bits(with_res))


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_last_chunk_reduced_in_gemm_matches_serial(lib, act):
    """The overlapped schedules reduce a call's last chunk inside its GEMM (the fused kernel) and the
    other chunks with the shard-sum kernel; SERIAL uses the shard-sum kernel throughout.  On ragged
    shapes (F_i and M not multiples of the tile sizes) every split gives the same bits, including a
    single chunk (p = q = 1), which is reduced in its GEMM alone."""
    M, h, Fi, t = 384, 256, 136, 2
    X, A, B = real_inputs(M, h, Fi, t, act, seed=9)
    dX, dA, dB = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    for p, q in [(1, 1), (2, 1), (1, 2), (3, 2)]:
        serial = host_bits(lib.fwd(dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=dm.SCHED_SERIAL), dX, dA, dB)[0])
        for sched in (dm.SCHED_INTRA, dm.SCHED_INTER):
            got = host_bits(lib.fwd(dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=sched), dX, dA, dB)[0])
            assert np.array_equal(got, serial), (p, q, sched)
