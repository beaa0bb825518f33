"""The measurement hooks behind the exposed-reduction figure: domino_debug_skip_reduce (the same
schedule with no reduction) and domino_timing_trace (the launch timeline)."""
import numpy as np
import pytest

from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import Lib, dev_bf16, host_bits

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
    dm.domino_debug_skip_reduce(L.h, False)
    st, site = L.status()
    L.close()
    assert st == 0, f"device error word set: site {site:#x}"


def mlp_inputs(M, h, F, t, act, seed=3):
    a_rows = 2 * F if act in synth.GATED else F
    X = dev_bf16(synth.normal_bf16((M, h), 0, 1, seed, synth.TID_X))
    A = dev_bf16(synth.normal_bf16((a_rows, h), 0, 0.02, seed, synth.TID_A))
    B = dev_bf16(synth.normal_bf16((t, h, F // t), 0, 0.02, seed, synth.TID_B))
    return X, A, B


@pytest.mark.parametrize("sched", [dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_INTER])
def test_skip_reduce_leaves_outputs_and_restores(lib, sched):
    import torch
    M, h, F, t = 1024, 512, 1536, 4
    cfg = dm.make_cfg(M, h, F, t, 2, 2, synth.ACT_SWIGLU, sched=sched)
    X, A, B = mlp_inputs(M, h, F, t, synth.ACT_SWIGLU)
    ref, _ = lib.fwd(cfg, X, A, B)
    ws, n = lib.workspace(cfg, dm.PASS_FWD)
    # with the hook on, no shard-sum writes Y: a sentinel pattern survives the forward
    Y = torch.full((M, h), 3.0, dtype=torch.bfloat16, device="cuda")
    n0 = dm.domino_launch_count(lib.h)
    dm.domino_debug_skip_reduce(lib.h, True)
    try:
        dm.domino_mlp_fwd(lib.h, cfg, X, A, B, Y, None, ws, n)
        torch.cuda.synchronize()
    finally:
        dm.domino_debug_skip_reduce(lib.h, False)
    assert bool((Y == 3.0).all()), "a reduction ran with the hook on"
    # every column chunk of every row chunk launched its (empty) stand-in after its GEMMs:
    # 2 first linears + 4 second linears + 4 stand-ins
    assert dm.domino_launch_count(lib.h) - n0 == 2 + 4 + 4
    # hook off: the normal path again, bit for bit
    Y2, _ = lib.fwd(cfg, X, A, B)
    assert np.array_equal(host_bits(Y2), host_bits(ref))


def test_skip_reduce_copies_the_residual_in_stacks(lib):
    import torch
    M, h, F, t, L = 512, 256, 1024, 2, 3
    cfg = dm.make_cfg(M, h, F, t, 2, 2, synth.ACT_GELU, sched=dm.SCHED_INTER, layers=L)
    Z = dev_bf16(synth.normal_bf16((M, h), 0, 1, 4, synth.TID_X))
    A = dev_bf16(np.concatenate([synth.normal_bf16((F, h), 0, 0.02, 4, synth.TID_A, l) for l in range(L)]))
    B = dev_bf16(np.concatenate([synth.normal_bf16((t, h, F // t), 0, 0.02, 4, synth.TID_B, l) for l in range(L)]))
    dm.domino_debug_skip_reduce(lib.h, True)
    try:
        out = lib.stack(cfg, Z, A, B)
    finally:
        dm.domino_debug_skip_reduce(lib.h, False)
    # each layer's output is its residual: the stack passes its input through
    assert torch.equal(out.view(torch.int16), Z.view(torch.int16))


def test_skip_reduce_refuses_the_fused_schedule(lib):
    import torch
    M, h, F, t = 512, 256, 1024, 2
    cfg = dm.make_cfg(M, h, F, t, 2, 1, synth.ACT_GELU, sched=dm.SCHED_FUSED)
    X, A, B = mlp_inputs(M, h, F, t, synth.ACT_GELU)
    ws, n = lib.workspace(cfg, dm.PASS_FWD)
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    n0 = dm.domino_launch_count(lib.h)
    dm.domino_debug_skip_reduce(lib.h, True)
    try:
        with pytest.raises(dm.DominoError) as e:
            dm.domino_mlp_fwd(lib.h, cfg, X, A, B, Y, None, ws, n)
    finally:
        dm.domino_debug_skip_reduce(lib.h, False)
    assert e.value.status == 2
    assert dm.domino_launch_count(lib.h) == n0


def test_timing_trace_lists_every_launch(lib):
    import torch
    M, h, F, t = 1024, 512, 1536, 4
    cfg = dm.make_cfg(M, h, F, t, 2, 1, synth.ACT_GELU, sched=dm.SCHED_INTRA)
    X, A, B = mlp_inputs(M, h, F, t, synth.ACT_GELU)
    ws, n = lib.workspace(cfg, dm.PASS_FWD)
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    dm.domino_timing_reset(lib.h)
    dm.domino_timing_enable(lib.h, True)
    n0 = dm.domino_launch_count(lib.h)
    dm.domino_mlp_fwd(lib.h, cfg, X, A, B, Y, None, ws, n)
    torch.cuda.synchronize()
    dm.domino_timing_enable(lib.h, False)
    tr = dm.domino_timing_trace(lib.h)
    assert len(tr) == dm.domino_launch_count(lib.h) - n0
    # row chunk 0: first linear, second linear, shard-sum; row chunk 1 (the last): first linear,
    # second linear with the reduction fused
    assert [k for k, _, _ in tr] == [dm.K_GEMM_FWD1, dm.K_GEMM_FWD2, dm.K_SHARD_SUM, dm.K_GEMM_FWD1, dm.K_GEMM_FWD2]
    assert tr[0][1] == 0.0
    for k, a, b in tr:
        assert 0.0 <= a <= b
    # the shard-sum of chunk 0 starts after the GEMM that wrote its partials ended
    assert tr[2][1] >= tr[1][2]
    dm.domino_timing_reset(lib.h)
