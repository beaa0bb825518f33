"""CUDA Graph capture of the chunk pipeline.

The library forks its compute and reduction streams from the caller's stream with events and
joins them back, so a caller can capture a forward + backward (or a layer stack) into a CUDA
graph and replay it.  One eager call per entry point must precede the capture (it performs the
one-time kernel attribute set-up).  Replays must reproduce the eager results bit for bit.
"""
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
    st, site = L.status()
    L.close()
    assert st == 0, f"device error word set: site {site:#x}"


@pytest.mark.parametrize("sched", [dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_FUSED])
def test_fwd_bwd_graph_replay_bit_identical(lib, sched):
    import torch
    M, h, Fi, t, p, q, act = 512, 256, 192, 4, 2, 2, synth.ACT_SWIGLU
    s = synth.MlpShape("g", M, h, Fi * t, act, t, p, q, backward=True)
    d = synth.make_inputs(s, seed=21)
    X, A, B, gY = dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0]), dev_bf16(d["gY"])
    cfg = dm.make_cfg(M, h, s.F, t, p, q, act, sched=sched)
    n = max(dm.domino_workspace_size(cfg, dm.PASS_FWD), dm.domino_workspace_size(cfg, dm.PASS_BWD))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    S = torch.empty((M, s.a_rows), dtype=torch.bfloat16, device="cuda")
    gX = torch.empty_like(Y)
    gA = torch.zeros((s.a_rows, h), dtype=torch.float32, device="cuda")
    gB = torch.zeros((t, h, Fi), dtype=torch.float32, device="cuda")

    def step(stream):
        gA.zero_()
        gB.zero_()
        dm.domino_mlp_fwd(lib.h, cfg, X, A, B, Y, S, ws, n, stream)
        dm.domino_mlp_bwd(lib.h, cfg, X, A, B, S, gY, gX, gA, gB, ws, n, stream)

    step(torch.cuda.current_stream())  # eager: the reference and the one-time set-up
    torch.cuda.synchronize()
    ref = [host_bits(Y), host_bits(gX), gA.cpu().numpy().copy(), gB.cpu().numpy().copy()]
    for o in (Y, gX):
        o.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step(side)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(Y), ref[0])
        assert np.array_equal(host_bits(gX), ref[1])
        assert np.array_equal(gA.cpu().numpy(), ref[2])
        assert np.array_equal(gB.cpu().numpy(), ref[3])


def test_stack_graph_replay_bit_identical(lib):
    import torch
    L, M, h, F, t, p, q = 2, 256, 128, 256, 2, 2, 2
    s = synth.MlpShape("s", M, h, F, synth.ACT_GELU, t, p, q, layers=L, layernorm=True)
    d = synth.make_inputs(s, seed=22)
    Z, A, B = dev_bf16(d["X"]), dev_bf16(d["A"]), dev_bf16(d["B"])
    cfg = dm.make_cfg(M, h, F, t, p, q, synth.ACT_GELU, sched=dm.SCHED_INTER, layers=L)
    n = dm.domino_workspace_size(cfg, dm.PASS_STACK)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(Z)
    dm.domino_stack_fwd(lib.h, cfg, Z, A, B, out, ws, n)
    torch.cuda.synchronize()
    ref = host_bits(out)
    out.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dm.domino_stack_fwd(lib.h, cfg, Z, A, B, out, ws, n, side)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), ref)


def replay_matches(fn, out):
    """Eager call, then capture + replay on a side stream; the replayed output must match bit for bit."""
    import torch
    fn(torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = host_bits(out) if out.dtype == torch.bfloat16 else out.cpu().numpy().copy()
    out.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn(side)
    g.replay()
    torch.cuda.synchronize()
    got = host_bits(out) if out.dtype == torch.bfloat16 else out.cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("sched", [dm.SCHED_INTER, dm.SCHED_FUSED])
def test_block_graph_replay_bit_identical(lib, sched):
    """The Transformer block stack (attention kernel included) under capture."""
    import torch
    L, nseq, seq, h, heads, F, t, p, q = 2, 2, 128, 256, 2, 512, 2, 2, 2
    s = synth.MlpShape("b", nseq * seq, h, F, synth.ACT_GELU, t, p, q, layers=L, layernorm=True, seq=seq,
                       heads=heads, w_std=0.0625)
    d = synth.make_inputs(s, seed=23)
    Z, Wq, Wo, A, B = (dev_bf16(d[k]) for k in ("X", "Wqkv", "Wo", "A", "B"))
    cfg = dm.make_cfg(s.M, h, F, t, p, q, synth.ACT_GELU, sched=sched, layers=L, heads=heads, seq=seq)
    n = dm.domino_workspace_size(cfg, dm.PASS_BLOCK)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(Z)
    replay_matches(lambda st: dm.domino_block_fwd(lib.h, cfg, Z, Wq, Wo, A, B, out, ws, n, st), out)


def test_fp8_graph_replay_bit_identical(lib):
    import torch
    M, h, Fi, t, p, q = 512, 256, 128, 4, 2, 1
    sc = (2.0 ** -6, 2.0 ** -11, 2.0 ** -11, 2.0 ** -7)
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    X8 = u8(synth.e4m3_codes((M, h), 1.0, sc[0], 24, synth.TID_X))
    A8 = u8(synth.e4m3_codes((2 * Fi * t, h), 0.02, sc[1], 24, synth.TID_A))
    B8 = u8(synth.e4m3_codes((t, h, Fi), 0.02, sc[2], 24, synth.TID_B))
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, synth.ACT_SWIGLU, sched=dm.SCHED_INTRA)
    n = dm.domino_workspace_size(cfg, dm.PASS_FWD_FP8)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    replay_matches(lambda st: dm.domino_mlp_fwd_fp8(lib.h, cfg, X8, A8, B8, sc, Y, ws, n, st), Y)
