"""domino_mlp_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns the whole memory pool, a serving loop that
forbids allocations after warm-up) cannot hand the library a workspace, so this entry point takes
its scratch from a fixed 64 MiB array built into the library.  The test checks, through the C ABI,
that two calls in a row give bit for bit the result of domino_mlp_fwd with a caller workspace
(both run the same kernels in the same order) under every schedule, the second call running on
the scratch the first left dirty; that the output also meets the oracle's tolerance; and that a
problem too large for the array, or a bad handle, is refused without launching anything.  It lives
in its own file, collected last, and sets everything up itself so it also passes alone in a fresh
process.
"""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import Lib, assert_tol, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu

SCHEDS = {"serial": dm.SCHED_SERIAL, "intra": dm.SCHED_INTRA, "inter": dm.SCHED_INTER, "fused": dm.SCHED_FUSED}


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


def inputs(M, h, Fi, t, act, seed):
    a_rows = (2 if act in synth.GATED else 1) * Fi * t
    X = synth.normal_bf16((M, h), 0, 1, seed, synth.TID_X)
    A = synth.normal_bf16((a_rows, h), 0, 0.02, seed, synth.TID_A)
    B = synth.normal_bf16((t, h, Fi), 0, 0.02, seed, synth.TID_B)
    return (X, A, B), (dev_bf16(X), dev_bf16(A), dev_bf16(B)), a_rows


@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_noalloc_bit_identical_to_workspace_forward_twice(lib, act, sched):
    import torch
    # 2 x 2 chunks of 512 x 256 over ragged tiles (F_i = 384 is 1.5 tiles of 256)
    M, h, Fi, t, p, q = 1024, 512, 384, 4, 2, 2
    cfg = dm.make_cfg(M, h, Fi * t, t, p, q, act, sched=SCHEDS[sched])
    assert dm.domino_workspace_size(cfg, dm.PASS_FWD) <= 64 << 20
    for seed in (11, 12):   # two calls in a row; the second runs on a scratch the first left dirty
        host, (X, A, B), a_rows = inputs(M, h, Fi, t, act, seed)
        ref, ref_save = lib.fwd(cfg, X, A, B, save=True)
        Y = torch.full((M, h), float("nan"), dtype=torch.bfloat16, device="cuda")
        S = torch.empty((M, a_rows), dtype=torch.bfloat16, device="cuda")
        dm.domino_mlp_fwd_noalloc(lib.h, cfg, X, A, B, Y, S)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(Y), host_bits(ref)), f"noalloc Y differs from the workspace forward, seed {seed}"
        assert np.array_equal(host_bits(S), host_bits(ref_save)), f"noalloc act_save differs, seed {seed}"
        if sched == "intra":
            # rows at both ends of each row chunk and of a 256-row tile, plus a few in between
            rows = np.unique(np.concatenate([[0, 255, 256, 511, 512, 767, 768, 1023],
                                             synth.sample_indices(M, 8, seed)]))
            Yref = oracle.mlp_fwd(host[0], host[1], host[2], t, act, rows=rows)
            assert_tol(host_f64(Y)[rows], Yref, f"noalloc Y against the oracle, seed {seed}")


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    import torch
    cfg = dm.make_cfg(32768, 4096, 14336, 8, 2, 1, synth.ACT_SWIGLU)
    assert dm.domino_workspace_size(cfg, dm.PASS_FWD) > 64 << 20
    n0 = dm.domino_launch_count(lib.h)
    X = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dm.DominoError) as e:
        dm.domino_mlp_fwd_noalloc(lib.h, cfg, X, X, X, X, None)
    assert e.value.status == 4
    assert "64" in dm.domino_last_error() or "bytes" in dm.domino_last_error()
    assert dm.domino_launch_count(lib.h) == n0


def test_noalloc_refuses_a_null_handle(lib):
    import torch
    cfg = dm.make_cfg(256, 256, 1024, 2, 2, 1, synth.ACT_GELU)
    X = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dm.DominoError) as e:
        dm.domino_mlp_fwd_noalloc(None, cfg, X, X, X, X, None)
    assert e.value.status == 1
