"""Failure paths on the GPU, exercised without faulting, trapping or hanging the device.

* A bounded device-side wait that can never complete (an mbarrier nothing arrives on) gives up
  after its time limit, records DOMINO_ERR_TIMEOUT in the error word and returns; the context
  stays usable and the next real call is correct.
* A launch failure injected on the host mid-schedule returns an error after joining the internal
  streams back into the caller's stream; later calls are correct.
"""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import Lib, assert_tol, dev_bf16, host_bits, host_f64

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
    L.close()


def small_problem(seed=30):
    M, h, Fi, t, act = 256, 128, 128, 2, synth.ACT_GELU
    s = synth.MlpShape("f", M, h, Fi * t, act, t, 2, 2)
    d = synth.make_inputs(s, seed=seed)
    return s, d, dm.make_cfg(M, h, s.F, t, 2, 2, act)


def test_bounded_wait_times_out_and_context_survives(lib):
    import torch
    assert lib.status() == (0, 0)
    dm.domino_selftest_wait_timeout(lib.h, 20000)  # 20 ms
    st, site = lib.status()
    assert st == 6 and site == dm.SELFTEST_SITE
    assert lib.status() == (0, 0), "reading the status clears it"
    s, d, cfg = small_problem()
    Y, _ = lib.fwd(cfg, dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0]))
    assert_tol(host_f64(Y), oracle.mlp_fwd(d["X"], d["A"][0], d["B"][0], s.t, s.act), "Y after timeout")
    with pytest.raises(dm.DominoError):
        dm.domino_selftest_wait_timeout(lib.h, 0)


@pytest.mark.parametrize("nth", [1, 3, 6])
def test_injected_launch_failure_returns_cleanly(lib, nth):
    import torch
    s, d, cfg = small_problem(31)
    X, A, B = dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0])
    ref, _ = lib.fwd(cfg, X, A, B)
    ref = host_bits(ref)
    Y = torch.zeros((s.M, s.h), dtype=torch.bfloat16, device="cuda")
    ws, n = lib.workspace(cfg, dm.PASS_FWD)
    n0 = dm.domino_launch_count(lib.h)
    dm.domino_debug_fail_launch(lib.h, nth)
    with pytest.raises(dm.DominoError) as e:
        dm.domino_mlp_fwd(lib.h, cfg, X, A, B, Y, None, ws, n)
    assert e.value.status == 5 and "injected" in str(e.value)
    assert dm.domino_launch_count(lib.h) == n0 + nth - 1
    # the caller's stream was joined: work enqueued after the failed call sees a consistent state
    torch.cuda.current_stream().synchronize()
    assert lib.status() == (0, 0)
    Y2, _ = lib.fwd(cfg, X, A, B)
    assert np.array_equal(host_bits(Y2), ref)
