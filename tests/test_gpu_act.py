"""The epilogues' activation functions (domino_act_eval) against the oracle's double-precision
definitions.  GeLU's Phi is computed from erf by Abramowitz & Stegun 7.1.26 (|error| <= 1.5e-7)
with the hardware exponential; SiLU from the hardware exponential and approximate division."""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def grid():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from comm_overlap_gb300 import build
    build.build()
    rng = np.random.default_rng(5)
    x = np.concatenate([np.linspace(-12, 12, 24001), rng.standard_normal(4000) * 3]).astype(np.float32)
    return x


def evaluate(act, a, b=None):
    import torch
    ta = torch.from_numpy(a).cuda()
    tb = torch.from_numpy(b).cuda() if b is not None else None
    out, da, db = (torch.empty_like(ta) for _ in range(3))
    dm.domino_act_eval(act, ta, tb, out, da, db, ta.numel())
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), da.cpu().numpy().astype(np.float64), db.cpu().numpy()


@pytest.mark.parametrize("act", [dm.ACT_GELU, dm.ACT_RELU, dm.ACT_NONE])
def test_plain_activations_match_double(grid, act):
    x = grid[np.abs(grid) > 1e-3] if act == dm.ACT_RELU else grid  # the relu kink is a convention
    out, da, consistency = evaluate(act, x)
    xd = x.astype(np.float64)
    ref = oracle.act(act, xd)
    dref = oracle.act_grad(act, xd)
    scale = np.maximum(1.0, np.abs(xd))
    assert np.max(np.abs(out - ref) / scale) < 4e-7
    assert np.max(np.abs(da - dref)) < 5e-7
    assert np.all(consistency == 0.0)


@pytest.mark.parametrize("act", [dm.ACT_SWIGLU, dm.ACT_BILINEAR])
def test_gated_activations_match_double(grid, act):
    rng = np.random.default_rng(6)
    g = grid
    u = (rng.standard_normal(g.size) * 2).astype(np.float32)
    out, dg, du = evaluate(act, g, u)
    gd, ud = g.astype(np.float64), u.astype(np.float64)
    ref = np.array([oracle.glu(act, a, b) for a, b in zip(gd, ud)])
    rdg = np.array([oracle.glu_dg(act, a, b) for a, b in zip(gd, ud)])
    rdu = np.array([oracle.glu_du(act, a, b) for a, b in zip(gd, ud)])
    tol = 2e-6 if act == dm.ACT_SWIGLU else 1e-7
    assert np.max(np.abs(out - ref) / np.maximum(1.0, np.abs(ref))) < tol
    assert np.max(np.abs(dg - rdg) / np.maximum(1.0, np.abs(rdg))) < tol
    assert np.max(np.abs(du.astype(np.float64) - rdu) / np.maximum(1.0, np.abs(rdu))) < tol
