"""Canary guards: no entry point writes outside its workspace or its output arrays.

Every workspace and output buffer is placed between two 64 KiB guard regions filled with a byte
pattern; after the call (ragged shapes: row chunks and feature shards not multiples of the 128-
or 256-wide tiles, every schedule) the guards must be intact.
"""
import numpy as np
import pytest

from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import dev_bf16

pytestmark = pytest.mark.gpu

GUARD = 65536
PATTERN = 0xA5


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


class Guarded:
    """A device array of `shape` / `dtype` between two guard regions (and, for workspaces, a raw
    byte region of `nbytes`)."""

    def __init__(self, shape=None, dtype=None, nbytes=None, zero=False):
        import torch
        if nbytes is None:
            nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + max(nbytes, 1) + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        inner = self.buf[GUARD:GUARD + nbytes]
        if zero:
            inner.zero_()
        self.t = inner.view(dtype).view(shape) if shape is not None else inner

    def intact(self):
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool((head == PATTERN).all().item()) and bool((tail == PATTERN).all().item())


def check_all(**bufs):
    import torch
    torch.cuda.synchronize()
    bad = [k for k, b in bufs.items() if not b.intact()]
    assert not bad, f"guard bytes overwritten next to: {bad}"


def ws_for(cfg, pass_):
    return Guarded(nbytes=dm.domino_workspace_size(cfg, pass_))


@pytest.mark.parametrize("sched", [dm.SCHED_INTRA, dm.SCHED_FUSED])
@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_mlp_fwd_bwd_stay_inside(handle, sched, act):
    import torch
    M, h, Fi, t, p, q = 384, 256, 136, 2, 2, 2
    s = synth.MlpShape("c", M, h, Fi * t, act, t, p, q, backward=True)
    d = synth.make_inputs(s, seed=41)
    X, A, B, gY = dev_bf16(d["X"]), dev_bf16(d["A"][0]), dev_bf16(d["B"][0]), dev_bf16(d["gY"])
    cfg = dm.make_cfg(M, h, s.F, t, p, q, act, sched=sched)
    wf, wb = ws_for(cfg, dm.PASS_FWD), ws_for(cfg, dm.PASS_BWD)
    Y = Guarded((M, h), torch.bfloat16)
    S = Guarded((M, s.a_rows), torch.bfloat16)
    gX = Guarded((M, h), torch.bfloat16)
    gA = Guarded((s.a_rows, h), torch.float32, zero=True)
    gB = Guarded((t, h, Fi), torch.float32, zero=True)
    dm.domino_mlp_fwd(handle, cfg, X, A, B, Y.t, S.t, wf.t, wf.nbytes)
    dm.domino_mlp_bwd(handle, cfg, X, A, B, S.t, gY, gX.t, gA.t, gB.t, wb.t, wb.nbytes)
    check_all(ws_fwd=wf, ws_bwd=wb, Y=Y, act_save=S, gX=gX, gA=gA, gB=gB)


@pytest.mark.parametrize("sched", [dm.SCHED_INTER, dm.SCHED_FUSED])
def test_stack_train_stays_inside(handle, sched):
    import torch
    L, M, h, F, t, p, q = 2, 384, 256, 272, 2, 2, 2
    s = synth.MlpShape("c2", M, h, F, synth.ACT_GELU, t, p, q, layers=L, layernorm=True, backward=True)
    d = synth.make_inputs(s, seed=42)
    Z, A, B, gZ = dev_bf16(d["X"]), dev_bf16(d["A"]), dev_bf16(d["B"]), dev_bf16(d["gY"])
    cfg = dm.make_cfg(M, h, F, t, p, q, synth.ACT_GELU, sched=sched, layers=L, ln_eps=1e-5)
    wf, wb = ws_for(cfg, dm.PASS_STACK), ws_for(cfg, dm.PASS_STACK_BWD)
    save = Guarded(nbytes=dm.domino_stack_save_size(cfg))
    out = Guarded((M, h), torch.bfloat16)
    gZin = Guarded((M, h), torch.bfloat16)
    gA = Guarded((L, F, h), torch.float32, zero=True)
    gB = Guarded((L, t, h, F // t), torch.float32, zero=True)
    dm.domino_stack_fwd_train(handle, cfg, Z, A, B, out.t, save.t, wf.t, save_bytes=save.nbytes,
                              workspace_bytes=wf.nbytes)
    dm.domino_stack_bwd(handle, cfg, A, B, save.t, gZ, gZin.t, gA.t, gB.t, wb.t, save_bytes=save.nbytes,
                        workspace_bytes=wb.nbytes)
    check_all(ws_fwd=wf, ws_bwd=wb, save=save, out=out, gZ_in=gZin, gA=gA, gB=gB)


@pytest.mark.parametrize("sched", [dm.SCHED_INTER, dm.SCHED_FUSED])
def test_block_and_attention_stay_inside(handle, sched):
    import torch
    L, nseq, seq, h, heads, F, t, p, q = 1, 2, 200, 256, 2, 512, 2, 2, 2
    s = synth.MlpShape("c3", nseq * seq, h, F, synth.ACT_GELU, t, p, q, layers=L, layernorm=True, seq=seq,
                       heads=heads, w_std=0.0625)
    d = synth.make_inputs(s, seed=43)
    Z, Wq, Wo, A, B = (dev_bf16(d[k]) for k in ("X", "Wqkv", "Wo", "A", "B"))
    cfg = dm.make_cfg(s.M, h, F, t, p, q, synth.ACT_GELU, sched=sched, layers=L, heads=heads, seq=seq)
    wblk = ws_for(cfg, dm.PASS_BLOCK)
    out = Guarded((s.M, h), torch.bfloat16)
    dm.domino_block_fwd(handle, cfg, Z, Wq, Wo, A, B, out.t, wblk.t, wblk.nbytes)
    acfg = dm.make_cfg(s.M, h, 0, t, p, q, sched=sched, heads=heads, seq=seq, attn_ctas=3)
    wat = ws_for(acfg, dm.PASS_ATTN)
    Y = Guarded((s.M, h), torch.bfloat16)
    dm.domino_attn_fwd(handle, acfg, Z, Wq[0], Wo[0], Y.t, wat.t, wat.nbytes)
    check_all(ws_block=wblk, out=out, ws_attn=wat, Y=Y)


def test_fp8_forward_stays_inside(handle):
    import torch
    M, h, Fi, t, p, q = 384, 256, 144, 2, 2, 2
    sc = (2.0 ** -6, 2.0 ** -11, 2.0 ** -11, 2.0 ** -7)
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    X8 = u8(synth.e4m3_codes((M, h), 1.0, sc[0], 44, synth.TID_X))
    A8 = u8(synth.e4m3_codes((2 * Fi * t, h), 0.02, sc[1], 44, synth.TID_A))
    B8 = u8(synth.e4m3_codes((t, h, Fi), 0.02, sc[2], 44, synth.TID_B))
    for sched in (dm.SCHED_INTRA, dm.SCHED_FUSED):
        cfg = dm.make_cfg(M, h, Fi * t, t, p, q, synth.ACT_SWIGLU, sched=sched)
        w = ws_for(cfg, dm.PASS_FWD_FP8)
        Y = Guarded((M, h), torch.bfloat16)
        dm.domino_mlp_fwd_fp8(handle, cfg, X8, A8, B8, sc, Y.t, w.t, w.nbytes)
        check_all(ws=w, Y=Y)
