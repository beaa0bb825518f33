"""GPU parity of the attention sublayer (domino_attn_fwd) and the Transformer block stack
(domino_block_fwd) against the CPU oracle (oracle_attn.c), in double.

Head dimension 128 (the kernel's); sequences shorter than, equal to and not a multiple of the
128-position block; several heads per shard; row chunks of whole sequences; column chunks of the
output projection; every schedule.  Row-split and schedule variants must be bit-identical.
"""
import numpy as np
import pytest

import oracle
from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth
from gpu_helpers import assert_tol, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu


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


def attn_inputs(nseq, seq, h, t, seed):
    M = nseq * seq
    X = synth.normal_bf16((M, h), 0.0, 1.0, seed, synth.TID_X)
    # query/key weights of std 1/sqrt(h) give scores of unit spread: a softmax far from uniform
    Wqkv = synth.normal_bf16((3 * h, h), 0.0, h ** -0.5, seed, synth.TID_WQKV)
    Wo = synth.normal_bf16((t, h, h // t), 0.0, h ** -0.5, seed, synth.TID_WO)
    return X, Wqkv, Wo


def run_attn(handle, X, Wqkv, Wo, h, heads, seq, t, p=1, q=1, sched=dm.SCHED_INTRA, attn_ctas=0):
    import torch
    M = X.shape[0]
    cfg = dm.make_cfg(M, h, 0, t, p, q, sched=sched, heads=heads, seq=seq, attn_ctas=attn_ctas)
    Y = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    n = dm.domino_workspace_size(cfg, dm.PASS_ATTN)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    dm.domino_attn_fwd(handle, cfg, dev_bf16(X), dev_bf16(Wqkv), dev_bf16(Wo), Y, ws, n)
    torch.cuda.synchronize()
    return Y


# (nseq, seq, h, heads, t, p, q)
SHAPES = [
    (2, 128, 256, 2, 2, 1, 1),    # one block per sequence
    (2, 200, 256, 2, 1, 2, 1),    # a partial second block; one sequence per row chunk
    (2, 320, 512, 4, 2, 2, 2),    # three blocks, two heads per shard, column chunks
    (5, 40, 256, 2, 2, 1, 1),     # sequences shorter than a block
    (1, 384, 384, 3, 3, 1, 3),    # three shards of one head, n = 128
]


@pytest.mark.parametrize("shape", SHAPES)
def test_attention_matches_oracle(handle, shape):
    nseq, seq, h, heads, t, p, q = shape
    X, Wqkv, Wo = attn_inputs(nseq, seq, h, t, 60)
    Y = run_attn(handle, X, Wqkv, Wo, h, heads, seq, t, p, q)
    ref = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq)
    assert_tol(host_f64(Y), ref, "attention sublayer output")


def test_attention_splits_and_schedules_bit_identical(handle):
    nseq, seq, h, heads, t = 4, 256, 512, 4, 2
    X, Wqkv, Wo = attn_inputs(nseq, seq, h, t, 61)
    base = host_bits(run_attn(handle, X, Wqkv, Wo, h, heads, seq, t, 1, 1))
    for sched in (dm.SCHED_SERIAL, dm.SCHED_INTRA, dm.SCHED_FUSED):
        for p, q in ((2, 1), (4, 2), (1, 4)):
            got = host_bits(run_attn(handle, X, Wqkv, Wo, h, heads, seq, t, p, q, sched))
            assert np.array_equal(got, base), (sched, p, q)


@pytest.mark.parametrize("nseq,seq", [(3, 1000), (2, 640), (4, 100)])
def test_attention_grid_budget_bit_identical(handle, nseq, seq):
    """The persistent kernel on a capped grid: a few CTAs walk all work units in turn (Q reloads,
    K/V rings and O hand-backs carried across items and units), bit-identical to one unit per CTA;
    the one-CTA run is also held to the oracle.  Units: pairs of query-block pairs (odd pair counts
    leave a one-item unit; a single block leaves one-tile items)."""
    h, heads, t = 512, 4, 2
    X, Wqkv, Wo = attn_inputs(nseq, seq, h, t, 64)
    base = host_bits(run_attn(handle, X, Wqkv, Wo, h, heads, seq, t))
    for ctas in (1, 2, 5, 23):
        Y = run_attn(handle, X, Wqkv, Wo, h, heads, seq, t, attn_ctas=ctas)
        assert np.array_equal(host_bits(Y), base), ctas
        if ctas == 1:
            assert_tol(host_f64(Y), oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq), "attention on one CTA")


def test_attention_validation(handle):
    import torch
    X = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((768, 256), dtype=torch.bfloat16, device="cuda")
    Wo = torch.zeros((2, 256, 128), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty_like(X)
    for kw, status in ((dict(heads=4, seq=128), 2),     # head dimension 64
                       (dict(heads=2, seq=96), 1),      # M % seq
                       (dict(heads=2, seq=0), 1),
                       (dict(heads=3, seq=128), 1)):    # h % heads
        cfg = dm.make_cfg(256, 256, 0, 2, 1, 1, **kw)
        with pytest.raises(dm.DominoError) as e:
            dm.domino_attn_fwd(handle, cfg, X, W, Wo, Y, None, 0)
        assert e.value.status == status, kw


def block_inputs(nseq, seq, h, F, t, act, L, seed):
    gated = act in synth.GATED
    a_rows = 2 * F if gated else F
    Z = synth.normal_bf16((nseq * seq, h), 0.0, 1.0, seed, synth.TID_X)
    Wqkv = np.stack([synth.normal_bf16((3 * h, h), 0.0, h ** -0.5, seed, synth.TID_WQKV, l) for l in range(L)])
    Wo = np.stack([synth.normal_bf16((t, h, h // t), 0.0, 0.02, seed, synth.TID_WO, l) for l in range(L)])
    A = np.stack([synth.normal_bf16((a_rows, h), 0.0, 0.02, seed, synth.TID_A, l) for l in range(L)])
    B = np.stack([synth.normal_bf16((t, h, F // t), 0.0, 0.02, seed, synth.TID_B, l) for l in range(L)])
    return Z, Wqkv, Wo, A, B


def run_block(handle, Z, Wqkv, Wo, A, B, h, F, heads, seq, t, act, p, q, sched):
    import torch
    L = Wqkv.shape[0]
    M = Z.shape[0]
    cfg = dm.make_cfg(M, h, F, t, p, q, act, sched=sched, layers=L, ln_eps=1e-5, heads=heads, seq=seq)
    out = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    n = dm.domino_workspace_size(cfg, dm.PASS_BLOCK)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    dm.domino_block_fwd(handle, cfg, dev_bf16(Z), dev_bf16(Wqkv), dev_bf16(Wo), dev_bf16(A), dev_bf16(B), out, ws, n)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_block_stack_matches_oracle(handle, act):
    nseq, seq, h, heads, t, F, L, p, q = 2, 192, 256, 2, 2, 512, 2, 2, 2
    Z, Wqkv, Wo, A, B = block_inputs(nseq, seq, h, F, t, act, L, 62)
    out = run_block(handle, Z, Wqkv, Wo, A, B, h, F, heads, seq, t, act, p, q, dm.SCHED_INTER)
    ref = oracle.block_fwd(Z, Wqkv, Wo, A, B, t, heads, seq, act, 1e-5)
    assert_tol(host_f64(out), ref.reshape(-1, h), "block stack output")


def test_block_schedules_bit_identical(handle):
    nseq, seq, h, heads, t, F, L, act = 4, 128, 256, 2, 2, 512, 2, synth.ACT_GELU
    Z, Wqkv, Wo, A, B = block_inputs(nseq, seq, h, F, t, act, L, 63)
    base = host_bits(run_block(handle, Z, Wqkv, Wo, A, B, h, F, heads, seq, t, act, 1, 1, dm.SCHED_SERIAL))
    for sched in (dm.SCHED_INTRA, dm.SCHED_INTER, dm.SCHED_FUSED):
        for p, q in ((2, 2), (4, 1)):
            got = host_bits(run_block(handle, Z, Wqkv, Wo, A, B, h, F, heads, seq, t, act, p, q, sched))
            assert np.array_equal(got, base), (sched, p, q)


@pytest.mark.slow
def test_block_full_size_sampled(handle):
    """The 4-layer GPT-3 6.7B-shaped block stack at full size: the first 160 positions (two query
    blocks) of two sequences, one in each row chunk, against the oracle."""
    import torch
    s = synth.SHAPES["gpt3_6.7b_block4"]
    d = synth.make_inputs(s, seed=0)
    out = run_block(handle, d["X"], d["Wqkv"], d["Wo"], d["A"], d["B"], s.h, s.F, s.heads, s.seq, s.t, s.act, s.p,
                    s.q, dm.SCHED_INTER)
    seqs = [1, s.M // s.seq - 1]
    upto = 160
    ref = oracle.block_fwd(d["X"], d["Wqkv"], d["Wo"], d["A"], d["B"], s.t, s.heads, s.seq, s.act, 1e-5,
                           seqs=seqs, upto=upto)
    rows = np.concatenate([np.arange(q * s.seq, q * s.seq + upto) for q in seqs])
    got = host_f64(out[torch.from_numpy(rows).cuda()])
    assert_tol(got, ref.reshape(-1, s.h), "block stack, sampled sequences")
