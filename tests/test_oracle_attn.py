"""Pins of the attention and transformer-block oracle (oracle_attn.c) against what does not come
from the oracle itself: PyTorch's float64 scaled_dot_product_attention and layer_norm (library
routines), closed forms (the first position attends only to itself; all-zero queries give the
running mean of the values), the head-shard decomposition, and structural invariants (row and
prefix subsets, independence of sequences).  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from comm_overlap_gb300 import synth


def f64(a):
    return synth.bf16_bits_to_f32(a).astype(np.float64)


def attn_inputs(nseq, seq, h, heads, seed, wstd=0.25):
    M = nseq * seq
    X = synth.normal_bf16((M, h), 0.0, 1.0, seed, synth.TID_X)
    Wqkv = synth.normal_bf16((3 * h, h), 0.0, wstd, seed, synth.TID_WQKV)
    return X, Wqkv


def wo_shards(h, t, seed, layer=0, std=0.25):
    return synth.normal_bf16((t, h, h // t), 0.0, std, seed, synth.TID_WO, layer)


def torch_attn(x, Wqkv, Wo, t, heads, seq):
    """Reference in float64: project, causal SDPA per sequence and head, output projection."""
    M, h = x.shape
    d, nhi = h // heads, heads // t
    W = torch.from_numpy(f64(Wqkv)).reshape(t, 3, nhi, d, h)
    Wq, Wk, Wv = (W[:, j].reshape(heads, d, h) for j in range(3))
    xt = torch.as_tensor(x, dtype=torch.float64)

    def proj(Wm):  # heads x nseq x seq x d
        return torch.einsum("mk,hek->hme", xt, Wm).reshape(heads, M // seq, seq, d)

    o = torch.nn.functional.scaled_dot_product_attention(proj(Wq), proj(Wk), proj(Wv), is_causal=True)
    o = o.reshape(heads, M, d).permute(1, 0, 2).reshape(M, heads * d)
    Wo_full = torch.cat(list(torch.from_numpy(f64(Wo))), dim=1)  # h x (t * h/t)
    return (o @ Wo_full.T).numpy()


SHAPES = [  # (nseq, seq, h, heads, t)
    (2, 5, 16, 4, 2),
    (3, 7, 24, 6, 3),
    (2, 9, 16, 2, 1),
    (4, 1, 8, 2, 2),
    (1, 12, 32, 8, 4),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_attn_matches_torch_sdpa(shape):
    nseq, seq, h, heads, t = shape
    X, Wqkv = attn_inputs(nseq, seq, h, heads, 1)
    Wo = wo_shards(h, t, 1)
    got = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq)
    ref = torch_attn(f64(X), Wqkv, Wo, t, heads, seq)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("shape", SHAPES)
def test_attn_sharded_equals_plain(shape):
    nseq, seq, h, heads, t = shape
    X, Wqkv = attn_inputs(nseq, seq, h, heads, 2)
    Wo = wo_shards(h, t, 2)
    a = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq)
    b = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq, sharded=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def value_rows(x, Wqkv, t, heads):
    """v_p for every position (M x heads*d, global head order) from the storage layout."""
    M, h = x.shape
    d, nhi = h // heads, heads // t
    W = f64(Wqkv).reshape(t, 3, nhi, d, h)
    Wv = W[:, 2].reshape(heads * d, h)
    return x @ Wv.T


def wo_full(Wo):
    return np.concatenate(list(f64(Wo)), axis=1)


def test_attn_first_position_is_value_projection():
    nseq, seq, h, heads, t = 3, 6, 16, 4, 2
    X, Wqkv = attn_inputs(nseq, seq, h, heads, 3)
    Wo = wo_shards(h, t, 3)
    Y = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq)
    V = value_rows(f64(X), Wqkv, t, heads)
    for s in range(nseq):
        r = s * seq
        np.testing.assert_allclose(Y[r], V[r] @ wo_full(Wo).T, rtol=1e-12, atol=1e-12)


def test_attn_zero_queries_average_the_causal_prefix():
    """With all query weights zero every score is 0: each position averages the values of
    positions 0..pos of its own sequence (pins the causal mask and the sequence boundaries)."""
    nseq, seq, h, heads, t = 2, 7, 16, 4, 2
    X, Wqkv = attn_inputs(nseq, seq, h, heads, 4)
    Wqkv = Wqkv.copy()
    Wqkv.reshape(t, 3, h // t, h)[:, 0] = 0  # query rows of every shard
    Wo = wo_shards(h, t, 4)
    Y = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq)
    V = value_rows(f64(X), Wqkv, t, heads)
    for s in range(nseq):
        for p in range(seq):
            o = V[s * seq:s * seq + p + 1].mean(axis=0)
            np.testing.assert_allclose(Y[s * seq + p], o @ wo_full(Wo).T, rtol=1e-12, atol=1e-12)


def test_attn_row_subset_and_sequence_independence():
    nseq, seq, h, heads, t = 3, 5, 16, 4, 2
    X, Wqkv = attn_inputs(nseq, seq, h, heads, 5)
    Wo = wo_shards(h, t, 5)
    full = oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq)
    rows = np.array([14, 0, 7, 4, 10])
    np.testing.assert_allclose(oracle.attn_fwd(X, Wqkv, Wo, t, heads, seq, rows=rows), full[rows], rtol=1e-12,
                               atol=1e-12)
    # swapping two sequences swaps their outputs and leaves the third alone
    Xs = X.copy()
    Xs[0:seq], Xs[2 * seq:3 * seq] = X[2 * seq:3 * seq], X[0:seq]
    sw = oracle.attn_fwd(Xs, Wqkv, Wo, t, heads, seq)
    np.testing.assert_allclose(sw[0:seq], full[2 * seq:3 * seq], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sw[seq:2 * seq], full[seq:2 * seq], rtol=1e-12, atol=1e-12)


def test_attn_rejects_bad_shapes():
    X, Wqkv = attn_inputs(2, 4, 16, 4, 6)
    Wo = wo_shards(16, 2, 6)
    with pytest.raises(ValueError):
        oracle.attn_fwd(X, Wqkv, Wo, 2, 4, 3)   # M % seq
    with pytest.raises(ValueError):
        oracle.attn_fwd(X, Wqkv, Wo, 3, 4, 4)   # heads % t


# ---- the block stack ---------------------------------------------------------------------------

def block_weights(L, h, F, heads, t, act, seed):
    gated = act in synth.GATED
    a_rows = 2 * F if gated else F
    Wqkv = np.stack([synth.normal_bf16((3 * h, h), 0.0, 0.2, seed, synth.TID_WQKV, l) for l in range(L)])
    Wo = np.stack([wo_shards(h, t, seed, l, 0.2) for l in range(L)])
    A = np.stack([synth.normal_bf16((a_rows, h), 0.0, 0.2, seed, synth.TID_A, l) for l in range(L)])
    B = np.stack([synth.normal_bf16((t, h, F // t), 0.0, 0.2, seed, synth.TID_B, l) for l in range(L)])
    return Wqkv, Wo, A, B


def torch_block(Z, Wqkv, Wo, A, B, t, heads, seq, act, eps):
    z = f64(Z)
    L = Wqkv.shape[0]
    M, h = z.shape
    F = B.shape[1] * B.shape[3]
    Fi = F // t
    for l in range(L):
        ln = torch.nn.functional.layer_norm(torch.from_numpy(z), (h,), eps=eps).numpy()
        z = z + torch_attn(ln, Wqkv[l], Wo[l], t, heads, seq)
        ln = torch.nn.functional.layer_norm(torch.from_numpy(z), (h,), eps=eps)
        Af = torch.from_numpy(f64(A[l]))
        if act in synth.GATED:
            gate = torch.cat([Af[i * 2 * Fi:i * 2 * Fi + Fi] for i in range(t)])
            up = torch.cat([Af[i * 2 * Fi + Fi:(i + 1) * 2 * Fi] for i in range(t)])
            g, u = ln @ gate.T, ln @ up.T
            H = torch.nn.functional.silu(g) * u if act == synth.ACT_SWIGLU else g * u
        else:
            H = ln @ Af.T
            H = torch.nn.functional.gelu(H) if act == synth.ACT_GELU else torch.relu(H)
        Bf = torch.cat(list(torch.from_numpy(f64(B[l]))), dim=1)
        z = z + (H @ Bf.T).numpy()
    return z


@pytest.mark.parametrize("act", [synth.ACT_GELU, synth.ACT_SWIGLU])
def test_block_matches_torch_composition(act):
    nseq, seq, h, heads, t, F, L = 2, 6, 16, 4, 2, 32, 2
    Z = synth.normal_bf16((nseq * seq, h), 0.0, 1.0, 7, synth.TID_X)
    Wqkv, Wo, A, B = block_weights(L, h, F, heads, t, act, 7)
    got = oracle.block_fwd(Z, Wqkv, Wo, A, B, t, heads, seq, act, 1e-5)
    ref = torch_block(Z, Wqkv, Wo, A, B, t, heads, seq, act, 1e-5).reshape(nseq, seq, h)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


def test_block_zero_layers_prefix_and_sequence_subset():
    nseq, seq, h, heads, t, F, L, act = 3, 8, 16, 4, 2, 32, 2, synth.ACT_GELU
    Z = synth.normal_bf16((nseq * seq, h), 0.0, 1.0, 8, synth.TID_X)
    Wqkv, Wo, A, B = block_weights(L, h, F, heads, t, act, 8)
    ident = oracle.block_fwd(Z, Wqkv[:0], Wo[:0], A[:0], B[:0], t, heads, seq, act)
    np.testing.assert_array_equal(ident.reshape(-1, h), f64(Z))
    full = oracle.block_fwd(Z, Wqkv, Wo, A, B, t, heads, seq, act)
    part = oracle.block_fwd(Z, Wqkv, Wo, A, B, t, heads, seq, act, seqs=[2, 0], upto=5)
    np.testing.assert_allclose(part[0], full[2, :5], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part[1], full[0, :5], rtol=1e-12, atol=1e-12)
