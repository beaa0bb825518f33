"""Seeded synthetic inputs for the chunked tensor-parallel MLP.

This module is the only code shared between the CPU oracle's tests and the GPU
path's tests and benchmark.  It draws numbers and lays them out in the storage
format the library expects; it performs none of the method's arithmetic (no
matmul, activation, normalisation or reduction).

Storage format (row-major, nn.Linear ``[out, in]`` orientation):

* ``X``  : ``M x h`` bf16, tokens batch-major, so a row chunk is a contiguous
  block of rows.
* ``A``  : ``t`` contiguous shards.  Non-gated activations: shard ``i`` is
  ``F_i x h``; gated (SwiGLU, bilinear): shard ``i`` is ``2F_i x h`` with the
  ``F_i`` gate rows first and the ``F_i`` up rows second.  ``F_i = F / t``.
* ``B``  : ``t`` contiguous shards, shard ``i`` is ``h x F_i``.
* ``gY`` : ``M x h`` bf16 (backward only).

All floating-point draws are float32 from numpy's Philox counter-based bit
generator, keyed by ``(seed, tensor id, layer)``, then rounded to bf16 with
round-to-nearest-even.  Integer-valued draws (for exactness tests) come from
the same generator.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# Activation codes.  They mirror ``domino_act`` in include/domino.h and the
# oracle's own constants; each side defines them independently.
ACT_NONE, ACT_RELU, ACT_GELU, ACT_SWIGLU, ACT_BILINEAR = 0, 1, 2, 3, 4
GATED = (ACT_SWIGLU, ACT_BILINEAR)

# tensor ids used to derive independent sub-streams
TID_X, TID_A, TID_B, TID_GY, TID_GA0, TID_GB0, TID_MISC = 1, 2, 3, 4, 5, 6, 7
TID_WQKV, TID_WO = 8, 9  # attention sublayer weights


def _rng(seed: int, tid: int, layer: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tid, layer])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


_CHUNK = 1 << 22


def _normal_block(n: int, mean: float, std: float, g: np.random.Generator) -> np.ndarray:
    x = g.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return f32_to_bf16_bits(x)


def normal_bf16(shape, mean: float, std: float, seed: int, tid: int, layer: int = 0) -> np.ndarray:
    """bf16 bits of N(mean, std) draws, shape ``shape``.

    Tensors larger than 4 Mi elements are drawn in 4 Mi-element blocks, block ``b`` from its own
    Philox stream keyed by (seed, tid, layer, b), on a thread pool; the values do not depend on
    the number of threads.
    """
    n = int(np.prod(shape))
    if n <= _CHUNK:
        return _normal_block(n, mean, std, _rng(seed, tid, layer)).reshape(shape)
    import concurrent.futures as cf
    import os
    out = np.empty(n, dtype=np.uint16)
    nblk = (n + _CHUNK - 1) // _CHUNK

    def work(b):
        lo, hi = b * _CHUNK, min(n, (b + 1) * _CHUNK)
        g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tid, layer, b])))
        out[lo:hi] = _normal_block(hi - lo, mean, std, g)

    with cf.ThreadPoolExecutor(max_workers=min(nblk, os.cpu_count() or 4)) as ex:
        list(ex.map(work, range(nblk)))
    return out.reshape(shape)


def ternary_bf16(shape, seed: int, tid: int, layer: int = 0, p_zero: float = 0.5) -> np.ndarray:
    """bf16 bits of values in {-1, 0, +1}; zero with probability ``p_zero``."""
    n = int(np.prod(shape))
    g = _rng(seed, tid, layer)
    u = g.random(n, dtype=np.float32)
    s = g.integers(0, 2, n, dtype=np.int8) * 2 - 1
    v = np.where(u < p_zero, 0, s).astype(np.float32)
    return f32_to_bf16_bits(v).reshape(shape)


def normal_f32(shape, mean: float, std: float, seed: int, tid: int, layer: int = 0) -> np.ndarray:
    """float32 N(mean, std) draws (used for initial fp32 gradient buffers)."""
    n = int(np.prod(shape))
    g = _rng(seed, tid, layer)
    x = g.standard_normal(n, dtype=np.float32) * np.float32(std) + np.float32(mean)
    return x.reshape(shape)


def e4m3_codes(shape, std: float, scale: float, seed: int, tid: int, layer: int = 0) -> np.ndarray:
    """FP8 E4M3 codes (uint8) of N(0, std) draws stored with per-tensor scale ``scale``: the draw
    divided by the scale, clipped to the largest finite magnitude 448, cast by PyTorch's
    float8_e4m3fn conversion (nearest, ties to even)."""
    import torch
    v = normal_f32(shape, 0.0, std, seed, tid, layer) / np.float32(scale)
    v = np.clip(v, -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@dataclasses.dataclass(frozen=True)
class MlpShape:
    """One workload of the chunked tensor-parallel MLP."""
    name: str
    M: int          # tokens (batch x seq)
    h: int          # hidden size
    F: int          # ffn size (per branch for gated activations)
    act: int
    t: int          # weight shards (emulated tensor-parallel ranks)
    p: int          # row chunks of X
    q: int          # column chunks of B's output dim
    layers: int = 1
    layernorm: bool = False   # pre-LN + residual stack
    backward: bool = False
    batch: int = 0
    seq: int = 0
    x_std: float = 1.0
    w_std: float = 0.02
    heads: int = 0            # > 0: Transformer blocks (attention sublayer before each MLP)

    @property
    def Fi(self) -> int:
        return self.F // self.t

    @property
    def gated(self) -> bool:
        return self.act in GATED

    @property
    def a_rows(self) -> int:
        """Rows of all A shards together (2F for gated activations)."""
        return 2 * self.F if self.gated else self.F

    @property
    def attention(self) -> bool:
        return self.heads > 0

    def attn_flops(self) -> float:
        """Flops of one attention sublayer: the QKV and output projections (2 M h 3h + 2 M h h) and
        the causal attention, 4 M d per visible key-query pair summed over heads (q.k and p.v),
        i.e. 4 h M (seq + 1) / 2 for a full sequence."""
        if not self.attention:
            return 0.0
        core = 4.0 * self.h * self.M * (self.seq + 1) / 2.0
        return 2.0 * self.M * self.h * 3 * self.h + 2.0 * self.M * self.h * self.h + core

    def gemm_flops(self) -> float:
        """Dense GEMM (and attention) flops of one pass: forward, plus backward (2x) if enabled."""
        fwd = 2.0 * self.M * self.h * self.a_rows + 2.0 * self.M * self.F * self.h + self.attn_flops()
        return self.layers * fwd * (3.0 if self.backward else 1.0)


# The five workloads.  Shapes follow GPT-3 2.7B / Llama-2 7B / GPT-3 6.7B /
# Llama-3 8B MLP blocks; the data is synthetic.
SHAPES = {
    "tiny_gelu": MlpShape("tiny_gelu", 256, 256, 1024, ACT_GELU, 2, 2, 1, batch=4, seq=64),
    "gpt3_2.7b_mlp": MlpShape("gpt3_2.7b_mlp", 16384, 2560, 10240, ACT_GELU, 8, 2, 1, batch=8, seq=2048),
    "llama2_7b_swiglu": MlpShape("llama2_7b_swiglu", 16384, 4096, 11008, ACT_SWIGLU, 8, 1, 2, batch=4, seq=4096),
    "gpt3_6.7b_stack4": MlpShape("gpt3_6.7b_stack4", 32768, 4096, 16384, ACT_GELU, 4, 2, 2, layers=4,
                                 layernorm=True, batch=16, seq=2048),
    "llama3_8b_swiglu_fwdbwd": MlpShape("llama3_8b_swiglu_fwdbwd", 32768, 4096, 14336, ACT_SWIGLU, 8, 2, 1,
                                        backward=True, batch=8, seq=4096),
    # the GPT-3 6.7B stack with its attention sublayers (32 heads of 128): full Transformer blocks
    "gpt3_6.7b_block4": MlpShape("gpt3_6.7b_block4", 32768, 4096, 16384, ACT_GELU, 4, 2, 2, layers=4,
                                 layernorm=True, batch=16, seq=2048, heads=32),
}


def make_inputs(s: MlpShape, seed: int = 0, integer: bool = False, layers: int | None = None) -> dict:
    """Seeded inputs for shape ``s`` as bf16 bit arrays (uint16).

    Keys: X [M,h]; A [L, t*(2)F_i, h]; B [L, t, h, F_i]; gY [M,h] if backward; for attention
    shapes Wqkv [L, 3h, h] (t shards of query, key and value heads) and Wo [L, t, h, h/t].
    ``integer=True`` draws every tensor from {-1, 0, +1}.
    """
    L = s.layers if layers is None else layers
    out = {}
    if integer:
        out["X"] = ternary_bf16((s.M, s.h), seed, TID_X)
        out["A"] = np.stack([ternary_bf16((s.a_rows, s.h), seed, TID_A, l) for l in range(L)])
        out["B"] = np.stack([ternary_bf16((s.t, s.h, s.Fi), seed, TID_B, l) for l in range(L)])
        if s.backward:
            out["gY"] = ternary_bf16((s.M, s.h), seed, TID_GY)
    else:
        out["X"] = normal_bf16((s.M, s.h), 0.0, s.x_std, seed, TID_X)
        out["A"] = np.stack([normal_bf16((s.a_rows, s.h), 0.0, s.w_std, seed, TID_A, l) for l in range(L)])
        out["B"] = np.stack([normal_bf16((s.t, s.h, s.Fi), 0.0, s.w_std, seed, TID_B, l) for l in range(L)])
        if s.backward:
            out["gY"] = normal_bf16((s.M, s.h), 0.0, 1.0, seed, TID_GY)
        if s.attention:
            out["Wqkv"] = np.stack([normal_bf16((3 * s.h, s.h), 0.0, s.w_std, seed, TID_WQKV, l) for l in range(L)])
            out["Wo"] = np.stack([normal_bf16((s.t, s.h, s.h // s.t), 0.0, s.w_std, seed, TID_WO, l)
                                  for l in range(L)])
    return out


def sample_indices(n: int, k: int, seed: int, tid: int = TID_MISC) -> np.ndarray:
    """``k`` sorted distinct indices in [0, n), always including 0 and n-1."""
    if k >= n:
        return np.arange(n, dtype=np.int64)
    g = _rng(seed, tid, 99)
    mid = g.choice(np.arange(1, n - 1), size=max(k - 2, 0), replace=False)
    return np.unique(np.concatenate([[0, n - 1], mid]).astype(np.int64))
