"""Shared helpers for the GPU parity tests: moving bf16 bit arrays to and from the device,
running the library through its C ABI, and the parity tolerance."""
from __future__ import annotations

import numpy as np

from comm_overlap_gb300 import domino as dm
from comm_overlap_gb300 import synth


def dev_bf16(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def host_f64(t) -> np.ndarray:
    import torch
    bits = t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def host_bits(t) -> np.ndarray:
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Exact values (representable in float32) rounded to bf16 (RNE), as float64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64)), "not exact in fp32"
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(f)).astype(np.float64)


def within_tol(got: np.ndarray, ref: np.ndarray, rel: float = 1e-2, abs_: float = 1e-3):
    """The parity bar: max|got - ref| <= rel * max|ref| + abs."""
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = rel * (float(np.max(np.abs(ref))) if ref.size else 0.0) + abs_
    return err <= bound, err, bound


def assert_tol(got, ref, what="", rel=1e-2, abs_=1e-3):
    ok, err, bound = within_tol(got, ref, rel, abs_)
    assert ok, f"{what}: max abs err {err:.4g} > bound {bound:.4g}"


class Lib:
    """One library handle plus workspace management for tests."""

    def __init__(self):
        self.h = dm.domino_create()
        self._ws = None

    def close(self):
        dm.domino_destroy(self.h)

    def workspace(self, cfg, pass_):
        import torch
        n = dm.domino_workspace_size(cfg, pass_)
        if n == 0:
            return None, 0
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        return self._ws, n

    def fwd(self, cfg, X, A, B, save=False):
        import torch
        Y = torch.empty((cfg.M, cfg.h), dtype=torch.bfloat16, device="cuda")
        a_rows = 2 * cfg.ffn if cfg.act in synth.GATED else cfg.ffn
        S = torch.empty((cfg.M, a_rows), dtype=torch.bfloat16, device="cuda") if save else None
        ws, n = self.workspace(cfg, dm.PASS_FWD)
        dm.domino_mlp_fwd(self.h, cfg, X, A, B, Y, S, ws, n)
        torch.cuda.synchronize()
        return Y, S

    def bwd(self, cfg, X, A, B, S, gY, gA0, gB0):
        import torch
        gX = torch.empty((cfg.M, cfg.h), dtype=torch.bfloat16, device="cuda")
        gA = gA0.clone()
        gB = gB0.clone()
        ws, n = self.workspace(cfg, dm.PASS_BWD)
        dm.domino_mlp_bwd(self.h, cfg, X, A, B, S, gY, gX, gA, gB, ws, n)
        torch.cuda.synchronize()
        return gX, gA, gB

    def stack(self, cfg, Z, A, B):
        import torch
        out = torch.empty_like(Z)
        ws, n = self.workspace(cfg, dm.PASS_STACK)
        dm.domino_stack_fwd(self.h, cfg, Z, A, B, out, ws, n)
        torch.cuda.synchronize()
        return out

    def status(self):
        return dm.domino_device_status(self.h)


TILE_M = 256   # output rows of one GEMM tile (a CTA pair's 2 x 128)
TILE_N = 256   # output columns of one GEMM tile


def edge_rows(M: int, m: int, seed: int, n_random: int = 12) -> np.ndarray:
    """Rows where a row-indexing mistake would show: both sides of every row-chunk boundary (m - 1,
    m, ...), of the first tile boundaries inside a chunk (127/128 inside a CTA's half, 255/256
    between tiles) and of the chunk's last tile (m - 256 .. m - 1, the last round of the persistent
    grid), plus `n_random` rows drawn at random (0 and M - 1 always among them)."""
    rows = set(synth.sample_indices(M, n_random, seed).tolist())
    for c0 in range(0, M, m):
        for off in (0, 1, 127, 128, TILE_M - 1, TILE_M, m - TILE_M - 1, m - TILE_M, m - 129, m - 128, m - 1):
            if 0 <= off < m:
                rows.add(c0 + off)
    return np.array(sorted(rows), dtype=np.int64)


def edge_feats(Fi: int, t: int, seed: int, n_random: int = 6) -> np.ndarray:
    """ffn features to check in the weight gradients: the first and last feature of every shard and
    both sides of the shard's first tile boundary (TILE_N - 1, TILE_N), plus `n_random` at random."""
    feats = set(synth.sample_indices(Fi * t, n_random, seed).tolist())
    for i in range(t):
        for j in (0, TILE_N - 1, TILE_N, Fi - 1):
            if 0 <= j < Fi:
                feats.add(i * Fi + j)
    return np.array(sorted(feats), dtype=np.int64)
