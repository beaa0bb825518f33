"""PyTorch module around the chunked tensor-parallel MLP (argument marshalling only).

`DominoMLP` holds the t weight shards as bf16 parameters, A as `[t * (2) F_i, h]` and B as
`[t, h, F_i]` (nn.Linear [out, in] layout per shard, the layout of include/domino.h), and calls
`domino_mlp_fwd` / `domino_mlp_bwd` through `comm_overlap_gb300.domino`: every step of the forward
and backward runs in the library's kernels; this file only allocates outputs and passes pointers.

The forward saves the first-linear output (act_save) for the backward.  The backward writes the
input gradient and, as the Megatron recipe does ("04 · TP/SP 的通信-计算 overlap 与工程优化", §1:
weight gradients accumulated in fp32 main_grad by the weight-gradient GEMM), accumulates the
weight gradients into fp32 buffers `A.main_grad`, `B.main_grad` (`fuse_wgrad=True`, the default;
the parameters' `.grad` then stays None), or returns them as ordinary bf16 `.grad`
(`fuse_wgrad=False`).
"""
from __future__ import annotations

import torch

from . import domino as dm


class _DominoMLPFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, A, B, module):
        M = X.shape[0]
        cfg = module._cfg(M)
        Y = torch.empty((M, module.h), dtype=torch.bfloat16, device=X.device)
        S = torch.empty((M, module.a_rows), dtype=torch.bfloat16, device=X.device)
        ws, n = module._workspace(cfg)
        dm.domino_mlp_fwd(module.handle, cfg, X, A, B, Y, S, ws, n)
        ctx.save_for_backward(X, A, B, S)
        ctx.module = module
        return Y

    @staticmethod
    def backward(ctx, gY):
        X, A, B, S = ctx.saved_tensors
        module = ctx.module
        cfg = module._cfg(X.shape[0])
        gY = gY.contiguous().to(torch.bfloat16)
        gX = torch.empty_like(X)
        if module.fuse_wgrad:
            gA, gB = A.main_grad, B.main_grad
        else:
            gA = torch.zeros(A.shape, dtype=torch.float32, device=A.device)
            gB = torch.zeros(B.shape, dtype=torch.float32, device=B.device)
        ws, n = module._workspace(cfg)
        dm.domino_mlp_bwd(module.handle, cfg, X, A, B, S, gY, gX, gA, gB, ws, n)
        if module.fuse_wgrad:
            return gX, None, None, None
        return gX, gA.to(A.dtype), gB.to(B.dtype), None


class DominoMLP(torch.nn.Module):
    """Y = sum_i act(X A_i^T) B_i^T over t weight shards, with p row chunks, q column chunks and the
    given schedule (`dm.SCHED_*`).  Input and output: [M, h] bf16 on the current CUDA device; M must
    be divisible by p."""

    def __init__(self, h: int, ffn: int, t: int, p: int = 1, q: int = 1, act: int = dm.ACT_SWIGLU,
                 sched: int = dm.SCHED_INTRA, fuse_wgrad: bool = True, init_std: float = 0.02,
                 device: str | torch.device = "cuda"):
        super().__init__()
        if ffn % t:
            raise ValueError("ffn must be divisible by t")
        self.h, self.ffn, self.t, self.p, self.q, self.act, self.sched = h, ffn, t, p, q, act, sched
        self.fuse_wgrad = fuse_wgrad
        gated = act in (dm.ACT_SWIGLU, dm.ACT_BILINEAR)
        self.a_rows = 2 * ffn if gated else ffn
        self.A = torch.nn.Parameter(torch.empty((self.a_rows, h), dtype=torch.bfloat16, device=device))
        self.B = torch.nn.Parameter(torch.empty((t, h, ffn // t), dtype=torch.bfloat16, device=device))
        with torch.no_grad():
            self.A.normal_(0.0, init_std)
            self.B.normal_(0.0, init_std)
        if fuse_wgrad:
            self.A.main_grad = torch.zeros(self.A.shape, dtype=torch.float32, device=device)
            self.B.main_grad = torch.zeros(self.B.shape, dtype=torch.float32, device=device)
        self.handle = dm.domino_create()
        self._ws = None

    def _cfg(self, M: int):
        return dm.make_cfg(M, self.h, self.ffn, self.t, self.p, self.q, self.act, sched=self.sched)

    def _workspace(self, cfg):
        n = max(dm.domino_workspace_size(cfg, dm.PASS_FWD), dm.domino_workspace_size(cfg, dm.PASS_BWD))
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 1), dtype=torch.uint8, device=self.A.device)
        return self._ws, n

    def zero_main_grad(self) -> None:
        if self.fuse_wgrad:
            self.A.main_grad.zero_()
            self.B.main_grad.zero_()

    def forward(self, X: torch.Tensor) -> torch.Tensor:
        if X.dtype != torch.bfloat16 or X.dim() != 2 or X.shape[1] != self.h:
            raise ValueError("X must be a [M, h] bf16 tensor")
        return _DominoMLPFunction.apply(X.contiguous(), self.A, self.B, self)

    def close(self) -> None:
        if self.handle:
            dm.domino_destroy(self.handle)
            self.handle = None
