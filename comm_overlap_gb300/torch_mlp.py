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

`DominoStack` does the same for L layers of the pre-LN residual stack Z += MLP(LN(Z)) (A as
`[L, (2) F, h]`, B as `[L, t, h, F_i]`): its forward with gradients enabled is
`domino_stack_fwd_train`, which keeps the LayerNorm outputs, the first-linear outputs and the
LayerNorm statistics for `domino_stack_bwd` ("实现与优化", figure 10: the forward schedule run in
reverse); without gradients it is `domino_stack_fwd`.
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


class _DominoStackFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Z, A, B, module):
        M = Z.shape[0]
        cfg = module._cfg(M)
        out = torch.empty_like(Z)
        save = torch.empty(max(dm.domino_stack_save_size(cfg), 1), dtype=torch.uint8, device=Z.device)
        ws, n = module._workspace(cfg)
        dm.domino_stack_fwd_train(module.handle, cfg, Z, A, B, out, save, ws, save_bytes=save.numel(),
                                  workspace_bytes=n)
        ctx.save_for_backward(A, B, save)
        ctx.module = module
        ctx.M = M
        return out

    @staticmethod
    def backward(ctx, gZ):
        A, B, save = ctx.saved_tensors
        module = ctx.module
        cfg = module._cfg(ctx.M)
        gZ = gZ.contiguous().to(torch.bfloat16)
        gZ_in = torch.empty_like(gZ)
        if module.fuse_wgrad:
            gA, gB = A.main_grad, B.main_grad
        else:
            gA = torch.zeros(A.shape, dtype=torch.float32, device=A.device)
            gB = torch.zeros(B.shape, dtype=torch.float32, device=B.device)
        ws, n = module._workspace(cfg)
        dm.domino_stack_bwd(module.handle, cfg, A, B, save, gZ, gZ_in, gA, gB, ws, save_bytes=save.numel(),
                            workspace_bytes=n)
        if module.fuse_wgrad:
            return gZ_in, None, None, None
        return gZ_in, gA.to(A.dtype), gB.to(B.dtype), None


class DominoStack(torch.nn.Module):
    """L layers of Z += sum_i act(LN(Z) A_i^T) B_i^T (pre-LN, no affine LayerNorm parameters, the
    residual added before the one bf16 rounding of each layer), with p row chunks, q column chunks
    and the given schedule (`dm.SCHED_*`, INTER by default).  Input and output: [M, h] bf16 on the
    current CUDA device; M must be divisible by p."""

    def __init__(self, layers: int, h: int, ffn: int, t: int, p: int = 1, q: int = 1, act: int = dm.ACT_GELU,
                 sched: int = dm.SCHED_INTER, ln_eps: float = 1e-5, fuse_wgrad: bool = True,
                 init_std: float = 0.02, device: str | torch.device = "cuda"):
        super().__init__()
        if ffn % t:
            raise ValueError("ffn must be divisible by t")
        self.layers, self.h, self.ffn, self.t, self.p, self.q = layers, h, ffn, t, p, q
        self.act, self.sched, self.ln_eps, self.fuse_wgrad = act, sched, ln_eps, fuse_wgrad
        gated = act in (dm.ACT_SWIGLU, dm.ACT_BILINEAR)
        a_rows = 2 * ffn if gated else ffn
        self.A = torch.nn.Parameter(torch.empty((layers, a_rows, h), dtype=torch.bfloat16, device=device))
        self.B = torch.nn.Parameter(torch.empty((layers, t, h, ffn // t), dtype=torch.bfloat16, device=device))
        with torch.no_grad():
            self.A.normal_(0.0, init_std)
            self.B.normal_(0.0, init_std)
        if fuse_wgrad:
            self.A.main_grad = torch.zeros(self.A.shape, dtype=torch.float32, device=device)
            self.B.main_grad = torch.zeros(self.B.shape, dtype=torch.float32, device=device)
        self.handle = dm.domino_create()
        self._ws = None

    def _cfg(self, M: int):
        return dm.make_cfg(M, self.h, self.ffn, self.t, self.p, self.q, self.act, sched=self.sched,
                           layers=self.layers, ln_eps=self.ln_eps)

    def _workspace(self, cfg):
        n = max(dm.domino_workspace_size(cfg, dm.PASS_STACK), dm.domino_workspace_size(cfg, dm.PASS_STACK_BWD))
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 1), dtype=torch.uint8, device=self.A.device)
        return self._ws, n

    def zero_main_grad(self) -> None:
        if self.fuse_wgrad:
            self.A.main_grad.zero_()
            self.B.main_grad.zero_()

    def forward(self, Z: torch.Tensor) -> torch.Tensor:
        if Z.dtype != torch.bfloat16 or Z.dim() != 2 or Z.shape[1] != self.h:
            raise ValueError("Z must be a [M, h] bf16 tensor")
        Z = Z.contiguous()
        if torch.is_grad_enabled() and (Z.requires_grad or self.A.requires_grad or self.B.requires_grad):
            return _DominoStackFunction.apply(Z, self.A, self.B, self)
        cfg = self._cfg(Z.shape[0])
        out = torch.empty_like(Z)
        ws, n = self._workspace(cfg)
        dm.domino_stack_fwd(self.handle, cfg, Z, self.A, self.B, out, ws, n)
        return out

    def close(self) -> None:
        if self.handle:
            dm.domino_destroy(self.handle)
            self.handle = None
