"""Thin Python binding of libdomino.so (include/domino.h), same names as the C ABI.

Argument marshalling only: tensors are passed as device pointers
(``Tensor.data_ptr()``), streams as ``cudaStream_t`` handles; every step of the
computation runs in the library's CUDA kernels.  If the library is missing the
calls raise ``DominoError`` -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdomino.so")

DOMINO_OK = 0
STATUS = {0: "DOMINO_OK", 1: "DOMINO_ERR_INVALID_ARG", 2: "DOMINO_ERR_UNSUPPORTED", 3: "DOMINO_ERR_ALIGNMENT",
          4: "DOMINO_ERR_WORKSPACE", 5: "DOMINO_ERR_CUDA", 6: "DOMINO_ERR_TIMEOUT", 7: "DOMINO_ERR_DEVICE"}
ACT_NONE, ACT_RELU, ACT_GELU, ACT_SWIGLU, ACT_BILINEAR = 0, 1, 2, 3, 4
SCHED_SERIAL, SCHED_INTRA, SCHED_INTER, SCHED_FUSED = 0, 1, 2, 3
PASS_FWD, PASS_BWD, PASS_STACK, PASS_STACK_BWD, PASS_ATTN, PASS_BLOCK, PASS_FWD_FP8 = 0, 1, 2, 3, 4, 5, 6
(K_GEMM_FWD1, K_GEMM_FWD2, K_SHARD_SUM, K_LAYERNORM, K_GEMM_DGRAD_H, K_GEMM_WGRAD_B, K_GEMM_DGRAD_X,
 K_GEMM_WGRAD_A, K_LN_BWD, K_GEMM_QKV, K_ATTN, K_GEMM_OPROJ) = range(12)
KERNEL_NAMES = ["gemm_fwd1", "gemm_fwd2", "shard_sum", "layernorm", "gemm_dgrad_h", "gemm_wgrad_b",
                "gemm_dgrad_x", "gemm_wgrad_a", "layernorm_bwd", "gemm_qkv", "attention", "gemm_oproj"]


class DominoError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class domino_cfg(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("h", ctypes.c_int64), ("ffn", ctypes.c_int64), ("t", ctypes.c_int32),
                ("p", ctypes.c_int32), ("q", ctypes.c_int32), ("act", ctypes.c_int32), ("sched", ctypes.c_int32),
                ("layers", ctypes.c_int32), ("ln_eps", ctypes.c_float), ("flags", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("seq", ctypes.c_int32), ("reduce_ctas", ctypes.c_int32),
                ("attn_ctas", ctypes.c_int32)]


def make_cfg(M, h, ffn, t, p=1, q=1, act=ACT_GELU, sched=SCHED_INTRA, layers=1, ln_eps=1e-5, flags=0, heads=0,
             seq=0, reduce_ctas=0, attn_ctas=0) -> domino_cfg:
    return domino_cfg(M, h, ffn, t, p, q, act, sched, layers, ln_eps, flags, heads, seq, reduce_ctas, attn_ctas)


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_S = ctypes.c_int32

_SIGS = {
    "domino_create": [ctypes.POINTER(ctypes.c_void_p)],
    "domino_destroy": [_P],
    "domino_workspace_size": [ctypes.POINTER(domino_cfg), ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)],
    "domino_mlp_fwd": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "domino_mlp_bwd": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "domino_mlp_fwd_noalloc": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, _P],
    "domino_stack_fwd": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "domino_stack_save_size": [ctypes.POINTER(domino_cfg), ctypes.POINTER(ctypes.c_size_t)],
    "domino_stack_fwd_train": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, ctypes.c_size_t, _P,
                               ctypes.c_size_t, _P],
    "domino_stack_bwd": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, ctypes.c_size_t, _P, _P, _P, _P, _P,
                         ctypes.c_size_t, _P],
    "domino_mlp_fwd_fp8": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, ctypes.POINTER(ctypes.c_float), _P, _P,
                           ctypes.c_size_t, _P],
    "domino_attn_fwd": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "domino_block_fwd": [_P, ctypes.POINTER(domino_cfg), _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "domino_shard_sum": [_P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, _P, ctypes.c_int64, _P,
                         ctypes.c_int64, _P],
    "domino_act_eval": [ctypes.c_int32, _P, _P, _P, _P, _P, ctypes.c_int64, _P],
    "domino_device_status": [_P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
    "domino_timing_enable": [_P, ctypes.c_int32],
    "domino_timing_reset": [_P],
    "domino_timing_read": [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)],
    "domino_launch_count": [_P, ctypes.POINTER(ctypes.c_int64)],
    "domino_selftest_wait_timeout": [_P, ctypes.c_uint32, _P],
    "domino_debug_fail_launch": [_P, ctypes.c_int32],
    "domino_debug_skip_reduce": [_P, ctypes.c_int32],
    "domino_timing_trace": [_P, ctypes.c_int64, _P, _P, _P, ctypes.POINTER(ctypes.c_int64)],
    "domino_status_string": [ctypes.c_int32],
    "domino_last_error": [],
}


def lib() -> ctypes.CDLL:
    """The loaded library; raises DominoError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise DominoError(5, f"{LIB_PATH} is missing: build it with `python -m comm_overlap_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, args in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_char_p if name in ("domino_status_string", "domino_last_error") else _S
            _lib = L
    return _lib


def _check(status: int):
    if status != DOMINO_OK:
        raise DominoError(status, lib().domino_last_error().decode())


def _ptr(x):
    """Device pointer of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def domino_status_string(status: int) -> str:
    return lib().domino_status_string(status).decode()


def domino_last_error() -> str:
    return lib().domino_last_error().decode()


def domino_create() -> int:
    h = ctypes.c_void_p()
    _check(lib().domino_create(ctypes.byref(h)))
    return h.value


def domino_destroy(handle: int) -> None:
    _check(lib().domino_destroy(handle))


def domino_workspace_size(cfg: domino_cfg, pass_: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().domino_workspace_size(ctypes.byref(cfg), pass_, ctypes.byref(n)))
    return n.value


def domino_mlp_fwd(handle, cfg, X, A, B, Y, act_save, workspace, workspace_bytes=None, stream=None) -> None:
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None and workspace is not None else (
        workspace_bytes or 0)
    _check(lib().domino_mlp_fwd(handle, ctypes.byref(cfg), _ptr(X), _ptr(A), _ptr(B), _ptr(Y), _ptr(act_save),
                                _ptr(workspace), wb, _stream(stream)))


def domino_mlp_bwd(handle, cfg, X, A, B, act_save, gY, gX, gA, gB, workspace, workspace_bytes=None,
                   stream=None) -> None:
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None and workspace is not None else (
        workspace_bytes or 0)
    _check(lib().domino_mlp_bwd(handle, ctypes.byref(cfg), _ptr(X), _ptr(A), _ptr(B), _ptr(act_save), _ptr(gY),
                                _ptr(gX), _ptr(gA), _ptr(gB), _ptr(workspace), wb, _stream(stream)))


def domino_mlp_fwd_noalloc(handle, cfg, X, A, B, Y, act_save, stream=None) -> None:
    """domino_mlp_fwd without a workspace argument: the scratch is the library's fixed 64 MiB
    device array (for callers that cannot allocate); see include/domino.h."""
    _check(lib().domino_mlp_fwd_noalloc(handle, ctypes.byref(cfg), _ptr(X), _ptr(A), _ptr(B), _ptr(Y),
                                        _ptr(act_save), _stream(stream)))


def domino_stack_fwd(handle, cfg, Z_in, A, B, Z_out, workspace, workspace_bytes=None, stream=None) -> None:
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None and workspace is not None else (
        workspace_bytes or 0)
    _check(lib().domino_stack_fwd(handle, ctypes.byref(cfg), _ptr(Z_in), _ptr(A), _ptr(B), _ptr(Z_out),
                                  _ptr(workspace), wb, _stream(stream)))


def _nbytes(buf, given):
    if given is not None:
        return given
    return 0 if buf is None else buf.numel() * buf.element_size()


def domino_mlp_fwd_fp8(handle, cfg, X8, A8, B8, scales, Y, workspace, workspace_bytes=None, stream=None) -> None:
    """scales = (sx, sa, sb, sh); X8, A8, B8 are uint8 tensors of E4M3 codes."""
    sc = (ctypes.c_float * 4)(*[float(v) for v in scales])
    _check(lib().domino_mlp_fwd_fp8(handle, ctypes.byref(cfg), _ptr(X8), _ptr(A8), _ptr(B8), sc, _ptr(Y),
                                    _ptr(workspace), _nbytes(workspace, workspace_bytes), _stream(stream)))


def domino_attn_fwd(handle, cfg, X, Wqkv, Wo, Y, workspace, workspace_bytes=None, stream=None) -> None:
    _check(lib().domino_attn_fwd(handle, ctypes.byref(cfg), _ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(Y), _ptr(workspace),
                                 _nbytes(workspace, workspace_bytes), _stream(stream)))


def domino_block_fwd(handle, cfg, Z_in, Wqkv, Wo, A, B, Z_out, workspace, workspace_bytes=None, stream=None) -> None:
    _check(lib().domino_block_fwd(handle, ctypes.byref(cfg), _ptr(Z_in), _ptr(Wqkv), _ptr(Wo), _ptr(A), _ptr(B),
                                  _ptr(Z_out), _ptr(workspace), _nbytes(workspace, workspace_bytes),
                                  _stream(stream)))


def domino_stack_save_size(cfg) -> int:
    n = ctypes.c_size_t()
    _check(lib().domino_stack_save_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def domino_stack_fwd_train(handle, cfg, Z_in, A, B, Z_out, save, workspace, save_bytes=None, workspace_bytes=None,
                           stream=None) -> None:
    _check(lib().domino_stack_fwd_train(handle, ctypes.byref(cfg), _ptr(Z_in), _ptr(A), _ptr(B), _ptr(Z_out),
                                        _ptr(save), _nbytes(save, save_bytes), _ptr(workspace),
                                        _nbytes(workspace, workspace_bytes), _stream(stream)))


def domino_stack_bwd(handle, cfg, A, B, save, gZ_out, gZ_in, gA, gB, workspace, save_bytes=None,
                     workspace_bytes=None, stream=None) -> None:
    _check(lib().domino_stack_bwd(handle, ctypes.byref(cfg), _ptr(A), _ptr(B), _ptr(save), _nbytes(save, save_bytes),
                                  _ptr(gZ_out), _ptr(gZ_in), _ptr(gA), _ptr(gB), _ptr(workspace),
                                  _nbytes(workspace, workspace_bytes), _stream(stream)))


def domino_shard_sum(P, t, rows, cols, residual, ld_res, Y, ld_y, stream=None) -> None:
    _check(lib().domino_shard_sum(_ptr(P), t, rows, cols, _ptr(residual), ld_res, _ptr(Y), ld_y, _stream(stream)))


def domino_act_eval(act, a, b, out, da, db, n, stream=None) -> None:
    _check(lib().domino_act_eval(act, _ptr(a), _ptr(b), _ptr(out), _ptr(da), _ptr(db), n, _stream(stream)))


def domino_device_status(handle) -> tuple[int, int]:
    st, site = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().domino_device_status(handle, ctypes.byref(st), ctypes.byref(site)))
    return st.value, site.value


def domino_timing_enable(handle, enable: bool) -> None:
    _check(lib().domino_timing_enable(handle, int(bool(enable))))


def domino_timing_reset(handle) -> None:
    _check(lib().domino_timing_reset(handle))


def domino_timing_read(handle, kind: int) -> tuple[int, float]:
    n, ms = ctypes.c_int64(), ctypes.c_double()
    _check(lib().domino_timing_read(handle, kind, ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


SELFTEST_SITE = 0x7F0


def domino_selftest_wait_timeout(handle, timeout_us: int, stream=None) -> None:
    _check(lib().domino_selftest_wait_timeout(handle, timeout_us, _stream(stream)))


def domino_debug_fail_launch(handle, nth: int) -> None:
    _check(lib().domino_debug_fail_launch(handle, nth))


def domino_debug_skip_reduce(handle, enable: bool) -> None:
    _check(lib().domino_debug_skip_reduce(handle, int(bool(enable))))


def domino_timing_trace(handle):
    """Timed launches since the last reset, in issue order: list of (kind, start_ms, end_ms)."""
    n = ctypes.c_int64()
    _check(lib().domino_timing_trace(handle, 0, None, None, None, ctypes.byref(n)))
    cap = n.value
    kinds = (ctypes.c_int32 * max(cap, 1))()
    t0 = (ctypes.c_double * max(cap, 1))()
    t1 = (ctypes.c_double * max(cap, 1))()
    _check(lib().domino_timing_trace(handle, cap, kinds, t0, t1, ctypes.byref(n)))
    return [(int(kinds[i]), float(t0[i]), float(t1[i])) for i in range(min(cap, n.value))]


def domino_launch_count(handle) -> int:
    n = ctypes.c_int64()
    _check(lib().domino_launch_count(handle, ctypes.byref(n)))
    return n.value
