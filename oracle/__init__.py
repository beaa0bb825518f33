"""Python access to the CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package.  It wraps liboracle.so (plain C, double precision) with
numpy arrays.  Inputs are either bf16 bit patterns (uint16) or float64 arrays;
the storage format is the one described in oracle.h.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import build as _build

ACT_NONE, ACT_RELU, ACT_GELU, ACT_SWIGLU, ACT_BILINEAR = 0, 1, 2, 3, 4
_GATED = (ACT_SWIGLU, ACT_BILINEAR)

_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_D = ctypes.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            for name in ("oracle_mlp_fwd_bf16", "oracle_mlp_fwd_f64"):
                f = getattr(L, name)
                f.argtypes = [_I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _I64, _I, _P, _P]
                f.restype = _I
            for name in ("oracle_mlp_bwd_bf16", "oracle_mlp_bwd_f64"):
                f = getattr(L, name)
                f.argtypes = [_I64, _I64, _I64, _I, _I, _P, _P, _P, _P, _P, _I64, _P, _P, _I64, _P, _P]
                f.restype = _I
            for name in ("oracle_layernorm_bf16", "oracle_layernorm_f64"):
                f = getattr(L, name)
                f.argtypes = [_I64, _I64, _D, _P, _P, _I64, _P]
                f.restype = _I
            L.oracle_stack_fwd_bf16.argtypes = [_I, _I64, _I64, _I64, _I, _I, _D, _P, _P, _P, _P, _I64, _P]
            L.oracle_stack_fwd_bf16.restype = _I
            for name in ("oracle_stack_bwd_bf16", "oracle_stack_bwd_f64"):
                f = getattr(L, name)
                f.argtypes = [_I, _I64, _I64, _I64, _I, _I, _D, _P, _P, _P, _P, _P, _I64, _P, _P, _P]
                f.restype = _I
            for name in ("oracle_act", "oracle_act_grad"):
                getattr(L, name).argtypes = [_I, _D]
                getattr(L, name).restype = _D
            for name in ("oracle_glu", "oracle_glu_dg", "oracle_glu_du"):
                getattr(L, name).argtypes = [_I, _D, _D]
                getattr(L, name).restype = _D
            L.oracle_attn_fwd_bf16.argtypes = [_I64, _I64, _I, _I64, _I, _P, _P, _P, _P, _I64, _I, _P]
            L.oracle_attn_fwd_bf16.restype = _I
            L.oracle_block_fwd_bf16.argtypes = [_I, _I64, _I64, _I64, _I, _I64, _I, _I, _D, _P, _P, _P, _P, _P, _P,
                                                _I64, _I64, _P]
            L.oracle_block_fwd_bf16.restype = _I
            L.oracle_mlp_fwd_fp8.argtypes = [_I64, _I64, _I64, _I, _I, _P, _P, _P, _D, _D, _D, _D, _P, _I64, _P, _P]
            L.oracle_mlp_fwd_fp8.restype = _I
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = _D
            L.oracle_e4m3_encode.argtypes = [_D]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_num_threads.restype = _I
            _lib = L
    return _lib


def _kind(*arrays):
    dts = {a.dtype for a in arrays}
    if dts == {np.dtype(np.uint16)}:
        return "bf16"
    if dts == {np.dtype(np.float64)}:
        return "f64"
    raise TypeError(f"oracle inputs must all be uint16 (bf16 bits) or all float64, got {dts}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, len(r)


def _shape(X, A, B, t, act):
    M, h = X.shape
    Fi = B.shape[-1]
    F = Fi * t
    rows_a = 2 * F if act in _GATED else F
    if A.shape[-2:] != (rows_a, h) or B.shape[-3:] != (t, h, Fi):
        raise ValueError(f"shape mismatch: X {X.shape} A {A.shape} B {B.shape} t={t}")
    return M, h, F


def mlp_fwd(X, A, B, t, act, rows=None, sharded=False, return_h=False):
    """Y (n_rows x h, float64) of the tensor-parallel MLP; optionally H (n_rows x F)."""
    X, A, B = (np.ascontiguousarray(a) for a in (X, A, B))
    k = _kind(X, A, B)
    M, h, F = _shape(X, A, B, t, act)
    r, n = _rows(rows)
    n_out = n if r is not None else M
    Y = np.empty((n_out, h), np.float64)
    H = np.empty((n_out, F), np.float64) if return_h else None
    rc = getattr(lib(), f"oracle_mlp_fwd_{k}")(M, h, F, t, act, _ptr(X), _ptr(A), _ptr(B), _ptr(r), n,
                                             int(sharded), _ptr(Y), _ptr(H))
    if rc != 0:
        raise ValueError(f"oracle_mlp_fwd failed ({rc})")
    return (Y, H) if return_h else Y


def mlp_bwd(X, A, B, gY, t, act, rows=None, feats=None, want_dx=True, want_dw=True):
    """(dX, dA, dB) of the MLP for output gradient gY.

    dX: n_rows x h.  dA: n_feats x R x h (R = 2 for gated: gate row, up row).
    dB: n_feats x h with dB[ff, c] = dL/dBfull[c, f].
    """
    X, A, B, gY = (np.ascontiguousarray(a) for a in (X, A, B, gY))
    k = _kind(X, A, B, gY)
    M, h, F = _shape(X, A, B, t, act)
    r, n = _rows(rows)
    f, nf = _rows(feats)
    n_out = n if r is not None else M
    nf_out = nf if f is not None else F
    R = 2 if act in _GATED else 1
    dX = np.empty((n_out, h), np.float64) if want_dx else None
    dA = np.empty((nf_out, R, h), np.float64) if want_dw else None
    dB = np.empty((nf_out, h), np.float64) if want_dw else None
    rc = getattr(lib(), f"oracle_mlp_bwd_{k}")(M, h, F, t, act, _ptr(X), _ptr(A), _ptr(B), _ptr(gY),
                                             _ptr(r), n, _ptr(dX), _ptr(f), nf, _ptr(dA), _ptr(dB))
    if rc != 0:
        raise ValueError(f"oracle_mlp_bwd failed ({rc})")
    return dX, dA, dB


def layernorm(Z, eps=1e-5, rows=None):
    Z = np.ascontiguousarray(Z)
    k = _kind(Z)
    M, h = Z.shape
    r, n = _rows(rows)
    out = np.empty((n if r is not None else M, h), np.float64)
    rc = getattr(lib(), f"oracle_layernorm_{k}")(M, h, eps, _ptr(Z), _ptr(r), n, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_layernorm failed ({rc})")
    return out


def stack_fwd(Z, A, B, t, act, eps=1e-5, rows=None):
    """Z_L of the pre-LN residual stack; A: [L, a_rows, h], B: [L, t, h, F_i] (bf16 bits)."""
    Z, A, B = (np.ascontiguousarray(a) for a in (Z, A, B))
    if _kind(Z, A, B) != "bf16":
        raise TypeError("stack_fwd takes bf16 bit arrays")
    L = A.shape[0]
    M, h, F = _shape(Z, np.empty(A.shape[1:], A.dtype), np.empty(B.shape[1:], B.dtype), t, act)
    r, n = _rows(rows)
    out = np.empty((n if r is not None else M, h), np.float64)
    rc = lib().oracle_stack_fwd_bf16(L, M, h, F, t, act, eps, _ptr(Z), _ptr(A), _ptr(B), _ptr(r), n,
                                     _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_stack_fwd failed ({rc})")
    return out


def stack_bwd(Z, A, B, gZ, t, act, eps=1e-5, rows=None, want_w=False):
    """(gZ0, dA, dB) of the pre-LN residual stack for the output gradient gZ.

    A: [L, a_rows, h], B: [L, t, h, F_i].  gZ0: n_rows x h.  dA, dB (want_w, all rows only):
    the weight gradients in the A and B storage layouts, [L, a_rows, h] and [L, t, h, F_i].
    """
    Z, A, B, gZ = (np.ascontiguousarray(a) for a in (Z, A, B, gZ))
    k = _kind(Z, A, B, gZ)
    L = A.shape[0]
    M, h, F = _shape(Z, np.empty(A.shape[1:], A.dtype), np.empty(B.shape[1:], B.dtype), t, act)
    if want_w and rows is not None:
        raise ValueError("weight gradients need every row")
    r, n = _rows(rows)
    gZ0 = np.empty((n if r is not None else M, h), np.float64)
    dA = np.empty(A.shape, np.float64) if want_w else None
    dB = np.empty(B.shape, np.float64) if want_w else None
    rc = getattr(lib(), f"oracle_stack_bwd_{k}")(L, M, h, F, t, act, eps, _ptr(Z), _ptr(A), _ptr(B), _ptr(gZ),
                                               _ptr(r), n, _ptr(gZ0), _ptr(dA), _ptr(dB))
    if rc != 0:
        raise ValueError(f"oracle_stack_bwd failed ({rc})")
    return gZ0, dA, dB


def attn_fwd(X, Wqkv, Wo, t, heads, seq, rows=None, sharded=False):
    """Attention sublayer Y = sum over heads of causal attention(X) . Wo^T (no residual).

    X: M x h bf16 bits (sequences of `seq` consecutive tokens); Wqkv: (3h) x h as t shards of
    (3 h/t) x h (query heads, key heads, value heads); Wo: t x h x (h/t).  Returns n_rows x h.
    """
    X, Wqkv, Wo = (np.ascontiguousarray(a) for a in (X, Wqkv, Wo))
    assert X.dtype == np.uint16 and Wqkv.dtype == np.uint16 and Wo.dtype == np.uint16
    M, h = X.shape
    r, n = _rows(rows)
    Y = np.empty((n if r is not None else M, h), np.float64)
    rc = lib().oracle_attn_fwd_bf16(M, h, heads, seq, t, _ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(r), n, int(sharded),
                                    _ptr(Y))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd failed ({rc})")
    return Y


def block_fwd(Z, Wqkv, Wo, A, B, t, heads, seq, act, eps=1e-5, seqs=None, upto=None):
    """Pre-LN transformer block stack, L = Wqkv.shape[0] layers of Z += Attn(LN(Z)); Z += MLP(LN(Z)).

    Returns the selected sequences' positions 0 .. upto-1: n_seqs x upto x h (all sequences and
    positions by default).  Per-layer weights stacked on axis 0: Wqkv L x 3h x h, Wo L x t x h x h/t,
    A L x a_rows x h, B L x t x h x F/t.
    """
    Z, Wqkv, Wo, A, B = (np.ascontiguousarray(a) for a in (Z, Wqkv, Wo, A, B))
    M, h = Z.shape
    L = Wqkv.shape[0]
    F = B.shape[1] * B.shape[3]
    upto = seq if upto is None else int(upto)
    sq, ns = _rows(seqs)
    n_out = ns if sq is not None else M // seq
    out = np.empty((n_out, upto, h), np.float64)
    rc = lib().oracle_block_fwd_bf16(L, M, h, F, heads, seq, t, act, eps, _ptr(Z), _ptr(Wqkv), _ptr(Wo), _ptr(A),
                                     _ptr(B), _ptr(sq), ns, upto, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_block_fwd failed ({rc})")
    return out


def mlp_fwd_fp8(X8, A8, B8, t, act, scales, rows=None, return_h8=False):
    """FP8 forward: E4M3 codes (uint8) in the MLP layouts, scales = (sx, sa, sb, sh).  Returns Y
    (n_rows x h, double) and, with return_h8, the E4M3 codes of the quantised first-linear output."""
    X8, A8, B8 = (np.ascontiguousarray(a, dtype=np.uint8) for a in (X8, A8, B8))
    M, h = X8.shape
    F = B8.shape[-1] * t
    r, n = _rows(rows)
    n_out = n if r is not None else M
    Y = np.empty((n_out, h), np.float64)
    H8 = np.empty((n_out, F), np.uint8) if return_h8 else None
    sx, sa, sb, sh = (float(v) for v in scales)
    rc = lib().oracle_mlp_fwd_fp8(M, h, F, t, act, _ptr(X8), _ptr(A8), _ptr(B8), sx, sa, sb, sh, _ptr(r), n,
                                  _ptr(Y), _ptr(H8))
    if rc != 0:
        raise ValueError(f"oracle_mlp_fwd_fp8 failed ({rc})")
    return (Y, H8) if return_h8 else Y


def e4m3_decode(codes):
    f = lib().oracle_e4m3_decode
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([f(int(v)) for v in c.ravel()]).reshape(c.shape)


def e4m3_encode(x):
    f = lib().oracle_e4m3_encode
    a = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def act(a, z):
    f = lib().oracle_act
    return np.array([f(a, float(v)) for v in np.ravel(z)]).reshape(np.shape(z))


def act_grad(a, z):
    f = lib().oracle_act_grad
    return np.array([f(a, float(v)) for v in np.ravel(z)]).reshape(np.shape(z))


def glu(a, g, u):
    return lib().oracle_glu(a, float(g), float(u))


def glu_dg(a, g, u):
    return lib().oracle_glu_dg(a, float(g), float(u))


def glu_du(a, g, u):
    return lib().oracle_glu_du(a, float(g), float(u))


def num_threads() -> int:
    return int(lib().oracle_num_threads())
