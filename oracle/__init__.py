"""fp64 CPU oracle for the fused linear log-prob / cross-entropy LM head.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The product path (the CUDA
library and its binding) never imports this package, and this package imports
nothing from the product.

The arithmetic lives in ``flp_oracle.c`` (plain C, fp64, OpenMP over
independent rows); this module only compiles it and marshals numpy arrays.
Every function takes bf16 inputs as ``numpy.uint16`` bit patterns (the exact
bytes the GPU receives) or fp64 inputs, and returns fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flp_oracle.c")
_LIB = os.path.join(_HERE, "libflp_oracle.so")
_lock = threading.Lock()
_lib = None

FLPO_OK = 0
FLPO_INVALID_ARG = 1
FLPO_BAD_TARGET = 5


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) if stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            fwd_args = [p, p, p, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int, p, i64, p, p, p]
            bwd_args = [p, p, p, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int, p, p, p, i64,
                        ctypes.c_int, p, p]
            for name, args in (("flpo_forward_bf16", fwd_args), ("flpo_forward_f64", fwd_args),
                               ("flpo_backward_bf16", bwd_args), ("flpo_backward_f64", bwd_args)):
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            for name in ("flpo_backward_dw_cols_bf16", "flpo_backward_dw_cols_f64"):
                fn = getattr(lib, name)
                fn.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int, p, p, p,
                               i64, ctypes.c_int, p, p, p, p]
                fn.restype = ctypes.c_int
            lib.flpo_round_bf16.argtypes = [p, p, i64]
            lib.flpo_round_bf16.restype = None
            lib.flpo_loss.argtypes = [p, p, i64, i64, ctypes.c_int, p, p, p, ctypes.c_double,
                                      ctypes.c_double, ctypes.c_double, p, p, p]
            lib.flpo_loss.restype = ctypes.c_int
            lib.flpo_policy_loss.argtypes = [p, p, i64, i64, p, i64, p, p, p, ctypes.c_double,
                                             ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, p, p, p]
            lib.flpo_policy_loss.restype = ctypes.c_int
            lib.flpo_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().flpo_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(X, W, y):
    X = np.ascontiguousarray(X)
    W = np.ascontiguousarray(W)
    if X.dtype == np.uint16 and W.dtype == np.uint16:
        kind = "bf16"
    elif X.dtype == np.float64 and W.dtype == np.float64:
        kind = "f64"
    else:
        raise TypeError("X and W must both be uint16 (bf16 bits) or both float64")
    y = np.ascontiguousarray(y, dtype=np.int64)
    M, H = X.shape
    V, H2 = W.shape
    if H2 != H or y.shape != (M,):
        raise ValueError("shape mismatch")
    return X, W, y, kind, M, H, V


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.shape[0]


def forward(X, W, y, ignore_index=-100, scale=1.0, compute_entropy=True, rows=None,
            allow_bad_target=False):
    """Return (logprob, lse, entropy-or-None) for `rows` (all rows if None)."""
    lib = _load()
    X, W, y, kind, M, H, V = _prep(X, W, y)
    r, n = _rows(rows, M)
    logprob = np.zeros(n, np.float64)
    lse = np.zeros(n, np.float64)
    ent = np.zeros(n, np.float64) if compute_entropy else None
    fn = lib.flpo_forward_bf16 if kind == "bf16" else lib.flpo_forward_f64
    st = fn(_ptr(X), _ptr(W), _ptr(y), M, H, V, int(ignore_index), float(scale),
            int(bool(compute_entropy)), _ptr(r), n, _ptr(logprob), _ptr(lse), _ptr(ent))
    if st == FLPO_BAD_TARGET and not allow_bad_target:
        raise OracleError("target outside [0, V) that is not ignore_index")
    if st not in (FLPO_OK, FLPO_BAD_TARGET):
        raise OracleError(f"oracle forward failed with status {st}")
    return logprob, lse, ent


def backward(X, W, y, g_lp, g_ent, ignore_index=-100, scale=1.0, compute_entropy=True,
             rows=None, round_dz_bf16=False, want_dx=True, want_dw=True):
    """Return (dX_rows-or-None, dW-or-None).

    dX_rows[k] is the gradient row of rows[k]; dW sums the contributions of the
    listed rows only (all rows when rows is None)."""
    lib = _load()
    X, W, y, kind, M, H, V = _prep(X, W, y)
    r, n = _rows(rows, M)
    g_lp = None if g_lp is None else np.ascontiguousarray(g_lp, dtype=np.float64)
    g_ent = None if g_ent is None else np.ascontiguousarray(g_ent, dtype=np.float64)
    dx = np.zeros((n, H), np.float64) if want_dx else None
    dw = np.zeros((V, H), np.float64) if want_dw else None
    fn = lib.flpo_backward_bf16 if kind == "bf16" else lib.flpo_backward_f64
    st = fn(_ptr(X), _ptr(W), _ptr(y), M, H, V, int(ignore_index), float(scale),
            int(bool(compute_entropy)), _ptr(g_lp), _ptr(g_ent), _ptr(r), n,
            int(bool(round_dz_bf16)), _ptr(dx), _ptr(dw))
    if st not in (FLPO_OK, FLPO_BAD_TARGET):
        raise OracleError(f"oracle backward failed with status {st}")
    return dx, dw


def backward_dw_cols(X, W, y, g_lp, g_ent, cols, ignore_index=-100, scale=1.0,
                     compute_entropy=True, round_dz_bf16=False, with_forward=False):
    """dW restricted to the vocabulary rows `cols`, with every row's upstream
    gradient live: returns an fp64 array [len(cols), H] whose row c is
    sum_i dZ[i, cols[c]] X[i, :] over all rows i.  With `with_forward`,
    returns (dW_cols, logprob, lse, entropy-or-None) of every row as well
    (the same logit rows, formed once)."""
    lib = _load()
    X, W, y, kind, M, H, V = _prep(X, W, y)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    g_lp = None if g_lp is None else np.ascontiguousarray(g_lp, dtype=np.float64)
    g_ent = None if g_ent is None else np.ascontiguousarray(g_ent, dtype=np.float64)
    out = np.zeros((c.shape[0], H), np.float64)
    lp = np.zeros(M, np.float64) if with_forward else None
    lse = np.zeros(M, np.float64) if with_forward else None
    ent = np.zeros(M, np.float64) if (with_forward and compute_entropy) else None
    fn = lib.flpo_backward_dw_cols_bf16 if kind == "bf16" else lib.flpo_backward_dw_cols_f64
    st = fn(_ptr(X), _ptr(W), _ptr(y), M, H, V, int(ignore_index), float(scale),
            int(bool(compute_entropy)), _ptr(g_lp), _ptr(g_ent), _ptr(c), c.shape[0],
            int(bool(round_dz_bf16)), _ptr(out), _ptr(lp), _ptr(lse), _ptr(ent))
    if st not in (FLPO_OK, FLPO_BAD_TARGET):
        raise OracleError(f"oracle backward_dw_cols failed with status {st}")
    return (out, lp, lse, ent) if with_forward else out


def round_bf16(a) -> np.ndarray:
    """The oracle's fp32 -> bf16 rounding of each element (uint16 bit patterns)."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    out = np.zeros(f.shape, np.uint16)
    _load().flpo_round_bf16(_ptr(f), _ptr(out), f.size)
    return out


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


LOSS_NLL_MEAN = 1
LOSS_GRPO = 2
LOSS_NLL_SUM = 3
IS_TOKEN, IS_SEQUENCE = 0, 1
AGG_TOKEN_MEAN, AGG_SEQUENCE_MEAN, AGG_SUM_OVER = 0, 1, 2


def loss(logprob, y, kind, ignore_index=-100, old_logprob=None, advantage=None,
         ref_logprob=None, eps_low=0.2, eps_high=0.2, beta=0.0):
    """Loss head on per-row log-probs: returns (per_row, grad_logprob, scalar)."""
    lib = _load()
    lp = np.ascontiguousarray(logprob, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.int64)
    M = lp.shape[0]
    conv = (lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64))
    old, adv, ref = conv(old_logprob), conv(advantage), conv(ref_logprob)
    per_row = np.zeros(M)
    grad = np.zeros(M)
    out = np.zeros(1)
    st = lib.flpo_loss(_ptr(lp), _ptr(y), M, int(ignore_index), int(kind), _ptr(old), _ptr(adv),
                       _ptr(ref), float(eps_low), float(eps_high), float(beta), _ptr(per_row),
                       _ptr(grad), _ptr(out))
    if st != FLPO_OK:
        raise OracleError(f"oracle loss failed with status {st}")
    return per_row, grad, float(out[0])


def policy_loss(logprob, y, old_logprob, advantage, seq_offsets=None, ignore_index=-100,
                ref_logprob=None, eps_low=0.2, eps_high=0.2, beta=0.0, is_level=IS_TOKEN,
                aggregation=AGG_TOKEN_MEAN, normalizer=0.0):
    """Policy-gradient loss over sequences: returns (per_row, grad_logprob, scalar).
    seq_offsets: int64 [B + 1] row offsets of the sequences (None: one sequence)."""
    lib = _load()
    lp = np.ascontiguousarray(logprob, dtype=np.float64)
    y = np.ascontiguousarray(y, dtype=np.int64)
    M = lp.shape[0]
    conv = (lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64))
    old, adv, ref = conv(old_logprob), conv(advantage), conv(ref_logprob)
    off = None if seq_offsets is None else np.ascontiguousarray(seq_offsets, dtype=np.int64)
    B = 0 if off is None else off.shape[0] - 1
    per_row = np.zeros(M)
    grad = np.zeros(M)
    out = np.zeros(1)
    st = lib.flpo_policy_loss(_ptr(lp), _ptr(y), M, int(ignore_index), _ptr(off), B, _ptr(old),
                              _ptr(adv), _ptr(ref), float(eps_low), float(eps_high), float(beta),
                              int(is_level), int(aggregation), float(normalizer), _ptr(per_row),
                              _ptr(grad), _ptr(out))
    if st != FLPO_OK:
        raise OracleError(f"oracle policy loss failed with status {st}")
    return per_row, grad, float(out[0])
