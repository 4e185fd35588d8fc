"""ctypes binding of ``libflp.so`` (the C ABI in ``include/flp.h``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  torch is used for device memory, streams and dtype bookkeeping.
Loading fails loudly (``FlpError``) when the library is missing; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libflp.so")

FLP_OK = 0
FLP_ERR_INVALID_ARG = 1
FLP_ERR_UNSUPPORTED = 2
FLP_ERR_WORKSPACE = 3
FLP_ERR_CUDA = 4
FLP_ERR_BAD_TARGET = 5
FLP_ERR_TIMEOUT = 6
FLP_F32 = 0
FLP_BF16 = 1

EXPORTS = ("flp_workspace_query", "flp_workspace_query_ex", "flp_forward", "flp_backward", "flp_get_error",
           "flp_set_phase_events", "flp_status_string", "flp_last_error_message",
           "flp_forward_noalloc", "flp_selftest_wait_timeout", "flp_loss", "flp_backward_ex",
           "flp_backward_plan", "flp_backward_schedule", "flp_selftest_dependency_timeout",
           "flp_selftest_dz_wait_timeout", "flp_policy_loss")
FLP_LOSS_NLL_MEAN = 1
FLP_LOSS_CLIPPED_SURROGATE = 2
FLP_LOSS_NLL_SUM = 3
FLP_IS_TOKEN = 0
FLP_IS_SEQUENCE = 1
FLP_AGG_TOKEN_MEAN = 0
FLP_AGG_SEQUENCE_MEAN = 1
FLP_AGG_SUM_OVER = 2
SELFTEST_WORKSPACE_BYTES = 1 << 20
SELFTEST_OUTPUT_OFFSET = 768 << 10  # the forward self-test's logprob, lse, entropy (fp32 [256] each)
STATIC_SCRATCH_BYTES = 16 << 20
FLP_BWD_AUTO = 0
FLP_BWD_SPLIT = 1
FLP_BWD_FUSED = 2
FLP_BWD_VSPLIT = 3
SCHEDULES = {"auto": FLP_BWD_AUTO, "split": FLP_BWD_SPLIT, "fused": FLP_BWD_FUSED,
             "vsplit": FLP_BWD_VSPLIT}
# phase k of flp_set_phase_events is recorded around events 2k, 2k+1; the
# backward records phase 2 (split: first wave's dZ launch; vsplit: first
# vocabulary chunk's; fused: the whole backward launch) and, except for the
# fused schedule, phase 3 (the matching dX and dW launch)
PHASES = ("fwd", "merge", "dz", "bwd_gemm")


class FlpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load the CUDA library (built by ``entropy_loss_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FlpError(FLP_ERR_CUDA, f"{path} is missing: build it with entropy_loss_gb300.build.build()")
    lib = ctypes.CDLL(path)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.flp_workspace_query.argtypes = [i64, i64, i64, i32, ctypes.POINTER(ctypes.c_size_t),
                                        ctypes.POINTER(ctypes.c_size_t)]
    lib.flp_workspace_query_ex.argtypes = [i64, i64, i64, i32, i64, ctypes.POINTER(ctypes.c_size_t),
                                           ctypes.POINTER(ctypes.c_size_t)]
    lib.flp_forward.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_float, i32, p, p, p, p,
                                ctypes.c_size_t, p]
    lib.flp_backward.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_float, i32, p, p, p, p, p,
                                 i32, p, i32, i32, p, ctypes.c_size_t, p]
    lib.flp_backward_ex.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_float, i32, p, p, p, p,
                                    p, i32, p, i32, i32, p, ctypes.c_size_t, i32, p]
    lib.flp_backward_ex.restype = i32
    lib.flp_backward_plan.argtypes = [i64, i64, i64, ctypes.c_size_t, i32,
                                      ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                      ctypes.POINTER(ctypes.c_int)]
    lib.flp_backward_plan.restype = i32
    lib.flp_backward_schedule.argtypes = [i64, i64, i64, ctypes.c_size_t, i32, i32,
                                          ctypes.POINTER(ctypes.c_int32), i64,
                                          ctypes.POINTER(ctypes.c_int64)]
    lib.flp_backward_schedule.restype = i32
    lib.flp_forward_noalloc.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_float, i32, p, p, p,
                                        p]
    lib.flp_forward_noalloc.restype = i32
    lib.flp_selftest_wait_timeout.argtypes = [p, ctypes.c_size_t, i32, i64, p]
    lib.flp_selftest_wait_timeout.restype = i32
    lib.flp_selftest_dependency_timeout.argtypes = [p, ctypes.c_size_t, i32, i64, p]
    lib.flp_selftest_dependency_timeout.restype = i32
    lib.flp_selftest_dz_wait_timeout.argtypes = [p, ctypes.c_size_t, i32, i64, p]
    lib.flp_selftest_dz_wait_timeout.restype = i32
    lib.flp_loss.argtypes = [p, p, i64, i64, i32, p, p, p, ctypes.c_float, ctypes.c_float,
                             ctypes.c_float, p, p, p, p]
    lib.flp_loss.restype = i32
    lib.flp_policy_loss.argtypes = [p, p, i64, i64, p, i64, p, p, p, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_float, i32, i32, ctypes.c_double, p, p, p, p]
    lib.flp_policy_loss.restype = i32
    lib.flp_get_error.argtypes = [p, p]
    lib.flp_set_phase_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
    lib.flp_set_phase_events.restype = i32
    lib.flp_status_string.argtypes = [i32]
    lib.flp_status_string.restype = ctypes.c_char_p
    lib.flp_last_error_message.argtypes = []
    lib.flp_last_error_message.restype = ctypes.c_char_p
    for name in ("flp_workspace_query", "flp_workspace_query_ex", "flp_forward", "flp_backward",
                 "flp_get_error"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != FLP_OK:
        lib = load()
        msg = lib.flp_status_string(status).decode()
        detail = lib.flp_last_error_message().decode()
        raise FlpError(status, f"{what}: {msg}" + (f" ({detail})" if detail else ""))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_query(M: int, H: int, V: int, compute_entropy: bool = True, chunk_rows: int = 0):
    """(forward bytes, backward bytes) on the current device; chunk_rows > 0
    sizes the backward for row waves of that many rows (flp_workspace_query_ex),
    else for the default waves (flp_workspace_query)."""
    f = ctypes.c_size_t(0)
    b = ctypes.c_size_t(0)
    lib = load()
    if chunk_rows > 0:
        _check(lib.flp_workspace_query_ex(M, H, V, int(compute_entropy), chunk_rows, ctypes.byref(f),
                                          ctypes.byref(b)), "flp_workspace_query_ex")
    else:
        _check(lib.flp_workspace_query(M, H, V, int(compute_entropy), ctypes.byref(f), ctypes.byref(b)),
               "flp_workspace_query")
    return f.value, b.value


def alloc_workspace(M: int, H: int, V: int, compute_entropy: bool = True, chunk_rows: int = 0,
                    device=None) -> torch.Tensor:
    """One uint8 device buffer large enough for both forward and backward."""
    f, b = workspace_query(M, H, V, compute_entropy, chunk_rows)
    return torch.empty(max(f, b), dtype=torch.uint8, device=device or "cuda")


def _need(t, dtype, shape, name):
    """t must be a contiguous CUDA tensor of `dtype` (or one of a tuple of
    dtypes) and `shape`: the C ABI sees only its data pointer."""
    ok_dtype = t.dtype in dtype if isinstance(dtype, tuple) else t.dtype == dtype
    if not ok_dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def _need_opt(t, dtype, shape, name):
    if t is not None:
        _need(t, dtype, shape, name)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _workspace(t):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("workspace: expected a contiguous CUDA tensor")
    return _ptr(t), _nbytes(t)


def forward(X, W, y, *, ignore_index: int = -100, scale: float = 1.0, compute_entropy: bool = True,
            workspace=None, logprob=None, lse=None, entropy=None, stream=None):
    """Per-row (logprob, lse, entropy-or-None) of softmax(scale * X W^T)."""
    M, H = X.shape
    V = W.shape[0]
    _need(X, torch.bfloat16, (M, H), "X")
    _need(W, torch.bfloat16, (V, H), "W")
    _need(y, torch.int64, (M,), "targets")
    dev = X.device
    logprob = torch.empty(M, dtype=torch.float32, device=dev) if logprob is None else logprob
    lse = torch.empty(M, dtype=torch.float32, device=dev) if lse is None else lse
    if compute_entropy and entropy is None:
        entropy = torch.empty(M, dtype=torch.float32, device=dev)
    if not compute_entropy:
        entropy = None
    for t, name in ((logprob, "logprob"), (lse, "lse"), (entropy, "entropy")):
        _need_opt(t, torch.float32, (M,), name)
    if workspace is None:
        workspace = alloc_workspace(M, H, V, compute_entropy, device=dev)
    ws_ptr, ws_bytes = _workspace(workspace)
    _check(load().flp_forward(_ptr(X), _ptr(W), _ptr(y), M, H, V, ignore_index, float(scale),
                              int(compute_entropy), _ptr(logprob), _ptr(lse), _ptr(entropy),
                              ws_ptr, ws_bytes, _stream(stream)), "flp_forward")
    return logprob, lse, entropy


def forward_noalloc(X, W, y, logprob, lse, entropy=None, *, ignore_index: int = -100,
                    scale: float = 1.0, compute_entropy: bool = True, stream=None):
    """flp_forward_noalloc: the forward without a workspace, for callers that
    cannot allocate device memory; its scratch is the library's fixed 16 MiB
    device array, shared by every call (calls that overlap on the GPU race).
    The outputs are caller-provided; nothing is allocated here."""
    M, H = X.shape
    V = W.shape[0]
    _need(X, torch.bfloat16, (M, H), "X")
    _need(W, torch.bfloat16, (V, H), "W")
    _need(y, torch.int64, (M,), "targets")
    _need(logprob, torch.float32, (M,), "logprob")
    _need(lse, torch.float32, (M,), "lse")
    if compute_entropy:
        _need(entropy, torch.float32, (M,), "entropy")
    _check(load().flp_forward_noalloc(_ptr(X), _ptr(W), _ptr(y), M, H, V, ignore_index,
                                      float(scale), int(compute_entropy), _ptr(logprob), _ptr(lse),
                                      _ptr(entropy if compute_entropy else None), _stream(stream)),
           "flp_forward_noalloc")
    return logprob, lse, entropy


def backward_plan(M: int, H: int, V: int, workspace_bytes: int, schedule: str = "auto"):
    """(wave rows, waves, schedule name) that `backward` runs with for this
    workspace size (for "vsplit", waves counts vocabulary chunks); host
    arithmetic only."""
    rows = ctypes.c_int64(0)
    waves = ctypes.c_int64(0)
    used = ctypes.c_int(0)
    _check(load().flp_backward_plan(M, H, V, workspace_bytes, SCHEDULES[schedule],
                                    ctypes.byref(rows), ctypes.byref(waves), ctypes.byref(used)),
           "flp_backward_plan")
    name = {v: k for k, v in SCHEDULES.items()}[used.value]
    return rows.value, waves.value, name


def backward_schedule(M: int, H: int, V: int, workspace_bytes: int, schedule: str = "auto",
                      pairs: int = 76):
    """The backward's units in ticket order as an int32 array of rows
    (launch, kind, wave, a, b); kind 0 dZ, 1 dX, 2 dW (see include/flp.h)."""
    import numpy as np
    lib = load()
    n = ctypes.c_int64(0)
    _check(lib.flp_backward_schedule(M, H, V, workspace_bytes, SCHEDULES[schedule], pairs, None, 0,
                                     ctypes.byref(n)), "flp_backward_schedule")
    out = np.zeros((n.value, 5), dtype=np.int32)
    _check(lib.flp_backward_schedule(M, H, V, workspace_bytes, SCHEDULES[schedule], pairs,
                                     out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n.value,
                                     ctypes.byref(n)), "flp_backward_schedule")
    return out


def backward(X, W, y, lse, entropy, grad_logprob, grad_entropy, *, ignore_index: int = -100,
             scale: float = 1.0, compute_entropy: bool = True, dX=None, dW=None,
             dx_dtype=torch.bfloat16, dw_dtype=torch.float32, accumulate_dW: bool = False,
             workspace=None, schedule: str = "auto", stream=None):
    """(dX, dW) for upstream gradients of logprob and entropy (None = zero).
    dW may be fp32 (accumulated in fp32 across waves) or bf16 (one wave only).
    schedule: "auto", "split" (per wave a dZ launch, then a dX/dW launch),
    "fused" (one persistent launch for every wave) or "vsplit" (all rows at
    once, the vocabulary in chunks: dX accumulates over the chunks in fp32)."""
    M, H = X.shape
    V = W.shape[0]
    _need(X, torch.bfloat16, (M, H), "X")
    _need(W, torch.bfloat16, (V, H), "W")
    _need(y, torch.int64, (M,), "targets")
    _need(lse, torch.float32, (M,), "lse")
    if compute_entropy:
        _need(entropy, torch.float32, (M,), "entropy")
    _need_opt(grad_logprob, torch.float32, (M,), "grad_logprob")
    if compute_entropy:
        _need_opt(grad_entropy, torch.float32, (M,), "grad_entropy")
    if schedule not in SCHEDULES:
        raise ValueError(f"schedule must be one of {sorted(SCHEDULES)}")
    dev = X.device
    if dX is None:
        dX = torch.empty(M, H, dtype=dx_dtype, device=dev)
    if dW is None:
        dW = torch.empty(V, H, dtype=dw_dtype, device=dev)
    _need(dX, (torch.bfloat16, torch.float32), (M, H), "dX")
    _need(dW, (torch.bfloat16, torch.float32), (V, H), "dW")
    dxt = FLP_F32 if dX.dtype == torch.float32 else FLP_BF16
    dwt = FLP_F32 if dW.dtype == torch.float32 else FLP_BF16
    if workspace is None:
        workspace = alloc_workspace(M, H, V, compute_entropy, device=dev)
    ws_ptr, ws_bytes = _workspace(workspace)
    _check(load().flp_backward_ex(_ptr(X), _ptr(W), _ptr(y), M, H, V, ignore_index, float(scale),
                                  int(compute_entropy), _ptr(lse),
                                  _ptr(entropy if compute_entropy else None), _ptr(grad_logprob),
                                  _ptr(grad_entropy if compute_entropy else None), _ptr(dX), dxt,
                                  _ptr(dW), dwt, int(accumulate_dW), ws_ptr, ws_bytes,
                                  SCHEDULES[schedule], _stream(stream)),
           "flp_backward_ex")
    return dX, dW


def set_phase_events(events) -> None:
    """Instrument the next calls on this thread: `events` is a list of up to 10
    torch.cuda.Event (or None) recorded around the kernel phases (start, stop)
    of PHASES in order; None turns the instrumentation off."""
    if not events:
        _check(load().flp_set_phase_events(None, 0), "flp_set_phase_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[(e.cuda_event if e is not None else None)
                                            for e in events])
    _check(load().flp_set_phase_events(arr, len(events)), "flp_set_phase_events")


def selftest_wait_timeout(stall_after: int, wait_limit_ns: int, workspace=None, stream=None) -> int:
    """Run the forward kernel with its producers stopped after `stall_after`
    stages (< 0: no stall) and every wait bounded by `wait_limit_ns`; returns
    the error status the run leaves (FLP_ERR_TIMEOUT when the stall was
    detected, FLP_OK for a normal run)."""
    if workspace is None:
        workspace = torch.empty(SELFTEST_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    return int(load().flp_selftest_wait_timeout(_ptr(workspace), _nbytes(workspace), stall_after,
                                                wait_limit_ns, _stream(stream)))


def selftest_dz_wait_timeout(stall_after: int, wait_limit_ns: int, workspace=None, stream=None) -> int:
    """Run the backward's dZ kernel on one internal 256 x 512 tile with its
    producers stopped after `stall_after` stages (< 0: no stall) and every wait
    bounded by `wait_limit_ns`; returns the error status the run leaves
    (FLP_ERR_TIMEOUT when the stall was detected, FLP_OK for a normal run)."""
    if workspace is None:
        workspace = torch.empty(SELFTEST_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    return int(load().flp_selftest_dz_wait_timeout(_ptr(workspace), _nbytes(workspace), stall_after,
                                                   wait_limit_ns, _stream(stream)))


def selftest_dependency_timeout(broken: bool, wait_limit_ns: int, workspace=None, stream=None) -> int:
    """Run one fused-schedule backward launch on a small internal problem;
    with `broken` its dX tile waits on a dZ tile that is never scheduled, so
    the dependency wait must give up after `wait_limit_ns`.  Returns the error
    status the run leaves (FLP_ERR_TIMEOUT when broken, FLP_OK otherwise)."""
    if workspace is None:
        workspace = torch.empty(SELFTEST_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    return int(load().flp_selftest_dependency_timeout(_ptr(workspace), _nbytes(workspace),
                                                      int(bool(broken)), wait_limit_ns,
                                                      _stream(stream)))


def loss(logprob, y, kind=FLP_LOSS_NLL_MEAN, *, ignore_index: int = -100, old_logprob=None,
         advantage=None, ref_logprob=None, eps_low: float = 0.2, eps_high: float = 0.2,
         beta: float = 0.0, per_token=True, stream=None):
    """Loss head on per-row log-probs: (scalar loss [1], grad_logprob [M],
    per-token terms [M] or None).  grad_logprob is the upstream gradient for
    `backward`."""
    M = logprob.shape[0]
    _need(logprob, torch.float32, (M,), "logprob")
    _need(y, torch.int64, (M,), "targets")
    for t, name in ((old_logprob, "old_logprob"), (advantage, "advantage"), (ref_logprob, "ref_logprob")):
        _need_opt(t, torch.float32, (M,), name)
    dev = logprob.device
    out = torch.empty(1, dtype=torch.float32, device=dev)
    grad = torch.empty(M, dtype=torch.float32, device=dev)
    per = torch.empty(M, dtype=torch.float32, device=dev) if per_token else None
    _check(load().flp_loss(_ptr(logprob), _ptr(y), M, ignore_index, int(kind), _ptr(old_logprob),
                           _ptr(advantage), _ptr(ref_logprob), float(eps_low), float(eps_high),
                           float(beta), _ptr(per), _ptr(grad), _ptr(out), _stream(stream)),
           "flp_loss")
    return out, grad, per


def policy_loss(logprob, y, old_logprob, advantage, *, seq_offsets=None, ignore_index: int = -100,
                ref_logprob=None, eps_low: float = 0.2, eps_high: float = 0.2, beta: float = 0.0,
                is_level: int = FLP_IS_TOKEN, aggregation: int = FLP_AGG_TOKEN_MEAN,
                normalizer: float = 0.0, per_token=True, stream=None):
    """Clipped-surrogate loss over sequences (flp_policy_loss): (scalar loss
    [1], grad_logprob [M], per-token terms [M] or None).  seq_offsets: int64
    [B + 1] device tensor of the sequences' row offsets (None: one sequence).
    aggregation FLP_AGG_SUM_OVER with normalizer = num_items_in_batch is dapo."""
    M = logprob.shape[0]
    _need(logprob, torch.float32, (M,), "logprob")
    _need(y, torch.int64, (M,), "targets")
    _need(old_logprob, torch.float32, (M,), "old_logprob")
    _need(advantage, torch.float32, (M,), "advantage")
    _need_opt(ref_logprob, torch.float32, (M,), "ref_logprob")
    B = 0
    if seq_offsets is not None:
        B = seq_offsets.shape[0] - 1
        _need(seq_offsets, torch.int64, (B + 1,), "seq_offsets")
    dev = logprob.device
    out = torch.empty(1, dtype=torch.float32, device=dev)
    grad = torch.empty(M, dtype=torch.float32, device=dev)
    per = torch.empty(M, dtype=torch.float32, device=dev) if per_token else None
    _check(load().flp_policy_loss(_ptr(logprob), _ptr(y), M, ignore_index, _ptr(seq_offsets), B,
                                  _ptr(old_logprob), _ptr(advantage), _ptr(ref_logprob),
                                  float(eps_low), float(eps_high), float(beta), int(is_level),
                                  int(aggregation), float(normalizer), _ptr(per), _ptr(grad),
                                  _ptr(out), _stream(stream)),
           "flp_policy_loss")
    return out, grad, per


def get_error(workspace, stream=None) -> int:
    """Synchronise the stream and return the workspace's error status code."""
    return int(load().flp_get_error(_ptr(workspace), _stream(stream)))


class FusedLinearLogprob(torch.autograd.Function):
    """autograd wrapper: returns (logprob, entropy-or-empty) of softmax(scale X W^T)."""

    @staticmethod
    def forward(ctx, X, W, y, ignore_index, scale, compute_entropy, workspace):
        lp, lse, ent = forward(X, W, y, ignore_index=ignore_index, scale=scale,
                               compute_entropy=compute_entropy, workspace=workspace)
        ctx.save_for_backward(X, W, y, lse, ent if ent is not None else lse.new_empty(0))
        ctx.cfg = (ignore_index, scale, compute_entropy, workspace)
        return lp, (ent if ent is not None else lse.new_empty(0))

    @staticmethod
    def backward(ctx, g_lp, g_ent):
        X, W, y, lse, ent = ctx.saved_tensors
        ignore_index, scale, compute_entropy, workspace = ctx.cfg
        g_lp = None if g_lp is None else g_lp.contiguous().float()
        g_ent = None if (g_ent is None or not compute_entropy) else g_ent.contiguous().float()
        # a bf16 weight gets its bf16 gradient straight from the epilogue when
        # one backward wave covers every row; otherwise fp32 waves, then a cast
        M, H, V = X.shape[0], X.shape[1], W.shape[0]
        wave_rows, _, _ = backward_plan(M, H, V, _nbytes(workspace))
        direct = W.dtype == torch.bfloat16 and wave_rows >= M
        dX, dW = backward(X, W, y, lse, ent if compute_entropy else None, g_lp, g_ent,
                          ignore_index=ignore_index, scale=scale, compute_entropy=compute_entropy,
                          dx_dtype=X.dtype, dw_dtype=torch.bfloat16 if direct else torch.float32,
                          workspace=workspace)
        return dX, dW.to(W.dtype), None, None, None, None, None


def fused_linear_logprob(X, W, y, ignore_index: int = -100, scale: float = 1.0,
                         compute_entropy: bool = True, workspace=None):
    """Differentiable per-row log-prob (and entropy) of the LM head."""
    if workspace is None:
        workspace = alloc_workspace(X.shape[0], X.shape[1], W.shape[0], compute_entropy,
                                    device=X.device)
    return FusedLinearLogprob.apply(X, W, y, ignore_index, scale, compute_entropy, workspace)
