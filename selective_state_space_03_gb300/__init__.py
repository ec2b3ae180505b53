"""Selective diagonal state-space scan on GB300: Python binding of libssm_scan.so.

The functions here only marshal arguments: they check shapes and dtypes of
torch CUDA tensors, allocate outputs with torch, and call the C ABI declared
in ``include/ssm_scan.h`` (``ssm_scan_fwd`` / ``ssm_scan_bwd``) on the current
torch stream. Every step of the scan runs in the library's CUDA kernels; there
is no fallback. If the library has not been built, the first call raises.

    y, hT, ckpt = ssm_scan_fwd(x, delta, A, b, c, h0, ckpt_interval=256)
    grads = ssm_scan_bwd(x, delta, A, b, c, h0, ckpt, dy, ckpt_interval=256)
    y, hT = selective_scan(x, delta, A, b, c, h0)        # autograd wrapper

Shapes: x, delta (B, T, D); A (D, 16); b, c (B, T, 16); h0 (B, D, 16).
x, delta, b, c (and dy) are float32 or bfloat16 (all the same); A, h0 and the
state, hT, checkpoints and gradients are float32.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libssm_scan.so")
# The same kernels with schedule overrides read from SSM_SCAN_FORCE_* environment variables,
# for tests that pin every schedule; selected only inside ``testing_library()``.
TESTING_LIB_PATH = os.path.join(_PKG, "_lib", "libssm_scan_testing.so")

SSM_IO_F32, SSM_IO_BF16 = 0, 1
MAX_BWD_CKPT_INTERVAL = 256   # longest checkpoint interval ssm_scan_bwd reads without a rebuild
STATUS = {0: "SSM_OK", 1: "SSM_ERR_INVALID_ARG", 2: "SSM_ERR_UNSUPPORTED", 3: "SSM_ERR_MISALIGNED",
          4: "SSM_ERR_WORKSPACE", 5: "SSM_ERR_CUDA", 6: "SSM_ERR_TIMEOUT"}
EXPORTS = ("ssm_scan_ckpt_bytes", "ssm_scan_fwd_workspace_bytes", "ssm_scan_bwd_workspace_bytes",
           "ssm_scan_bwd_ckpt_workspace_bytes", "ssm_scan_fwd", "ssm_scan_bwd", "ssm_scan_fwd_fused",
           "ssm_scan_bwd_fused", "ssm_scan_step", "ssm_scan_fwd_lookback_status", "ssm_status_str")


class ssm_scan_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("D", ctypes.c_int64), ("DS", ctypes.c_int64),
                ("io", ctypes.c_int32), ("ckpt_interval", ctypes.c_int32), ("chunk_len", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({lib().ssm_status_str(status).decode()})")


_lock = threading.Lock()
_libs = {}
_testing_depth = 0


def lib() -> ctypes.CDLL:
    """The loaded C library (the testing build inside ``testing_library()``); raises if it
    has not been built."""
    path = TESTING_LIB_PATH if _testing_depth > 0 else LIB_PATH
    with _lock:
        if path not in _libs:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; "
                                   f"g.build()\"` (needs nvcc); there is no CPU fallback")
            L = ctypes.CDLL(path)
            vp, sz, dp = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ssm_scan_desc)
            for name in ("ssm_scan_ckpt_bytes", "ssm_scan_fwd_workspace_bytes", "ssm_scan_bwd_workspace_bytes",
                         "ssm_scan_bwd_ckpt_workspace_bytes"):
                getattr(L, name).argtypes = [dp]
                getattr(L, name).restype = sz
            L.ssm_scan_fwd.argtypes = [dp] + [vp] * 9 + [vp, sz, vp]
            L.ssm_scan_fwd.restype = ctypes.c_int
            L.ssm_scan_bwd.argtypes = [dp] + [vp] * 15 + [vp, sz, vp]
            L.ssm_scan_bwd.restype = ctypes.c_int
            L.ssm_scan_fwd_fused.argtypes = [dp] + [vp] * 10 + [vp, sz, vp]
            L.ssm_scan_fwd_fused.restype = ctypes.c_int
            L.ssm_scan_bwd_fused.argtypes = [dp] + [vp] * 17 + [vp, sz, vp]
            L.ssm_scan_bwd_fused.restype = ctypes.c_int
            L.ssm_scan_fwd_lookback_status.argtypes = [dp, vp, sz, vp]
            L.ssm_scan_fwd_lookback_status.restype = ctypes.c_int
            L.ssm_status_str.argtypes = [ctypes.c_int]
            L.ssm_status_str.restype = ctypes.c_char_p
            _libs[path] = L
    return _libs[path]


@contextlib.contextmanager
def testing_library():
    """Route the calls made inside the block to libssm_scan_testing.so, whose schedule
    choices (lane layouts, chunk-parallel backward, look-back polling) follow the
    SSM_SCAN_FORCE_* / SSM_SCAN_LOOKBACK_POLLS / SSM_SCAN_TEST_LOOKBACK_DROP environment
    variables. For tests only; the release library ignores those variables."""
    global _testing_depth
    _testing_depth += 1
    try:
        yield
    finally:
        _testing_depth -= 1


SSM_SCAN_DETERMINISTIC = 1


def make_desc(B, T, D, DS=16, io=SSM_IO_F32, ckpt_interval=0, chunk_len=0, flags=0) -> ssm_scan_desc:
    return ssm_scan_desc(int(B), int(T), int(D), int(DS), int(io), int(ckpt_interval), int(chunk_len), int(flags))


# ---------------------------------------------------------------- torch marshalling

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _io_of(x):
    torch = _torch()
    if x.dtype == torch.float32:
        return SSM_IO_F32
    if x.dtype == torch.bfloat16:
        return SSM_IO_BF16
    raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")


def _check(t, shape, dtype, name, device):
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device} (contiguous={t.is_contiguous()})")


def _stream(stream, device):
    torch = _torch()
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _call(device, fn, *args):
    """Call into the library with the tensors' device current (the C ABI works on the
    current CUDA device)."""
    torch = _torch()
    with torch.cuda.device(device):
        return fn(*args)


def _workspace(nbytes, device):
    torch = _torch()
    if nbytes == 0:
        return None, 0
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


SSM_SCAN_DELTA_SOFTPLUS = 2
SSM_SCAN_LOOKBACK = 4
SSM_SCAN_STEP_INPUTS_READY = 8
SSM_ERR_TIMEOUT = 6

_last_lookback = {}     # device -> (desc, workspace) of the last forward call with lookback=True


def ssm_scan_fwd(x, delta, A, b, c, h0=None, *, ckpt_interval=0, chunk_len=0, y=None, hT=None, ckpt=None,
                 workspace=None, D_skip=None, delta_softplus=False, lookback=False, stream=None):
    """Forward scan. Returns (y, hT, ckpt); ckpt is None when ckpt_interval == 0.
    delta_softplus=True: delta holds raw values, the scan uses softplus(delta)
    (SSM_SCAN_DELTA_SOFTPLUS). D_skip (D,) float32: y += D_skip * x, through
    ssm_scan_fwd_fused. lookback=True sets SSM_SCAN_LOOKBACK (a chunked schedule
    runs as one launch with decoupled look-back); lookback_status() then reports
    whether any of its bounded waits ran out."""
    torch = _torch()
    B, T, D = x.shape
    DS = A.shape[1] if A.dim() == 2 else 16
    io = _io_of(x)
    dev = x.device
    _check(delta, (B, T, D), x.dtype, "delta", dev)
    _check(A, (D, DS), torch.float32, "A", dev)
    _check(b, (B, T, DS), x.dtype, "b", dev)
    _check(c, (B, T, DS), x.dtype, "c", dev)
    _check(h0, (B, D, DS), torch.float32, "h0", dev)
    _check(D_skip, (D,), torch.float32, "D_skip", dev)
    flags = (SSM_SCAN_DELTA_SOFTPLUS if delta_softplus else 0) | (SSM_SCAN_LOOKBACK if lookback else 0)
    desc = make_desc(B, T, D, DS, io, ckpt_interval, chunk_len, flags)
    L = lib()
    if y is None:
        y = torch.empty((B, T, D), dtype=x.dtype, device=dev)
    if hT is None:
        hT = torch.empty((B, D, DS), dtype=torch.float32, device=dev)
    if ckpt is None and ckpt_interval > 0:
        nslots = -(-T // ckpt_interval)
        ckpt = torch.empty((nslots, B, D, DS), dtype=torch.float32, device=dev)
    _check(y, (B, T, D), x.dtype, "y", dev)
    _check(hT, (B, D, DS), torch.float32, "hT", dev)
    need = _call(dev, L.ssm_scan_fwd_workspace_bytes, ctypes.byref(desc))
    if workspace is None:
        workspace, wsb = _workspace(need, dev)
    else:
        wsb = workspace.numel() * workspace.element_size()
    if D_skip is None:
        st = _call(dev, L.ssm_scan_fwd, ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(b), _ptr(c), _ptr(h0),
                            _ptr(y), _ptr(hT), _ptr(ckpt), _ptr(workspace), wsb, _stream(stream, dev))
    else:
        st = _call(dev, L.ssm_scan_fwd_fused, ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(b), _ptr(c),
                                  _ptr(D_skip), _ptr(h0), _ptr(y), _ptr(hT), _ptr(ckpt), _ptr(workspace), wsb,
                                  _stream(stream, dev))
    if st != 0:
        raise SSMError(st, "ssm_scan_fwd")
    if lookback:
        _last_lookback[dev] = (desc, workspace, wsb, stream)
    return y, hT, ckpt


def lookback_status(device=None):
    """Waits for the last ssm_scan_fwd(..., lookback=True) call on `device` and
    raises SSMError(SSM_ERR_TIMEOUT) if one of its look-back waits ran out
    (ssm_scan_fwd_lookback_status). Returns None otherwise."""
    torch = _torch()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if dev not in _last_lookback:
        return None
    desc, ws, wsb, stream = _last_lookback[dev]
    st = _call(dev, lib().ssm_scan_fwd_lookback_status, ctypes.byref(desc), _ptr(ws), wsb, _stream(stream, dev))
    if st != 0:
        raise SSMError(st, "ssm_scan_fwd_lookback_status")
    return None


def ssm_scan_bwd(x, delta, A, b, c, h0, ckpt, dy, ghT=None, *, ckpt_interval=0, grads=None, workspace=None,
                 deterministic=False, D_skip=None, delta_softplus=False, stream=None):
    """Backward scan. Returns dict(gx, gdelta, gA, gb, gc, gh0), all float32, plus
    gD_skip when D_skip is given (ssm_scan_bwd_fused). deterministic=True sets
    SSM_SCAN_DETERMINISTIC (fixed-order sums, bitwise reproducible gb, gc, gA);
    delta_softplus=True sets SSM_SCAN_DELTA_SOFTPLUS (gdelta w.r.t. the raw delta)."""
    torch = _torch()
    B, T, D = x.shape
    DS = A.shape[1]
    io = _io_of(x)
    dev = x.device
    _check(dy, (B, T, D), x.dtype, "dy", dev)
    _check(ghT, (B, D, DS), torch.float32, "ghT", dev)
    _check(h0, (B, D, DS), torch.float32, "h0", dev)
    _check(D_skip, (D,), torch.float32, "D_skip", dev)
    flags = (SSM_SCAN_DETERMINISTIC if deterministic else 0) | (SSM_SCAN_DELTA_SOFTPLUS if delta_softplus else 0)
    desc = make_desc(B, T, D, DS, io, ckpt_interval, 0, flags)
    L = lib()
    f32 = dict(dtype=torch.float32, device=dev)
    g = grads or {}
    out = {
        "gx": g.get("gx", torch.empty((B, T, D), **f32)),
        "gdelta": g.get("gdelta", torch.empty((B, T, D), **f32)),
        "gA": g.get("gA", torch.empty((D, DS), **f32)),
        "gb": g.get("gb", torch.empty((B, T, DS), **f32)),
        "gc": g.get("gc", torch.empty((B, T, DS), **f32)),
        "gh0": g.get("gh0", torch.empty((B, D, DS), **f32)),
    }
    if D_skip is not None:
        out["gD_skip"] = g.get("gD_skip", torch.empty((D,), **f32))
    # the library rebuilds checkpoints in the workspace when none are given or
    # when they are further apart than the backward reads directly
    rebuild = ckpt is None or not (0 < ckpt_interval <= MAX_BWD_CKPT_INTERVAL)
    # (with checkpoints, the workspace holds the chunk-parallel carries and deterministic partials)
    need = _call(dev, L.ssm_scan_bwd_workspace_bytes if rebuild else L.ssm_scan_bwd_ckpt_workspace_bytes,
                 ctypes.byref(desc))
    if workspace is None:
        workspace, wsb = _workspace(need, dev)
    else:
        wsb = workspace.numel() * workspace.element_size()
    if D_skip is None:
        st = _call(dev, L.ssm_scan_bwd, ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(b), _ptr(c), _ptr(h0),
                            _ptr(ckpt), _ptr(dy), _ptr(ghT), _ptr(out["gx"]), _ptr(out["gdelta"]), _ptr(out["gA"]),
                            _ptr(out["gb"]), _ptr(out["gc"]), _ptr(out["gh0"]), _ptr(workspace), wsb,
                            _stream(stream, dev))
    else:
        st = _call(dev, L.ssm_scan_bwd_fused, ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(b), _ptr(c),
                                  _ptr(D_skip), _ptr(h0), _ptr(ckpt), _ptr(dy), _ptr(ghT), _ptr(out["gx"]),
                                  _ptr(out["gdelta"]), _ptr(out["gA"]), _ptr(out["gb"]), _ptr(out["gc"]),
                                  _ptr(out["gh0"]), _ptr(out["gD_skip"]), _ptr(workspace), wsb, _stream(stream, dev))
    if st != 0:
        raise SSMError(st, "ssm_scan_bwd")
    return out


def ssm_scan_fwd_noalloc(x, delta, A, b, c, h0=None, *, ckpt_interval=0, chunk_len=0, y=None, hT=None, ckpt=None,
                         delta_softplus=False, stream=None):
    """Forward scan through ssm_scan_fwd_noalloc: the chunked schedule with its
    scratch in the library's fixed device array, for callers that cannot
    allocate scratch memory (outputs can be passed in so nothing is allocated
    here either). Returns (y, hT, ckpt)."""
    torch = _torch()
    L = lib()
    fn = L.ssm_scan_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(ssm_scan_desc)] + [ctypes.c_void_p] * 10
    fn.restype = ctypes.c_int
    B, T, D = x.shape
    DS = A.shape[1]
    dev = x.device
    for t_, shape, dt, name in ((delta, (B, T, D), x.dtype, "delta"), (A, (D, DS), torch.float32, "A"),
                                (b, (B, T, DS), x.dtype, "b"), (c, (B, T, DS), x.dtype, "c"),
                                (h0, (B, D, DS), torch.float32, "h0")):
        _check(t_, shape, dt, name, dev)
    desc = make_desc(B, T, D, DS, _io_of(x), ckpt_interval, chunk_len, SSM_SCAN_DELTA_SOFTPLUS if delta_softplus else 0)
    if y is None:
        y = torch.empty((B, T, D), dtype=x.dtype, device=dev)
    if hT is None:
        hT = torch.empty((B, D, DS), dtype=torch.float32, device=dev)
    if ckpt is None and ckpt_interval > 0:
        ckpt = torch.empty((-(-T // ckpt_interval), B, D, DS), dtype=torch.float32, device=dev)
    st = _call(dev, fn, ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(b), _ptr(c), _ptr(h0), _ptr(y), _ptr(hT),
            _ptr(ckpt), _stream(stream, dev))
    if st != 0:
        raise SSMError(st, "ssm_scan_fwd_noalloc")
    return y, hT, ckpt


def ssm_scan_step(x, delta, A, b, c, h, *, y=None, delta_softplus=False, inputs_ready=False, stream=None):
    """One decode step through ssm_scan_step: x, delta (B, D), b, c (B, DS) in the I/O
    dtype, A (D, DS) and the state h (B, D, DS) float32, which is updated in place.
    inputs_ready=True sets SSM_SCAN_STEP_INPUTS_READY (the kernel before this one on the
    stream writes none of x, delta, A, b, c). Returns y (B, D)."""
    torch = _torch()
    L = lib()
    fn = L.ssm_scan_step
    fn.argtypes = [ctypes.POINTER(ssm_scan_desc)] + [ctypes.c_void_p] * 8
    fn.restype = ctypes.c_int
    B, D = x.shape
    DS = A.shape[1]
    dev = x.device
    for t_, shape, dt, name in ((delta, (B, D), x.dtype, "delta"), (A, (D, DS), torch.float32, "A"),
                                (b, (B, DS), x.dtype, "b"), (c, (B, DS), x.dtype, "c"),
                                (h, (B, D, DS), torch.float32, "h")):
        _check(t_, shape, dt, name, dev)
    flags = (SSM_SCAN_DELTA_SOFTPLUS if delta_softplus else 0) | (SSM_SCAN_STEP_INPUTS_READY if inputs_ready else 0)
    desc = make_desc(B, 1, D, DS, _io_of(x), 0, 0, flags)
    if y is None:
        y = torch.empty((B, D), dtype=x.dtype, device=dev)
    st = _call(dev, fn, ctypes.byref(desc), _ptr(x), _ptr(delta), _ptr(A), _ptr(b), _ptr(c), _ptr(h), _ptr(y), _stream(stream, dev))
    if st != 0:
        raise SSMError(st, "ssm_scan_step")
    return y


def selective_scan(x, delta, A, b, c, h0=None, ckpt_interval=256, D_skip=None, delta_softplus=False):
    """Differentiable scan: returns (y, hT). Gradients flow to x, delta, A, b, c, h0 and
    D_skip; hT is differentiated too (its gradient enters the backward as ghT).
    delta_softplus=True scans with softplus(delta) (delta given raw, its gradient w.r.t. the
    raw values); D_skip (D,) float32 adds D_skip * x to y."""
    return _ScanFn.apply(x, delta, A, b, c, h0, D_skip, ckpt_interval, bool(delta_softplus))


def _make_autograd():
    torch = _torch()

    class ScanFn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, x, delta, A, b, c, h0, D_skip, K, softplus):
            y, hT, ckpt = ssm_scan_fwd(x, delta, A, b, c, h0, ckpt_interval=K, D_skip=D_skip,
                                       delta_softplus=softplus)
            ctx.save_for_backward(x, delta, A, b, c, h0, D_skip, ckpt)
            ctx.K = K
            ctx.softplus = softplus
            ctx.has_h0 = h0 is not None
            return y, hT

        @staticmethod
        def backward(ctx, dy, dhT):
            x, delta, A, b, c, h0, D_skip, ckpt = ctx.saved_tensors
            dy = torch.zeros_like(x) if dy is None else dy.to(x.dtype).contiguous()
            ghT = None if dhT is None else dhT.float().contiguous()
            g = ssm_scan_bwd(x, delta, A, b, c, h0, ckpt, dy, ghT, ckpt_interval=ctx.K, D_skip=D_skip,
                             delta_softplus=ctx.softplus)
            return (g["gx"].to(x.dtype), g["gdelta"].to(delta.dtype), g["gA"], g["gb"].to(b.dtype),
                    g["gc"].to(c.dtype), g["gh0"] if ctx.has_h0 else None,
                    g["gD_skip"] if D_skip is not None else None, None, None)

    return ScanFn


class _Lazy:
    _fn = None

    def apply(self, *args):
        if _Lazy._fn is None:
            _Lazy._fn = _make_autograd()
        return _Lazy._fn.apply(*args)


_ScanFn = _Lazy()

__all__ = ["lib", "ssm_scan_desc", "make_desc", "ssm_scan_fwd", "ssm_scan_bwd", "ssm_scan_step",
           "ssm_scan_fwd_noalloc", "selective_scan", "SSMError", "EXPORTS", "LIB_PATH", "SSM_IO_F32", "SSM_IO_BF16",
           "SSM_SCAN_DETERMINISTIC", "SSM_SCAN_DELTA_SOFTPLUS", "SSM_SCAN_LOOKBACK", "SSM_SCAN_STEP_INPUTS_READY",
           "SSM_ERR_TIMEOUT",
           "lookback_status", "testing_library", "TESTING_LIB_PATH"]
