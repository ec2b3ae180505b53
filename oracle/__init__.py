"""Float64 CPU oracle for the selective diagonal state-space scan.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline are the only callers. The product path (the CUDA library and its
Python binding) never imports this package, and this package never imports the
product. The arithmetic lives in ``ssm_oracle.c`` (plain C, float64, OpenMP over
independent (b, d) chains); this module compiles it with gcc on first use and
marshals numpy arrays.

Inputs are upcast exactly to float64 here: float32 arrays directly, bf16 arrays
(stored as ``np.uint16`` bit patterns) by widening the bits to float32 first.

Parity pins: every function here is pinned by ``tests/test_oracle.py`` against
closed forms, an explicit O(T^2) sum, invariants, finite differences, Euler
identities of the loss and a hand-worked dyadic example under ``tests/golden/``.

The fused variants (``fwd_fused``, ``bwd_fused``) add what the model on the
POPCORNBENCH trace page ("FW-GLM-5-1__l2_p30", its forward() op list and
kernel) does around the scan: delta = softplus(delta_raw) before it and the
skip y + x * D (one weight per channel) after it. They are written here in
numpy, as plain elementwise steps around the C scan, with the chain rule for
their gradients.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no host-specific flags); return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp = ctypes.c_int64, ctypes.c_void_p
            lib.ssm_oracle_fwd.argtypes = [i64] * 4 + [dp] * 8 + [i64, dp]
            lib.ssm_oracle_fwd.restype = ctypes.c_int
            lib.ssm_oracle_bwd.argtypes = [i64] * 4 + [dp] * 14
            lib.ssm_oracle_bwd.restype = ctypes.c_int
            lib.ssm_oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().ssm_oracle_threads())


def to_f64(a):
    """Exact float64 copy of a stored array (float32/float64, or bf16 bits as uint16)."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def fwd(x, delta, A, b, c, h0=None, ckpt_interval: int = 0):
    """Forward scan in float64. Returns dict(y, hT[, ckpt])."""
    x, delta, A, b, c, h0 = (to_f64(v) for v in (x, delta, A, b, c, h0))
    B, T, D = x.shape
    DS = A.shape[1]
    assert delta.shape == (B, T, D) and A.shape == (D, DS)
    assert b.shape == (B, T, DS) and c.shape == (B, T, DS)
    assert h0 is None or h0.shape == (B, D, DS)
    y = np.empty((B, T, D))
    hT = np.empty((B, D, DS))
    K = int(ckpt_interval)
    ckpt = np.empty(((T + K - 1) // K, B, D, DS)) if K > 0 else None
    rc = _load().ssm_oracle_fwd(B, T, D, DS, _p(x), _p(delta), _p(A), _p(b), _p(c), _p(h0),
                                _p(y), _p(hT), K, _p(ckpt))
    if rc != 0:
        raise RuntimeError(f"ssm_oracle_fwd failed ({rc})")
    out = {"y": y, "hT": hT}
    if ckpt is not None:
        out["ckpt"] = ckpt
    return out


def bwd(x, delta, A, b, c, h0, dy, ghT=None):
    """Backward in float64 for L = sum(dy*y) + sum(ghT*hT).

    Returns dict(gx, gdelta, gA, gb, gc, gh0)."""
    x, delta, A, b, c, h0, dy, ghT = (to_f64(v) for v in (x, delta, A, b, c, h0, dy, ghT))
    B, T, D = x.shape
    DS = A.shape[1]
    assert dy.shape == (B, T, D)
    assert ghT is None or ghT.shape == (B, D, DS)
    gx = np.empty((B, T, D))
    gdelta = np.empty((B, T, D))
    gA = np.empty((D, DS))
    gb = np.empty((B, T, DS))
    gc = np.empty((B, T, DS))
    gh0 = np.empty((B, D, DS))
    rc = _load().ssm_oracle_bwd(B, T, D, DS, _p(x), _p(delta), _p(A), _p(b), _p(c), _p(h0),
                                _p(dy), _p(ghT), _p(gx), _p(gdelta), _p(gA), _p(gb), _p(gc),
                                _p(gh0))
    if rc != 0:
        raise RuntimeError(f"ssm_oracle_bwd failed ({rc})")
    return {"gx": gx, "gdelta": gdelta, "gA": gA, "gb": gb, "gc": gc, "gh0": gh0}


def loss(y, hT, dy, ghT=None) -> float:
    """L = sum(dy*y) + sum(ghT*hT), the scalar the backward differentiates."""
    L = float(np.sum(to_f64(dy) * y))
    if ghT is not None:
        L += float(np.sum(to_f64(ghT) * hT))
    return L


def softplus(v):
    """log(1 + e^v) in float64 (the softplus the trace page applies to delta), overflow-free."""
    return np.logaddexp(0.0, v)


def sigmoid(v):
    """1 / (1 + e^-v) in float64: the derivative of softplus."""
    return 0.5 * (1.0 + np.tanh(0.5 * v))


def fwd_fused(x, delta, A, b, c, h0=None, D_skip=None, delta_softplus: bool = False, ckpt_interval: int = 0):
    """Forward with the trace page's prologue and epilogue: the scan runs on
    softplus(delta) when ``delta_softplus`` (delta then holds the raw values),
    and y gets + x * D_skip[d] when ``D_skip`` (shape (D,)) is given."""
    dl = to_f64(delta)
    if delta_softplus:
        dl = softplus(dl)
    out = fwd(x, dl, A, b, c, h0, ckpt_interval)
    if D_skip is not None:
        out["y"] = out["y"] + to_f64(x) * to_f64(D_skip)[None, None, :]
    return out


def bwd_fused(x, delta, A, b, c, h0, dy, ghT=None, D_skip=None, delta_softplus: bool = False):
    """Backward of ``fwd_fused`` for L = sum(dy*y) + sum(ghT*hT). gdelta is with
    respect to the raw delta when ``delta_softplus``; with ``D_skip`` the skip adds
    dy * D_skip to gx and returns gD_skip[d] = sum_{b,t} dy * x."""
    raw = to_f64(delta)
    dl = softplus(raw) if delta_softplus else raw
    g = bwd(x, dl, A, b, c, h0, dy, ghT)
    if delta_softplus:
        g["gdelta"] = g["gdelta"] * sigmoid(raw)
    if D_skip is not None:
        dy64, x64 = to_f64(dy), to_f64(x)
        g["gx"] = g["gx"] + dy64 * to_f64(D_skip)[None, None, :]
        g["gD_skip"] = np.einsum("btd,btd->d", dy64, x64)
    return g
