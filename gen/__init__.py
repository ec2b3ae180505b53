"""Seeded synthetic inputs for the selective diagonal state-space scan.

This module only draws random numbers and rounds them to the storage types. It
holds none of the scan's arithmetic: both the float64 oracle and the GPU path
receive the arrays it returns.

Recipe (the benchmark workloads of the selective-scan pages, restated):
  * every tensor has its own counter-based stream: numpy's Philox4x32-10 bit
    generator keyed by (seed, tensor id); ids A=0, delta=1, x=2, b=3, c=4,
    h0=5, dy=6, ghT=7, D_skip=8;
  * normals are numpy ``standard_normal`` draws in float64;
  * ``A = -exp(A_log)``: either ``A_log[d, s] = log(s + 1)`` (so ``A = -(s+1)``,
    the "int" recipe) or ``A_log = log(U[1, 16])`` (the "uniform" recipe),
    computed in float64 and rounded to float32 (A is always float32);
  * ``delta = softplus(z + shift)``, z ~ N(0, 1), evaluated stably in float64;
    with ``raw_delta`` the array holds ``z + shift`` itself (for the fused
    softplus prologue, which applies softplus inside the scan);
  * the skip weights ``D_skip`` (one per channel, float32) ~ N(0, 1) when asked
    for (the trace page initialises them to ones; random values make a wrong
    channel index visible);
  * x, b, c, dy ~ N(0, 1); h0 is zero or N(0, std^2) and always float32;
  * float64 values are rounded to float32 (round to nearest even); for bf16 I/O
    the float32 value is then rounded to bf16 (round to nearest even). bf16
    arrays are returned as ``np.uint16`` bit patterns.

The softplus and ``-exp`` here build inputs in the shape the pages' model feeds
the scan (projections and softplus sit outside the scan library).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

TENSOR_IDS = {"A": 0, "delta": 1, "x": 2, "b": 3, "c": 4, "h0": 5, "dy": 6, "ghT": 7, "D_skip": 8}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    D: int
    DS: int
    io: str              # "f32" or "bf16": dtype of x, delta, b, c, y, dy
    A_recipe: str        # "int": A[d,s] = -(s+1); "uniform": A = -U[1,16]
    delta_shift: float   # delta = softplus(N(0,1) + delta_shift)
    h0_std: float        # 0.0 means h0 = 0
    bwd: bool            # does the workload run the backward
    ckpt_interval: int   # checkpoint interval K for fwd+bwd workloads (0: none)
    chunk_T: int = 0     # >0: the sequence is processed as chained calls of this length


# The five benchmark workloads.
WORKLOADS = {
    1: Workload("fwd_f32_B2_T64_D32", 2, 64, 32, 16, "f32", "int", -4.0, 0.1, False, 0),
    2: Workload("fwdbwd_f32_B8_T1024_D256", 8, 1024, 256, 16, "f32", "uniform", -3.0, 0.0, True, 256),
    3: Workload("fwd_bf16_B8_T4096_D1536", 8, 4096, 1536, 16, "bf16", "int", -4.0, 0.0, False, 0),
    4: Workload("fwd_f32_B1_T65536_D2048_chained4096", 1, 65536, 2048, 16, "f32", "uniform", -3.0, 0.1,
                False, 0, chunk_T=4096),
    5: Workload("fwdbwd_bf16_B16_T2048_D5120", 16, 2048, 5120, 16, "bf16", "uniform", -4.0, 0.0, True, 256),
}


def workload(n: int, **overrides) -> Workload:
    """Workload ``n`` (1..5), optionally with fields (e.g. shapes) replaced."""
    return replace(WORKLOADS[n], **overrides)


def _rng(seed: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed), TENSOR_IDS[tensor]]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _store(v64: np.ndarray, io: str) -> np.ndarray:
    v32 = v64.astype(np.float32)
    return f32_to_bf16_bits(v32) if io == "bf16" else v32


def _normal(seed, tensor, shape, chunk=1 << 24) -> np.ndarray:
    g = _rng(seed, tensor)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for i in range(0, n, chunk):  # chunked only to bound temporaries; the stream is sequential
        out[i:i + chunk] = g.standard_normal(min(chunk, n - i))
    return out.reshape(shape)


def _softplus64(z: np.ndarray) -> np.ndarray:
    # log(1 + exp(z)) without overflow
    return np.logaddexp(0.0, z)


def make_inputs(w: Workload, seed: int = 0, with_grad_inputs: bool | None = None,
                with_ghT: bool = False, raw_delta: bool = False, with_skip: bool = False) -> dict:
    """Draw the inputs of workload ``w``.

    Returns a dict with x, delta, b, c (``w.io`` storage), A and h0 (float32,
    h0 is None when ``h0_std == 0``), and dy (``w.io``) when the workload runs
    the backward. ``with_ghT`` adds an upstream gradient for hT (float32).
    """
    B, T, D, DS = w.B, w.T, w.D, w.DS
    if with_grad_inputs is None:
        with_grad_inputs = w.bwd
    out = {"workload": w, "seed": seed}
    if w.A_recipe == "int":
        A_log = np.broadcast_to(np.log(np.arange(1, DS + 1, dtype=np.float64)), (D, DS))
    elif w.A_recipe == "uniform":
        A_log = np.log(1.0 + 15.0 * _rng(seed, "A").random((D, DS)))
    else:
        raise ValueError(w.A_recipe)
    out["A"] = (-np.exp(A_log)).astype(np.float32)
    z = _normal(seed, "delta", (B, T, D))
    z += w.delta_shift
    out["delta"] = _store(z if raw_delta else _softplus64(z), w.io)
    del z
    out["x"] = _store(_normal(seed, "x", (B, T, D)), w.io)
    out["b"] = _store(_normal(seed, "b", (B, T, DS)), w.io)
    out["c"] = _store(_normal(seed, "c", (B, T, DS)), w.io)
    if w.h0_std > 0:
        out["h0"] = (w.h0_std * _normal(seed, "h0", (B, D, DS))).astype(np.float32)
    else:
        out["h0"] = None
    if with_grad_inputs:
        out["dy"] = _store(_normal(seed, "dy", (B, T, D)), w.io)
    if with_ghT:
        out["ghT"] = _normal(seed, "ghT", (B, D, DS)).astype(np.float32)
    if with_skip:
        out["D_skip"] = _normal(seed, "D_skip", (D,)).astype(np.float32)
    return out


def elements(w: Workload) -> int:
    """Scan elements B*T*D*DS of a workload (the throughput unit)."""
    return w.B * w.T * w.D * w.DS


def io_bytes(io: str) -> int:
    return 2 if io == "bf16" else 4


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "elements", "f32_to_bf16_bits",
           "bf16_bits_to_f32", "io_bytes", "ceil_div", "TENSOR_IDS"]
