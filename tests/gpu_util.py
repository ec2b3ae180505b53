"""Helpers shared by the GPU parity tests: device transfer, tolerances, sampling,
schedule overrides."""
import contextlib
import os

import numpy as np

TOL = {  # max |got - ref| / (1 + |ref|), elementwise
    ("f32", "fwd"): 1e-4,
    ("f32", "grad"): 1e-3,
    ("bf16", "fwd"): 1e-2,
    ("bf16", "grad"): 1e-2,
}
GRADS = ("gx", "gdelta", "gA", "gb", "gc", "gh0")


def to_dev(a, device="cuda:0"):
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:   # bf16 bits
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def maxrel(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    if want.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")              # a NaN would compare as 'not greater' and pass silently
    return float(np.max(np.abs(got - want) / (1.0 + np.abs(want))))


def assert_close(got, want, io, kind, name):
    err = maxrel(got, want)
    tol = TOL[(io, kind)]
    assert err <= tol, f"{name}: max rel err {err:.3g} > {tol} ({io})"
    return err


def dev_inputs(inp, keys=("x", "delta", "A", "b", "c", "h0", "dy", "ghT")):
    return {k: to_dev(inp.get(k)) for k in keys}


def sample_indices(n, k, seed):
    """k distinct indices of range(n) including both ends."""
    r = np.random.default_rng(seed)
    if n <= k:
        return np.arange(n)
    mid = r.choice(np.arange(1, n - 1), size=k - 2, replace=False)
    return np.sort(np.concatenate([[0, n - 1], mid]))


def sub_inputs(inp, bsel, dsel):
    """Inputs of the sub-problem made of chains (b in bsel) x (d in dsel)."""
    out = {}
    for k in ("x", "delta", "dy"):
        if inp.get(k) is not None:
            out[k] = inp[k][bsel][:, :, dsel]
    for k in ("b", "c"):
        out[k] = inp[k][bsel]
    out["A"] = inp["A"][dsel]
    for k in ("h0", "ghT"):
        out[k] = None if inp.get(k) is None else inp[k][bsel][:, dsel]
    return out


@contextlib.contextmanager
def forced(**env):
    """Pin schedule choices for the block: set the SSM_SCAN_* override variables given
    (None = leave unset) and route the calls to the testing build of the library, the
    only one that reads them."""
    import selective_state_space_03_gb300 as ssm
    old = {k: os.environ.get(k) for k in env}
    for k, v in env.items():
        if v is not None:
            os.environ[k] = str(v)
    try:
        with ssm.testing_library():
            yield
    finally:
        for k, v in env.items():
            if v is None:
                continue
            if old[k] is None:
                del os.environ[k]
            else:
                os.environ[k] = old[k]
