"""Pins for the float64 oracle (CPU only).

Each test checks the oracle against something other than its own loop: a
hand-worked example, closed forms, an explicit O(T^2) sum that multiplies the
decays through sums of exponents, invariants, central finite differences,
Euler identities of the loss, and torch's float64 autograd. The mutation tests
at the end compile deliberately wrong copies of the oracle and check that these
pins reject each of them.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

import gen
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_problem(seed, B, T, D, DS, h0=True, ghT=False):
    r = np.random.default_rng(seed)
    p = {
        "x": r.standard_normal((B, T, D)),
        "delta": np.logaddexp(0.0, r.standard_normal((B, T, D)) - 1.0),
        "A": -np.exp(r.uniform(0.0, 2.0, (D, DS))),
        "b": r.standard_normal((B, T, DS)),
        "c": r.standard_normal((B, T, DS)),
        "h0": r.standard_normal((B, D, DS)) if h0 else None,
        "dy": r.standard_normal((B, T, D)),
        "ghT": r.standard_normal((B, D, DS)) if ghT else None,
    }
    return p


def run_fwd(p, **kw):
    return oracle.fwd(p["x"], p["delta"], p["A"], p["b"], p["c"], p["h0"], **kw)


def run_bwd(p):
    return oracle.bwd(p["x"], p["delta"], p["A"], p["b"], p["c"], p["h0"], p["dy"], p["ghT"])


# ---------------------------------------------------------------- golden fixture

def load_golden(name):
    env = {"__builtins__": {}, "ln2": math.log(2.0)}
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = np.array([float(eval(tok, env)) for tok in rest.split()])
    return vals


def test_golden_dyadic_worked_example():
    g = load_golden("dyadic_T3_DS2.txt")
    B, T, D, DS = (int(v) for v in g["B T D DS"])
    p = {
        "x": g["x"].reshape(B, T, D), "delta": g["delta"].reshape(B, T, D),
        "A": g["A"].reshape(D, DS), "b": g["b"].reshape(B, T, DS), "c": g["c"].reshape(B, T, DS),
        "h0": g["h0"].reshape(B, D, DS), "dy": g["dy"].reshape(B, T, D),
        "ghT": g["ghT"].reshape(B, D, DS),
    }
    f = run_fwd(p)
    np.testing.assert_allclose(f["y"].ravel(), g["y"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(f["hT"].ravel(), g["hT"], rtol=0, atol=1e-14)
    gr = run_bwd(p)
    for k in ("gx", "gdelta", "gA", "gb", "gc", "gh0"):
        np.testing.assert_allclose(gr[k].ravel(), g[k], rtol=0, atol=1e-14, err_msg=k)
    assert abs(oracle.loss(f["y"], f["hT"], p["dy"], p["ghT"]) - g["L"][0]) < 1e-14


# ---------------------------------------------------------------- forward pins

def test_geometric_series_closed_form():
    """Constant delta, b, x over t: h_t = a^(t+1) h0 + u (1 - a^(t+1)) / (1 - a)."""
    r = np.random.default_rng(1)
    B, T, D, DS = 2, 37, 3, 16
    delta0 = np.logaddexp(0, r.standard_normal((B, D)) - 2)
    x0 = r.standard_normal((B, D))
    b0 = r.standard_normal((B, DS))
    A = -np.exp(r.uniform(-1, 1.5, (D, DS)))
    h0 = r.standard_normal((B, D, DS))
    c = r.standard_normal((B, T, DS))
    p = {"x": np.repeat(x0[:, None, :], T, 1), "delta": np.repeat(delta0[:, None, :], T, 1),
         "b": np.repeat(b0[:, None, :], T, 1), "c": c, "A": A, "h0": h0}
    f = run_fwd(p)
    a = np.exp(delta0[:, :, None] * A[None])                    # (B, D, DS)
    u = delta0[:, :, None] * x0[:, :, None] * b0[:, None, :]   # (B, D, DS)
    for t in (0, 1, 5, T - 1):
        at = a ** (t + 1)
        ht = at * h0 + u * (1 - at) / (1 - a)
        yt = np.einsum("bds,bs->bd", ht, c[:, t])
        np.testing.assert_allclose(f["y"][:, t], yt, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(f["hT"], ht, rtol=1e-11, atol=1e-12)


def explicit_sum_forward(p):
    """y_t = sum_s c_t[s] (exp(A L_{0..t}) h0 + sum_k exp(A L_{k+1..t}) u_k), L = sums of delta."""
    x, delta, A, b, c, h0 = p["x"], p["delta"], p["A"], p["b"], p["c"], p["h0"]
    B, T, D = x.shape
    DS = A.shape[1]
    y = np.zeros((B, T, D))
    hT = np.zeros((B, D, DS))
    cs = np.concatenate([np.zeros((B, 1, D)), np.cumsum(delta, axis=1)], axis=1)  # cs[t] = sum_{<t}
    for t in range(T):
        h = np.exp(A[None] * (cs[:, t + 1])[:, :, None]) * (h0 if h0 is not None else 0.0)
        for k in range(t + 1):
            decay = np.exp(A[None] * (cs[:, t + 1] - cs[:, k + 1])[:, :, None])
            u = (delta[:, k] * x[:, k])[:, :, None] * b[:, k][:, None, :]
            h = h + decay * u
        y[:, t] = np.einsum("bds,bs->bd", h, c[:, t])
        hT = h
    return y, hT


def test_explicit_sum_bruteforce():
    p = rand_problem(2, B=2, T=9, D=3, DS=5)
    f = run_fwd(p)
    y, hT = explicit_sum_forward(p)
    np.testing.assert_allclose(f["y"], y, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(f["hT"], hT, rtol=1e-10, atol=1e-12)


def test_c_zero_gives_zero_readout():
    p = rand_problem(3, B=2, T=20, D=4, DS=16)
    p["c"] = np.zeros_like(p["c"])
    f = run_fwd(p)
    assert np.all(f["y"] == 0.0)
    assert np.any(f["hT"] != 0.0)


def test_x_zero_is_pure_decay_of_h0():
    p = rand_problem(4, B=2, T=25, D=3, DS=16)
    p["x"] = np.zeros_like(p["x"])
    f = run_fwd(p)
    cum = np.cumsum(p["delta"], axis=1)                            # (B, T, D)
    hT = np.exp(p["A"][None] * cum[:, -1][:, :, None]) * p["h0"]
    np.testing.assert_allclose(f["hT"], hT, rtol=1e-12, atol=1e-300)
    t = 11
    ht = np.exp(p["A"][None] * cum[:, t][:, :, None]) * p["h0"]
    np.testing.assert_allclose(f["y"][:, t], np.einsum("bds,bs->bd", ht, p["c"][:, t]), rtol=1e-11,
                               atol=1e-14)


def test_linearity_in_x_and_h0():
    p1 = rand_problem(5, B=2, T=15, D=3, DS=8)
    p2 = rand_problem(6, B=2, T=15, D=3, DS=8)
    p2.update({k: p1[k] for k in ("delta", "A", "b", "c")})
    ps = dict(p1, x=p1["x"] + p2["x"], h0=p1["h0"] + p2["h0"])
    f1, f2, fs = run_fwd(p1), run_fwd(p2), run_fwd(ps)
    np.testing.assert_allclose(fs["y"], f1["y"] + f2["y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fs["hT"], f1["hT"] + f2["hT"], rtol=1e-11, atol=1e-12)
    p3 = dict(p1, x=2.5 * p1["x"], h0=2.5 * p1["h0"])
    np.testing.assert_allclose(run_fwd(p3)["y"], 2.5 * f1["y"], rtol=1e-12, atol=1e-13)


def test_chunk_invariance_and_checkpoints_bitwise():
    p = rand_problem(7, B=2, T=50, D=4, DS=16)
    f = run_fwd(p, ckpt_interval=16)
    k = 16
    first = {key: (v[:, :k] if key in ("x", "delta", "b", "c", "dy") else v) for key, v in p.items()}
    second = {key: (v[:, k:] if key in ("x", "delta", "b", "c", "dy") else v) for key, v in p.items()}
    f1 = run_fwd(first)
    second["h0"] = f1["hT"]
    f2 = run_fwd(second)
    assert np.array_equal(np.concatenate([f1["y"], f2["y"]], axis=1), f["y"])
    assert np.array_equal(f2["hT"], f["hT"])
    # slot j = state entering step j*K
    assert f["ckpt"].shape == (4, 2, 4, 16)
    assert np.array_equal(f["ckpt"][0], p["h0"])
    assert np.array_equal(f["ckpt"][1], f1["hT"])
    for j in (2, 3):
        pj = {key: (v[:, :16 * j] if key in ("x", "delta", "b", "c", "dy") else v) for key, v in p.items()}
        assert np.array_equal(f["ckpt"][j], run_fwd(pj)["hT"])


def test_empty_and_degenerate_sizes():
    p = rand_problem(8, B=2, T=0, D=3, DS=16, ghT=True)
    f = run_fwd(p)
    assert f["y"].shape == (2, 0, 3)
    assert np.array_equal(f["hT"], p["h0"])
    g = run_bwd(p)
    assert np.array_equal(g["gh0"], p["ghT"]) and np.all(g["gA"] == 0)
    p0 = rand_problem(9, B=0, T=5, D=3, DS=16)
    assert run_fwd(p0)["y"].shape == (0, 5, 3)
    pn = rand_problem(10, B=2, T=6, D=3, DS=16, h0=False)
    fn = run_fwd(pn)
    fz = run_fwd(dict(pn, h0=np.zeros((2, 3, 16))))
    assert np.array_equal(fn["y"], fz["y"])


# ---------------------------------------------------------------- backward pins

def loss_of(p):
    f = run_fwd(p)
    return oracle.loss(f["y"], f["hT"], p["dy"], p["ghT"])


@pytest.mark.parametrize("with_ghT", [False, True])
def test_backward_central_finite_differences(with_ghT):
    p = rand_problem(11, B=2, T=5, D=3, DS=4, ghT=with_ghT)
    g = run_bwd(p)
    names = {"x": "gx", "delta": "gdelta", "A": "gA", "b": "gb", "c": "gc", "h0": "gh0"}
    for name, gname in names.items():
        theta = p[name]
        num = np.zeros_like(theta)
        for i in np.ndindex(theta.shape):
            step = 1e-6 * max(1.0, abs(theta[i]))
            old = theta[i]
            theta[i] = old + step
            lp = loss_of(p)
            theta[i] = old - step
            lm = loss_of(p)
            theta[i] = old
            num[i] = (lp - lm) / (2 * step)
        scale = max(1.0, np.max(np.abs(num)))
        np.testing.assert_allclose(g[gname], num, rtol=0, atol=1e-7 * scale, err_msg=gname)


def test_backward_euler_identities():
    """Identities that follow from homogeneity of the loss, checked per chain/batch/channel.

    I1: sum_s c gc = sum_d dy y per (b, t)           (L linear in c)
    I2: sum_t x gx + sum_s h0 gh0 = L_(b,d) per chain (L linear in (x, h0) jointly)
    I3: sum_{t,s} b gb + sum_{d,s} h0 gh0 = L_b       (L linear in (b, h0) jointly)
    I4: sum_{b,t} delta gdelta = sum_s A gA + sum_{b,t} x gx per d
        (delta -> k delta, A -> A / k, x -> x / k leaves L unchanged)
    """
    p = rand_problem(12, B=3, T=40, D=6, DS=16, ghT=True)
    f = run_fwd(p)
    g = run_bwd(p)
    Lchain = np.einsum("btd,btd->bd", p["dy"], f["y"]) + np.einsum("bds,bds->bd", p["ghT"], f["hT"])
    i1l = np.einsum("bts,bts->bt", p["c"], g["gc"])
    i1r = np.einsum("btd,btd->bt", p["dy"], f["y"])
    np.testing.assert_allclose(i1l, i1r, rtol=1e-11, atol=1e-11)
    i2 = np.einsum("btd,btd->bd", p["x"], g["gx"]) + np.einsum("bds,bds->bd", p["h0"], g["gh0"])
    np.testing.assert_allclose(i2, Lchain, rtol=1e-11, atol=1e-11)
    i3 = np.einsum("bts,bts->b", p["b"], g["gb"]) + np.einsum("bds,bds->b", p["h0"], g["gh0"])
    np.testing.assert_allclose(i3, Lchain.sum(1), rtol=1e-11, atol=1e-11)
    i4l = np.einsum("btd,btd->d", p["delta"], g["gdelta"])
    i4r = np.einsum("ds,ds->d", p["A"], g["gA"]) + np.einsum("btd,btd->d", p["x"], g["gx"])
    np.testing.assert_allclose(i4l, i4r, rtol=1e-10, atol=1e-10)


def test_backward_matches_torch_autograd_float64():
    torch = pytest.importorskip("torch")
    p = rand_problem(13, B=2, T=7, D=5, DS=16, ghT=True)
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()
          if k in ("x", "delta", "A", "b", "c", "h0")}
    h = tp["h0"]
    ys = []
    for t in range(p["x"].shape[1]):
        dt = tp["delta"][:, t, :, None]
        h = torch.exp(dt * tp["A"]) * h + dt * tp["b"][:, t, None, :] * tp["x"][:, t, :, None]
        ys.append((h * tp["c"][:, t, None, :]).sum(-1))
    y = torch.stack(ys, 1)
    L = (y * torch.tensor(p["dy"])).sum() + (h * torch.tensor(p["ghT"])).sum()
    grads = torch.autograd.grad(L, [tp[k] for k in ("x", "delta", "A", "b", "c", "h0")])
    g = run_bwd(p)
    for name, tg in zip(("gx", "gdelta", "gA", "gb", "gc", "gh0"), grads):
        np.testing.assert_allclose(g[name], tg.numpy(), rtol=1e-11, atol=1e-12, err_msg=name)
    np.testing.assert_allclose(run_fwd(p)["y"], y.detach().numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- fused prologue / epilogue pins

def test_softplus_and_sigmoid_values():
    v = np.linspace(-30.0, 30.0, 121)
    assert oracle.softplus(np.array(0.0)) == pytest.approx(math.log(2.0), rel=1e-15)
    np.testing.assert_allclose(oracle.softplus(v) - oracle.softplus(-v), v, rtol=0, atol=1e-13)   # sp(v) - sp(-v) = v
    np.testing.assert_allclose(oracle.softplus(np.array([50.0, 700.0])), [50.0, 700.0], rtol=1e-15)
    np.testing.assert_allclose(oracle.softplus(np.array([-40.0])), [math.exp(-40.0)], rtol=1e-12)
    assert oracle.sigmoid(np.array(0.0)) == 0.5
    np.testing.assert_allclose(oracle.sigmoid(v) + oracle.sigmoid(-v), 1.0, rtol=0, atol=1e-15)
    h = 1e-5
    num = (oracle.softplus(v + h) - oracle.softplus(v - h)) / (2 * h)                             # d softplus = sigmoid
    np.testing.assert_allclose(oracle.sigmoid(v), num, rtol=0, atol=1e-9)


def fused_problem(seed, B, T, D, DS, ghT=True):
    p = rand_problem(seed, B, T, D, DS, ghT=ghT)
    r = np.random.default_rng(seed + 1000)
    p["delta"] = r.standard_normal((B, T, D)) - 1.0       # raw values, softplus applied by the scan
    p["D_skip"] = r.standard_normal(D)
    return p


def fused_fwd(p, **kw):
    return oracle.fwd_fused(p["x"], p["delta"], p["A"], p["b"], p["c"], p["h0"], p["D_skip"], delta_softplus=True,
                            **kw)


def fused_bwd(p):
    return oracle.bwd_fused(p["x"], p["delta"], p["A"], p["b"], p["c"], p["h0"], p["dy"], p["ghT"], p["D_skip"],
                            delta_softplus=True)


def test_fused_skip_alone_when_readout_is_zero():
    p = fused_problem(21, B=2, T=9, D=5, DS=16)
    p["c"] = np.zeros_like(p["c"])
    y = fused_fwd(p)["y"]
    assert np.array_equal(y, p["x"] * p["D_skip"][None, None, :])


def test_fused_backward_central_finite_differences():
    p = fused_problem(22, B=2, T=5, D=3, DS=4)
    g = fused_bwd(p)

    def loss():
        f = fused_fwd(p)
        return oracle.loss(f["y"], f["hT"], p["dy"], p["ghT"])

    names = {"x": "gx", "delta": "gdelta", "A": "gA", "b": "gb", "c": "gc", "h0": "gh0", "D_skip": "gD_skip"}
    for name, gname in names.items():
        theta = p[name]
        num = np.zeros_like(theta)
        for i in np.ndindex(theta.shape):
            step = 1e-6 * max(1.0, abs(theta[i]))
            old = theta[i]
            theta[i] = old + step
            lp = loss()
            theta[i] = old - step
            lm = loss()
            theta[i] = old
            num[i] = (lp - lm) / (2 * step)
        scale = max(1.0, np.max(np.abs(num)))
        np.testing.assert_allclose(g[gname], num, rtol=0, atol=1e-7 * scale, err_msg=gname)


def test_fused_backward_matches_torch_autograd_float64():
    torch = pytest.importorskip("torch")
    p = fused_problem(23, B=2, T=7, D=5, DS=16)
    keys = ("x", "delta", "A", "b", "c", "h0", "D_skip")
    tp = {k: torch.tensor(p[k], dtype=torch.float64, requires_grad=True) for k in keys}
    dl_all = torch.nn.functional.softplus(tp["delta"])
    h = tp["h0"]
    ys = []
    for t in range(p["x"].shape[1]):
        dt = dl_all[:, t, :, None]
        h = torch.exp(dt * tp["A"]) * h + dt * tp["b"][:, t, None, :] * tp["x"][:, t, :, None]
        ys.append((h * tp["c"][:, t, None, :]).sum(-1))
    y = torch.stack(ys, 1) + tp["x"] * tp["D_skip"]
    L = (y * torch.tensor(p["dy"])).sum() + (h * torch.tensor(p["ghT"])).sum()
    grads = torch.autograd.grad(L, [tp[k] for k in keys])
    g = fused_bwd(p)
    for name, tg in zip(("gx", "gdelta", "gA", "gb", "gc", "gh0", "gD_skip"), grads):
        np.testing.assert_allclose(g[name], tg.numpy(), rtol=1e-11, atol=1e-12, err_msg=name)
    np.testing.assert_allclose(fused_fwd(p)["y"], y.detach().numpy(), rtol=1e-12, atol=1e-13)


def test_oracle_deterministic_across_thread_counts():
    p = rand_problem(14, B=2, T=30, D=37, DS=16, ghT=True)
    g1 = run_bwd(p)
    env = dict(os.environ, OMP_NUM_THREADS="1")
    code = ("import sys, numpy as np; sys.path.insert(0, %r); import oracle, pickle;"
            "p = pickle.load(open(%r, 'rb')); g = oracle.bwd(p['x'], p['delta'], p['A'], p['b'],"
            " p['c'], p['h0'], p['dy'], p['ghT']); pickle.dump(g, open(%r, 'wb'))")
    import pickle
    import tempfile
    with tempfile.TemporaryDirectory() as td:
        pin, pout = os.path.join(td, "p.pkl"), os.path.join(td, "g.pkl")
        pickle.dump(p, open(pin, "wb"))
        root = os.path.dirname(HERE)
        subprocess.run(["python", "-c", code % (root, pin, pout)], check=True, env=env)
        g2 = pickle.load(open(pout, "rb"))
    for k in g1:
        assert np.array_equal(g1[k], g2[k]), k


# ---------------------------------------------------------------- generator

def test_generator_deterministic_and_rounding():
    w = gen.workload(5, B=2, T=8, D=16)
    a = gen.make_inputs(w, seed=0)
    b = gen.make_inputs(w, seed=0)
    c = gen.make_inputs(w, seed=1)
    for k in ("x", "delta", "b", "c", "dy", "A"):
        assert np.array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k])
    assert a["x"].dtype == np.uint16 and a["A"].dtype == np.float32 and a["h0"] is None
    # round to nearest even on bf16: 1 + 2^-8 is a tie -> 1; 1 + 3*2^-8 -> 1 + 2^-6
    v = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5], dtype=np.float32)
    back = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(v))
    assert list(back) == [1.0, 1.0, 1 + 2 ** -6, -2.5]
    d = oracle.to_f64(a["delta"])
    assert d.min() > 0 and np.all(oracle.to_f64(a["A"]) < 0)
    w3 = gen.workload(3, B=1, T=4, D=8)
    A3 = gen.make_inputs(w3)["A"]
    assert np.array_equal(A3[0], -np.arange(1, 17, dtype=np.float32))


# ---------------------------------------------------------------- bf16 widening of the oracle

def bf16_value(bits):
    """A bf16 bit pattern's value from the format's definition (1 sign bit, 8 exponent
    bits with bias 127, 7 fraction bits), in plain Python arithmetic."""
    sign = -1.0 if bits & 0x8000 else 1.0
    e, f = (bits >> 7) & 0xFF, bits & 0x7F
    if e == 0xFF:
        return sign * math.inf if f == 0 else math.nan
    if e == 0:
        return sign * f * 2.0 ** -133          # subnormal: 0.f * 2^-126 = f * 2^-7 * 2^-126
    return sign * (1.0 + f / 128.0) * 2.0 ** (e - 127)


def test_bf16_widening_matches_the_format():
    # values fixed by the bf16 format itself, independent of any implementation
    fixed = {0x3F80: 1.0, 0xC020: -2.5, 0x8000: -0.0, 0x0000: 0.0, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
             0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126, 0x4049: 3.140625, 0xBF00: -0.5, 0x7F80: math.inf,
             0xFF80: -math.inf}
    bits = np.array(sorted(fixed), dtype=np.uint16)
    got = oracle.to_f64(bits)
    for b, v in zip(bits.tolist(), got.tolist()):
        assert v == fixed[b], hex(b)
        assert math.copysign(1.0, v) == math.copysign(1.0, fixed[b]), hex(b)   # -0.0 keeps its sign
    # every finite pattern against the format's definition
    every = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):        # the NaN patterns
        wide = oracle.to_f64(every)
    ref = np.array([bf16_value(int(b)) for b in every.tolist()])
    finite = np.isfinite(ref)
    assert np.array_equal(wide[finite], ref[finite])
    assert np.all(np.isnan(wide[np.isnan(ref)]))


def test_bf16_inputs_equal_their_float_values():
    # the oracle fed bf16 bit patterns gives bitwise the results of the same values given as floats
    w = gen.workload(5, B=2, T=40, D=24)
    inp = gen.make_inputs(w, seed=3)
    assert inp["x"].dtype == np.uint16
    as_float = {}
    for k in ("x", "delta", "b", "c", "dy"):
        flat = [bf16_value(int(v)) for v in inp[k].ravel().tolist()]
        as_float[k] = np.array(flat, dtype=np.float64).reshape(inp[k].shape)
    f1 = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], None, ckpt_interval=16)
    f2 = oracle.fwd(as_float["x"], as_float["delta"], inp["A"], as_float["b"], as_float["c"], None,
                    ckpt_interval=16)
    for k in f1:
        assert np.array_equal(f1[k], f2[k]), k
    g1 = oracle.bwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], None, inp["dy"])
    g2 = oracle.bwd(as_float["x"], as_float["delta"], inp["A"], as_float["b"], as_float["c"], None, as_float["dy"])
    for k in g1:
        assert np.array_equal(g1[k], g2[k]), k


# ---------------------------------------------------------------- mutation tests

MUTANTS = {
    # y read from the state before the update
    "readout_before_update": ("                h[s] = a * h[s] + u;\n                acc += h[s] * cm[(b * T + t) * DS + s];",
                              "                acc += h[s] * cm[(b * T + t) * DS + s];\n                h[s] = a * h[s] + u;"),
    # wrong sign in the decay
    "decay_sign": ("const double a = exp(dt * A[d * DS + s]);\n                const double u",
                   "const double a = exp(-dt * A[d * DS + s]);\n                const double u"),
    # gdelta loses the input-injection term
    "gdelta_drops_xq": ("gdelta[(b * T + t) * D + d] = r + xt * q;", "gdelta[(b * T + t) * D + d] = r;"),
    # adjoint carried with the current decay before it is used (off-by-one in time)
    "carry_off_by_one": ("g[s] = dyt * cm[bts] + g[s];                 /* g_t */\n                        const double a = exp(dt * A[d * DS + s]);",
                         "const double a = exp(dt * A[d * DS + s]);\n                        g[s] = dyt * cm[bts] + a * g[s];"),
    # gc reads h_{t-1} instead of h_t
    "gc_wrong_state": ("gcp[bts] += dyt * Hs[(t + 1) * DS + s];", "gcp[bts] += dyt * Hs[t * DS + s];"),
}


def _compile_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "ssm_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", str(path),
                    "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    i64, dp = ctypes.c_int64, ctypes.c_void_p
    lib.ssm_oracle_fwd.argtypes = [i64] * 4 + [dp] * 8 + [i64, dp]
    lib.ssm_oracle_bwd.argtypes = [i64] * 4 + [dp] * 14
    lib.ssm_oracle_threads.restype = ctypes.c_int
    return lib


def _pins_pass():
    try:
        test_golden_dyadic_worked_example()
        test_explicit_sum_bruteforce()
        test_backward_euler_identities()
        test_backward_central_finite_differences(True)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistakes(tmp_path, monkeypatch, name):
    assert _pins_pass()
    monkeypatch.setattr(oracle, "_lib", _compile_mutant(tmp_path, name))
    assert not _pins_pass(), f"mutant {name} slipped through the pins"
