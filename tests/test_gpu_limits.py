"""GPU parity at the size limits of the C ABI.

- B = 65535 (the largest batch), whole outputs against the oracle;
- D = 2^27 (the largest channel count the kernels' 32-bit in-tile offsets
  allow), sampled channels including the last one;
- more than 2^31 (b, t, d) elements, so every global offset needs 64 bits:
  sampled chains over the whole sequence, gA on sampled channels, and the
  identity sum_s c gc = sum_d dy y on the complete outputs;
- 4096 chunks in the chunked forward, in two launches and in one with look-back.

The large inputs are a seeded block from the generator repeated along one axis
on the device, so the oracle's sub-problems are the same repetition of the
block's sampled columns on the host. Tolerances as elsewhere: float32 I/O 1e-4
(forward) and 1e-3 (gradients), bf16 I/O 1e-2, as max |got - ref| / (1 + |ref|).
"""
import numpy as np
import pytest

import gen
import oracle
from gpu_util import GRADS, assert_close, dev_inputs, sample_indices, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_03_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


def ssm():
    import selective_state_space_03_gb300 as m
    return m


def test_largest_batch():
    import torch
    w = gen.workload(2, B=65535, T=3, D=8, h0_std=0.1)
    inp = gen.make_inputs(w, with_grad_inputs=True, with_ghT=True)
    t = dev_inputs(inp)
    y, hT, ck = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=2)
    g = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck, t["dy"], t["ghT"],
                           ckpt_interval=2)
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], ckpt_interval=2)
    gref = oracle.bwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp["dy"], inp["ghT"])
    for name, got in (("y", y), ("hT", hT), ("ckpt", ck)):
        assert_close(to_host(got), ref[name], "f32", "fwd", name)
    for k in GRADS:
        assert_close(to_host(g[k]), gref[k], "f32", "grad", k)


def test_largest_channel_count():
    import torch
    D, Dbase = 1 << 27, 4096
    base = gen.make_inputs(gen.workload(5, B=1, T=3, D=Dbase), with_grad_inputs=True)
    reps = D // Dbase
    tb = dev_inputs(base)
    t = {k: tb[k].repeat(1, 1, reps) for k in ("x", "delta", "dy")}
    t["A"] = tb["A"].repeat(reps, 1)
    del tb
    K = 4
    y, hT, ck = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], to_dev(base["b"]), to_dev(base["c"]), None,
                                   ckpt_interval=K)
    g = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], to_dev(base["b"]), to_dev(base["c"]), None, ck, t["dy"],
                           ckpt_interval=K)
    torch.cuda.synchronize()
    dsel = sample_indices(D, 8, 11)
    src = dsel % Dbase
    sub = {k: base[k][:, :, src] for k in ("x", "delta", "dy")}
    ref = oracle.fwd(sub["x"], sub["delta"], base["A"][src], base["b"], base["c"], None)
    gref = oracle.bwd(sub["x"], sub["delta"], base["A"][src], base["b"], base["c"], None, sub["dy"])
    di = torch.as_tensor(dsel, device=y.device)
    assert_close(to_host(y[:, :, di]), ref["y"], "bf16", "fwd", "y")
    assert_close(to_host(hT[:, di]), ref["hT"], "bf16", "fwd", "hT")
    for k in ("gx", "gdelta"):
        assert_close(to_host(g[k][:, :, di]), gref[k], "bf16", "grad", k)
    for k in ("gA", "gh0"):
        got = g[k][di] if k == "gA" else g[k][:, di]
        assert_close(to_host(got), gref[k], "bf16", "grad", k)
    del y, hT, ck, g, t
    torch.cuda.empty_cache()


def test_more_than_2_31_elements():
    import torch
    Tbase, reps, D = 4096, 128, 4160          # B*T*D = 2.18e9 > 2^31
    base = gen.make_inputs(gen.workload(5, B=1, T=Tbase, D=D), with_grad_inputs=True)
    tb = dev_inputs(base)
    t = {k: tb[k].repeat(1, reps, 1) for k in ("x", "delta", "dy", "b", "c")}
    A = tb["A"]
    del tb
    T = Tbase * reps
    assert T * D > 2 ** 31
    K = 256
    y, hT, ck = ssm().ssm_scan_fwd(t["x"], t["delta"], A, t["b"], t["c"], None, ckpt_interval=K)
    g = ssm().ssm_scan_bwd(t["x"], t["delta"], A, t["b"], t["c"], None, ck, t["dy"], ckpt_interval=K)
    torch.cuda.synchronize()
    dsel = sample_indices(D, 4, 12)
    sub = {k: np.tile(base[k][:, :, dsel], (1, reps, 1)) for k in ("x", "delta", "dy")}
    bt, ct = np.tile(base["b"], (1, reps, 1)), np.tile(base["c"], (1, reps, 1))
    ref = oracle.fwd(sub["x"], sub["delta"], base["A"][dsel], bt, ct, None)
    gref = oracle.bwd(sub["x"], sub["delta"], base["A"][dsel], bt, ct, None, sub["dy"])
    di = torch.as_tensor(dsel, device=y.device)
    assert_close(to_host(y[:, :, di]), ref["y"], "bf16", "fwd", "y")
    assert_close(to_host(hT[:, di]), ref["hT"], "bf16", "fwd", "hT")
    for k in ("gx", "gdelta"):
        assert_close(to_host(g[k][:, :, di]), gref[k], "bf16", "grad", k)
    assert_close(to_host(g["gA"][di]), gref["gA"], "bf16", "grad", "gA")
    assert_close(to_host(g["gh0"][:, di]), gref["gh0"], "bf16", "grad", "gh0")
    # sum_s c gc = sum_d dy y per (b, t) over the complete outputs, in float64, in slices of T
    worst = 0.0
    for t0 in range(0, T, 1 << 15):
        sl = slice(t0, t0 + (1 << 15))
        dyv, yv = t["dy"][:, sl].double(), y[:, sl].double()
        lhs = (t["c"][:, sl].double() * g["gc"][:, sl].double()).sum(-1)
        rhs = (dyv * yv).sum(-1)
        scale = (dyv.abs() * yv.abs()).sum(-1) + 1.0
        worst = max(worst, float(((lhs - rhs).abs() / scale).max()))
    assert worst < 1e-2, worst
    del y, hT, ck, g, t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("lookback", [False, True])
def test_four_thousand_chunks(lookback):
    import torch
    w = gen.workload(2, B=1, T=65536, D=8, h0_std=0.1)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    y, hT, _ = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], chunk_len=16,
                                  lookback=lookback)
    if lookback:
        ssm().lookback_status()
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(to_host(y), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(hT), ref["hT"], "f32", "fwd", "hT")
