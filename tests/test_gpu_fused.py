"""GPU parity of the fused prologue / epilogue against the oracle's fused functions.

SSM_SCAN_DELTA_SOFTPLUS (delta given raw, the scan uses softplus(delta)) and the
skip y += D_skip * x (ssm_scan_fwd_fused / ssm_scan_bwd_fused, with gD_skip)
are checked through every schedule that applies them: the one-pass forward in
both lane layouts, the chunked forward, the checkpoint rebuild, both backward
layouts, the chunk-parallel backward, the deterministic sums and the decode
step. Tolerances as for the plain scan: float32 I/O 1e-4 (y, hT) and 1e-3
(gradients), bf16 I/O 1e-2, as max |got - ref| / (1 + |ref|).
"""

import numpy as np
import pytest

import gen
import oracle
from gpu_util import GRADS, assert_close, dev_inputs, to_dev, to_host, forced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_03_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def ssm():
    import selective_state_space_03_gb300 as m
    return m




def fused_case(w, K, softplus=True, skip=True, chunk_len=0, lanes=None, kd=None, tpar=None, det=False,
               rebuild=False, seed=0):
    import torch
    inp = gen.make_inputs(w, seed=seed, with_grad_inputs=True, with_ghT=True, raw_delta=softplus,
                          with_skip=skip)
    t = dev_inputs(inp)
    Ds = to_dev(inp["D_skip"]) if skip else None
    with forced(SSM_SCAN_FORCE_LANES=lanes):
        y, hT, ckpt = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K,
                                         chunk_len=chunk_len, D_skip=Ds, delta_softplus=softplus)
    torch.cuda.synchronize()
    ref = oracle.fwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp.get("D_skip"),
                           delta_softplus=softplus, ckpt_interval=K)
    assert_close(to_host(y), ref["y"], w.io, "fwd", "y")
    assert_close(to_host(hT), ref["hT"], w.io, "fwd", "hT")
    if K > 0:
        assert_close(to_host(ckpt), ref["ckpt"], w.io, "fwd", "ckpt")
    with forced(SSM_SCAN_FORCE_BWD_KD=kd, SSM_SCAN_FORCE_BWD_TPAR=tpar):
        g = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], None if rebuild else ckpt,
                               t["dy"], t["ghT"], ckpt_interval=K, D_skip=Ds, delta_softplus=softplus,
                               deterministic=det)
    torch.cuda.synchronize()
    gref = oracle.bwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp["dy"],
                            inp["ghT"], inp.get("D_skip"), delta_softplus=softplus)
    for k in GRADS + (("gD_skip",) if skip else ()):
        assert_close(to_host(g[k]), gref[k], w.io, "grad", k)
    return g


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("softplus,skip", [(True, True), (True, False), (False, True)])
def test_fused_one_pass_and_backward(io, softplus, skip):
    fused_case(gen.workload(2, B=3, T=200, D=72, io=io, h0_std=0.1), K=64, softplus=softplus, skip=skip)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_two_lane_forward_and_two_channel_backward(io):
    fused_case(gen.workload(2, B=2, T=150, D=136, io=io, h0_std=0.1), K=32, lanes=2, kd=2, tpar=0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_four_lane_two_channel_forward(io):
    with forced(SSM_SCAN_FORCE_FWD_LAYOUT="4x2"):
        fused_case(gen.workload(2, B=2, T=150, D=72, io=io, h0_std=0.1), K=32)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_chunked_forward_chunk_parallel_backward(io):
    fused_case(gen.workload(2, B=2, T=230, D=40, io=io, h0_std=0.1), K=50, chunk_len=50, kd=1, tpar=1)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk_layout", ["4x2", "2x2"])
def test_fused_chunked_forward_two_channels_per_lane(io, chunk_layout):
    # softplus prologue and skip epilogue in both chunk passes, with 4 or 2 lanes per chain
    with forced(SSM_SCAN_FORCE_CHUNK_LAYOUT=chunk_layout):
        fused_case(gen.workload(2, B=2, T=230, D=40, io=io, h0_std=0.1), K=50, chunk_len=50, kd=2, tpar=0)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_unaligned_channels_and_rebuild(io):
    D = 37 if io == "f32" else 20
    fused_case(gen.workload(2, B=2, T=77, D=D, io=io, h0_std=0.1), K=24, rebuild=True)


@pytest.mark.parametrize("layout", [dict(kd=1, tpar=0), dict(kd=2, tpar=0), dict(kd=1, tpar=1)])
def test_fused_deterministic(layout):
    import torch
    w = gen.workload(2, B=3, T=160, D=200, io="bf16", h0_std=0.1)
    g1 = fused_case(w, K=64, det=True, **layout)
    g2 = fused_case(w, K=64, det=True, **layout)
    for k in GRADS + ("gD_skip",):
        assert torch.equal(g1[k], g2[k]), k


def test_fused_workload5_shape_reduced():
    fused_case(gen.workload(5, B=2, T=600, D=264), K=256)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_step_with_softplus(io):
    import torch
    w = gen.workload(2, B=3, T=12, D=72, io=io, h0_std=0.1)
    inp = gen.make_inputs(w, seed=4, raw_delta=True)
    t = dev_inputs(inp)
    h = t["h0"].clone()
    ys = [ssm().ssm_scan_step(t["x"][:, k].contiguous(), t["delta"][:, k].contiguous(), t["A"],
                              t["b"][:, k].contiguous(), t["c"][:, k].contiguous(), h, delta_softplus=True)
          for k in range(w.T)]
    torch.cuda.synchronize()
    ref = oracle.fwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], delta_softplus=True)
    assert_close(np.stack([to_host(v) for v in ys], axis=1), ref["y"], io, "fwd", "y")
    assert_close(to_host(h), ref["hT"], io, "fwd", "hT")


@pytest.mark.parametrize("softplus,skip", [(True, True), (False, True), (True, False)])
def test_fused_autograd_wrapper(softplus, skip):
    """selective_scan with the fused options: torch autograd reaches every input's gradient,
    D_skip's included, through the fused kernels."""
    import torch
    w = gen.workload(2, B=2, T=90, D=24, h0_std=0.1)
    inp = gen.make_inputs(w, with_grad_inputs=True, with_ghT=True, raw_delta=softplus, with_skip=skip)
    t = dev_inputs(inp)
    names = ("x", "delta", "A", "b", "c", "h0")
    leaves = {k: t[k].clone().requires_grad_(True) for k in names}
    Ds = to_dev(inp["D_skip"]).requires_grad_(True) if skip else None
    y, hT = ssm().selective_scan(*(leaves[k] for k in names), ckpt_interval=16, D_skip=Ds,
                                 delta_softplus=softplus)
    ((y * t["dy"]).sum() + (hT * t["ghT"]).sum()).backward()
    gref = oracle.bwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp["dy"],
                            inp["ghT"], inp.get("D_skip"), delta_softplus=softplus)
    for k, gk in zip(names, GRADS):
        assert_close(to_host(leaves[k].grad), gref[gk], "f32", "grad", gk)
    if skip:
        assert_close(to_host(Ds.grad), gref["gD_skip"], "f32", "grad", "gD_skip")


def test_fused_and_deterministic_workload5_full_size_sampled():
    """Workload 5 at full size with softplus on delta, the skip and fixed-order sums:
    sampled chains against the oracle, gD_skip and gA on sampled channels over all
    batches, gb and gc on one whole batch, and a second run bitwise equal."""
    import torch
    from gpu_util import sample_indices, sub_inputs
    w = gen.workload(5)
    inp = gen.make_inputs(w, raw_delta=True, with_skip=True)
    t = dev_inputs(inp)
    Ds = to_dev(inp["D_skip"])
    K = w.ckpt_interval
    y, hT, ck = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K, D_skip=Ds,
                                   delta_softplus=True)
    g = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck, t["dy"], ckpt_interval=K,
                           D_skip=Ds, delta_softplus=True, deterministic=True)
    g2 = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck, t["dy"], ckpt_interval=K,
                            D_skip=Ds, delta_softplus=True, deterministic=True)
    torch.cuda.synchronize()
    for k in GRADS + ("gD_skip",):
        assert torch.equal(g[k], g2[k]), k
    del g2
    bsel, dsel = sample_indices(w.B, 3, 7), sample_indices(w.D, 8, 8)
    sub = sub_inputs(inp, bsel, dsel)
    ref = oracle.fwd_fused(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], inp["D_skip"][dsel],
                           delta_softplus=True)
    gref = oracle.bwd_fused(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], sub["dy"], None,
                            inp["D_skip"][dsel], delta_softplus=True)
    bi, di = torch.as_tensor(bsel), torch.as_tensor(dsel)
    assert_close(to_host(y[bi][:, :, di]), ref["y"], "bf16", "fwd", "y")
    assert_close(to_host(hT[bi][:, di]), ref["hT"], "bf16", "fwd", "hT")
    for k in ("gx", "gdelta"):
        assert_close(to_host(g[k][bi][:, :, di]), gref[k], "bf16", "grad", k)
    assert_close(to_host(g["gh0"][bi][:, di]), gref["gh0"], "bf16", "grad", "gh0")
    sub = sub_inputs(inp, np.arange(w.B), dsel[:3])
    gref = oracle.bwd_fused(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], sub["dy"], None,
                            inp["D_skip"][dsel[:3]], delta_softplus=True)
    for k in ("gA", "gD_skip"):
        assert_close(to_host(g[k][torch.as_tensor(dsel[:3])]), gref[k], "bf16", "grad", k)
    sub = sub_inputs(inp, np.array([bsel[2]]), np.arange(w.D))
    gref = oracle.bwd_fused(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], sub["dy"], None,
                            inp["D_skip"], delta_softplus=True)
    for k in ("gb", "gc"):
        assert_close(to_host(g[k][int(bsel[2])][None]), gref[k], "bf16", "grad", k)
