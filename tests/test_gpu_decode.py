"""GPU parity of the single-step decode entry (ssm_scan_step) against the oracle.

One step with state h is the scan over T = 1 with h0 = h; T steps applied one
after another in place must give the scan over T steps (outputs per step, the
final state). Tolerances as for the forward: float32 I/O 1e-4, bf16 I/O 1e-2,
as max |got - ref| / (1 + |ref|).
"""
import numpy as np
import pytest

import gen
import oracle
from gpu_util import assert_close, dev_inputs, to_host

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


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("B,D", [(1, 1), (3, 37), (4, 200), (16, 5120)])
def test_one_step_is_the_scan_over_one_step(io, B, D):
    w = gen.workload(2, B=B, T=1, D=D, io=io, h0_std=0.5)
    inp = gen.make_inputs(w, seed=3)
    t = dev_inputs(inp)
    h = t["h0"].clone()
    y = ssm().ssm_scan_step(t["x"][:, 0].contiguous(), t["delta"][:, 0].contiguous(), t["A"],
                            t["b"][:, 0].contiguous(), t["c"][:, 0].contiguous(), h)
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(to_host(y)[:, None, :], ref["y"], io, "fwd", "y")
    assert_close(to_host(h), ref["hT"], io, "fwd", "hT")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_in_place_follow_the_scan(io):
    import torch
    w = gen.workload(2, B=2, T=40, D=72, io=io, h0_std=0.1)
    inp = gen.make_inputs(w, seed=5)
    t = dev_inputs(inp)
    h = t["h0"].clone()
    ys = []
    for k in range(w.T):
        ys.append(ssm().ssm_scan_step(t["x"][:, k].contiguous(), t["delta"][:, k].contiguous(), t["A"],
                                      t["b"][:, k].contiguous(), t["c"][:, k].contiguous(), h))
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    got = np.stack([to_host(v) for v in ys], axis=1)
    assert_close(got, ref["y"], io, "fwd", "y")
    assert_close(to_host(h), ref["hT"], io, "fwd", "hT")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_on_row_views(io):
    # with B = 1, x[:, k] is a view into the (1, T, D) tensor whose address is only element
    # aligned for odd D: the step takes such rows as they are
    import torch
    w = gen.workload(2, B=1, T=9, D=37, io=io, h0_std=0.1)
    inp = gen.make_inputs(w, seed=7)
    t = dev_inputs(inp)
    h = t["h0"].clone()
    ys = []
    for k in range(w.T):
        xk, dk = t["x"][:, k], t["delta"][:, k]
        assert xk.is_contiguous()
        ys.append(ssm().ssm_scan_step(xk, dk, t["A"], t["b"][:, k].contiguous(), t["c"][:, k].contiguous(), h))
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(np.stack([to_host(v) for v in ys], axis=1), ref["y"], io, "fwd", "y")
    assert_close(to_host(h), ref["hT"], io, "fwd", "hT")


def test_step_writes_only_its_outputs():
    import torch
    B, D = 3, 40
    w = gen.workload(2, B=B, T=1, D=D, h0_std=0.1)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    pad, canary = 64, 777.0
    hb = torch.full((B * D * 16 + 2 * pad,), canary, device="cuda:0")
    yb = torch.full((B * D + 2 * pad,), canary, device="cuda:0")
    h = hb[pad:pad + B * D * 16]
    h.copy_(t["h0"].reshape(-1))
    y = yb[pad:pad + B * D]
    ssm().ssm_scan_step(t["x"][:, 0].contiguous(), t["delta"][:, 0].contiguous(), t["A"],
                        t["b"][:, 0].contiguous(), t["c"][:, 0].contiguous(), h.view(B, D, 16), y=y.view(B, D))
    torch.cuda.synchronize()
    for full in (hb, yb):
        assert torch.all(full[:pad] == canary) and torch.all(full[-pad:] == canary)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_step_after_a_kernel_that_writes_its_inputs(io):
    # decode as a model runs it: another kernel (here torch's copy) writes x, delta, b and c into
    # the same buffers right before every step on the same stream; each step must read the new
    # values (a step is launched as a programmatic dependent, so it may be scheduled early, but
    # every load waits for the preceding kernel)
    import torch
    w = gen.workload(5, B=4, T=12, D=1024, io=io, h0_std=0.3)
    inp = gen.make_inputs(w, seed=9, with_grad_inputs=False)
    t = dev_inputs(inp)
    h = t["h0"].clone()
    xs, ds = torch.empty_like(t["x"][:, 0]), torch.empty_like(t["delta"][:, 0])
    bs, cs = torch.empty_like(t["b"][:, 0]), torch.empty_like(t["c"][:, 0])
    ys = []
    for k in range(w.T):
        xs.copy_(t["x"][:, k])
        ds.copy_(t["delta"][:, k])
        bs.copy_(t["b"][:, k])
        cs.copy_(t["c"][:, k])
        y = torch.empty_like(xs)
        ssm().ssm_scan_step(xs, ds, t["A"], bs, cs, h, y=y)
        ys.append(y)
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(np.stack([to_host(v) for v in ys], 1), ref["y"], io, "fwd", "y")
    assert_close(to_host(h), ref["hT"], io, "fwd", "h")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_with_inputs_declared_ready(io):
    # every step's inputs are computed before the first step is launched, so each step may load
    # them while the step before it finishes (SSM_SCAN_STEP_INPUTS_READY); only h waits
    import torch
    w = gen.workload(5, B=3, T=10, D=768, io=io, h0_std=0.3)
    inp = gen.make_inputs(w, seed=11, with_grad_inputs=False)
    t = dev_inputs(inp)
    steps = [tuple(t[k][:, i].contiguous() for k in ("x", "delta", "b", "c")) for i in range(w.T)]
    h = t["h0"].clone()
    ys = [ssm().ssm_scan_step(xk, dk, t["A"], bk, ck, h, inputs_ready=True) for xk, dk, bk, ck in steps]
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(np.stack([to_host(v) for v in ys], 1), ref["y"], io, "fwd", "y")
    assert_close(to_host(h), ref["hT"], io, "fwd", "h")
