"""GPU parity of the one-launch chunked forward (SSM_SCAN_LOOKBACK, decoupled
look-back) against the oracle, and its bounded waits.

The schedule computes the same function as the one-pass scan (the chunk maps
compose exactly in real arithmetic), so every case compares y, hT and the
checkpoints with the float64 oracle at the forward tolerances (float32 I/O
1e-4, bf16 I/O 1e-2, as max |got - ref| / (1 + |ref|)). The failure test makes
chunk 0 publish nothing (a testing aid of the library), so the waits of chunk
1 run out after a short poll budget: the launch must still finish, the status
query must report SSM_ERR_TIMEOUT, and the next call must work.
"""

import numpy as np
import pytest

import gen
import oracle
from gpu_util import assert_close, dev_inputs, to_dev, to_host, forced

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




def lookback_case(w, K, chunk_len, chunk_kd=None, softplus=False, skip=False, seed=0):
    import torch
    inp = gen.make_inputs(w, seed=seed, raw_delta=softplus, with_skip=skip)
    t = dev_inputs(inp)
    Ds = to_dev(inp["D_skip"]) if skip else None
    with forced(SSM_SCAN_FORCE_CHUNK_KD=chunk_kd):
        y, hT, ck = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K,
                                       chunk_len=chunk_len, D_skip=Ds, delta_softplus=softplus, lookback=True)
    ssm().lookback_status()
    torch.cuda.synchronize()
    ref = oracle.fwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp.get("D_skip"),
                           delta_softplus=softplus, ckpt_interval=K)
    assert_close(to_host(y), ref["y"], w.io, "fwd", "y")
    assert_close(to_host(hT), ref["hT"], w.io, "fwd", "hT")
    if K > 0:
        assert_close(to_host(ck), ref["ckpt"], w.io, "fwd", "ckpt")
    return y, hT


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk_kd", [1, 2])
@pytest.mark.parametrize("chunk_len", [32, 50, 129])
def test_lookback_ragged_chunks(io, chunk_kd, chunk_len):
    lookback_case(gen.workload(2, B=2, T=230, D=48, io=io, h0_std=0.1), K=64, chunk_len=chunk_len,
                  chunk_kd=chunk_kd)


@pytest.mark.parametrize("chunk_kd", [1, 2])
def test_lookback_long_chains_of_chunks(chunk_kd):
    # 125 chunks: a chunk may fold many predecessors' maps before it reaches an end state
    lookback_case(gen.workload(2, B=3, T=2000, D=40, h0_std=0.1), K=0, chunk_len=16, chunk_kd=chunk_kd)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_lookback_unaligned_channels(io):
    D = 37 if io == "f32" else 20
    lookback_case(gen.workload(2, B=3, T=300, D=D, io=io, h0_std=0.1), K=32, chunk_len=64, chunk_kd=2)
    lookback_case(gen.workload(2, B=3, T=300, D=D, io=io, h0_std=0.1), K=48, chunk_len=50, chunk_kd=1)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("softplus,skip", [(True, True), (False, True), (True, False)])
def test_lookback_fused_softplus_and_skip(io, softplus, skip):
    lookback_case(gen.workload(2, B=2, T=230, D=40, io=io, h0_std=0.1), K=50, chunk_len=50, chunk_kd=2,
                  softplus=softplus, skip=skip)


def test_lookback_automatic_schedule_matches_two_launches():
    """Workload 2's forward with the library's chunk schedule: one launch with look-back and
    the two-launch schedule agree with each other as with the oracle."""
    import torch
    w = gen.workload(2)
    y1, h1 = lookback_case(w, K=256, chunk_len=0)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    y2, h2, _ = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=256)
    torch.cuda.synchronize()
    assert_close(to_host(y1), to_host(y2).astype(np.float64), "f32", "fwd", "y")
    assert_close(to_host(h1), to_host(h2).astype(np.float64), "f32", "fwd", "hT")


def test_lookback_timeout_is_reported_and_the_context_survives():
    import torch
    m = ssm()
    w = gen.workload(2, B=2, T=256, D=32, h0_std=0.1)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    with forced(SSM_SCAN_TEST_LOOKBACK_DROP=1, SSM_SCAN_LOOKBACK_POLLS=2000):
        m.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], chunk_len=64, lookback=True)
    with pytest.raises(m.SSMError) as e:
        m.lookback_status()
    assert e.value.status == m.SSM_ERR_TIMEOUT
    # the GPU context is still good: the same call without the testing aid is correct
    lookback_case(w, K=0, chunk_len=64)
    torch.cuda.synchronize()


def test_release_library_ignores_the_testing_variables():
    # the same variables outside testing_library(): the release build has no such overrides,
    # so the look-back call completes normally and matches the oracle
    import os
    m = ssm()
    w = gen.workload(2, B=2, T=256, D=32, h0_std=0.1)
    inp = gen.make_inputs(w, with_grad_inputs=False)
    t = dev_inputs(inp)
    os.environ["SSM_SCAN_TEST_LOOKBACK_DROP"], os.environ["SSM_SCAN_LOOKBACK_POLLS"] = "1", "2000"
    try:
        y, hT, _ = m.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], chunk_len=64,
                                  lookback=True)
        m.lookback_status()                # raises on a timeout
    finally:
        del os.environ["SSM_SCAN_TEST_LOOKBACK_DROP"], os.environ["SSM_SCAN_LOOKBACK_POLLS"]
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(to_host(y), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(hT), ref["hT"], "f32", "fwd", "hT")


def test_lookback_grid_beyond_resident_ctas():
    # 256 chunks x 8 batches x 32 channel blocks = 65536 CTAs, far more than are resident at once:
    # a CTA only waits for CTAs that took an earlier ticket, so the launch still moves
    import torch
    from gpu_util import sample_indices, sub_inputs
    w = gen.workload(2, B=8, T=16384, D=512, h0_std=0.1)
    inp = gen.make_inputs(w, with_grad_inputs=False)
    t = dev_inputs(inp)
    y, hT, _ = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], chunk_len=64,
                                  lookback=True)
    ssm().lookback_status()
    bsel, dsel = sample_indices(w.B, 3, 1), sample_indices(w.D, 6, 2)
    sub = sub_inputs(inp, bsel, dsel)
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"])
    bi, di = torch.as_tensor(bsel), torch.as_tensor(dsel)
    assert_close(to_host(y[bi][:, :, di]), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(hT[bi][:, di]), ref["hT"], "f32", "fwd", "hT")


def test_lookback_workload4_full_size_chained_sampled():
    import torch
    from gpu_util import sample_indices, sub_inputs
    w = gen.workload(4)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    L = w.chunk_T
    h = t["h0"]
    y = torch.empty_like(t["x"])
    for k in range(w.T // L):
        sl = slice(L * k, L * (k + 1))
        yk, h, _ = ssm().ssm_scan_fwd(t["x"][:, sl].contiguous(), t["delta"][:, sl].contiguous(), t["A"],
                                      t["b"][:, sl].contiguous(), t["c"][:, sl].contiguous(), h, lookback=True)
        ssm().lookback_status()
        y[:, sl] = yk
    torch.cuda.synchronize()
    dsel = sample_indices(w.D, 12, 5)
    sub = sub_inputs(inp, np.array([0]), dsel)
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"])
    assert_close(to_host(y[:, :, torch.as_tensor(dsel)]), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(h[:, torch.as_tensor(dsel)]), ref["hT"], "f32", "fwd", "hT")
