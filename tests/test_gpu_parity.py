"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small and medium cases compare every output element; the full benchmark
workloads compare sampled (b, d) chains (y, hT, gx, gdelta, gh0), sampled
channels over all batches (gA), one whole batch over all channels (gb, gc),
and check the Euler identities of the loss on the full outputs.
Tolerances: float32 I/O 1e-4 (y, hT) and 1e-3 (gradients); bf16 I/O 1e-2;
all as max |got - ref| / (1 + |ref|).
"""

import numpy as np
import pytest

import gen
import oracle
from gpu_util import GRADS, assert_close, dev_inputs, sample_indices, sub_inputs, to_dev, to_host, forced

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




def run_case(w, K, chunk_len=0, seed=0, ghT=False, bwd=True, lanes=None, ckpt_to_bwd=True, bwd_kd=None,
             bwd_tpar=None, bwd_workspace=None, deterministic=False, fwd_layout=None, chunk_kd=None,
             chunk_layout=None):
    import torch
    inp = gen.make_inputs(w, seed=seed, with_grad_inputs=bwd, with_ghT=ghT)
    t = dev_inputs(inp)
    with forced(SSM_SCAN_FORCE_LANES=lanes, SSM_SCAN_FORCE_FWD_LAYOUT=fwd_layout, SSM_SCAN_FORCE_CHUNK_KD=chunk_kd,
                SSM_SCAN_FORCE_CHUNK_LAYOUT=chunk_layout):
        y, hT, ckpt = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K,
                                         chunk_len=chunk_len)
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], ckpt_interval=K)
    assert_close(to_host(y), ref["y"], w.io, "fwd", "y")
    assert_close(to_host(hT), ref["hT"], w.io, "fwd", "hT")
    if K > 0:
        assert_close(to_host(ckpt), ref["ckpt"], w.io, "fwd", "ckpt")
    if not bwd:
        return
    with forced(SSM_SCAN_FORCE_BWD_KD=bwd_kd, SSM_SCAN_FORCE_BWD_TPAR=bwd_tpar):
        g = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"],
                               ckpt if ckpt_to_bwd else None, t["dy"], t["ghT"], ckpt_interval=K,
                               workspace=bwd_workspace, deterministic=deterministic)
    torch.cuda.synchronize()
    gref = oracle.bwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp["dy"], inp.get("ghT"))
    for k in GRADS:
        assert_close(to_host(g[k]), gref[k], w.io, "grad", k)


# ---------------------------------------------------------------- whole-output cases

def test_workload1_fwd_bwd():
    run_case(gen.workload(1), K=16, ghT=True)


def test_workload1_chunked_schedule():
    run_case(gen.workload(1), K=16, chunk_len=16, bwd=False)


def test_workload2_full_fwd_bwd():
    run_case(gen.workload(2), K=256)


def test_workload2_one_pass_schedule():
    run_case(gen.workload(2), K=256, chunk_len=-1, bwd=False)


def test_workload3_shape_reduced_bf16():
    run_case(gen.workload(3, B=2, T=300, D=200), K=64)
    run_case(gen.workload(3, B=2, T=300, D=200), K=64, fwd_layout="4x2", bwd=False)


def test_workload5_shape_reduced_bf16():
    run_case(gen.workload(5, B=2, T=600, D=264), K=256, ghT=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["2x2", "4x2", "4x1"])
def test_forward_lane_layouts(io, layout):
    # D = 72 leaves a partial last CTA in every layout (32, 16, 8 channels per warp)
    run_case(gen.workload(1, B=3, T=100, D=72, io=io), K=32, chunk_len=-1, fwd_layout=layout, bwd=False)
    run_case(gen.workload(1, B=2, T=37, D=50, io=io), K=16, chunk_len=-1, fwd_layout=layout, bwd=False)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("bwd_kd", [1, 2])
def test_backward_channels_per_lane(io, bwd_kd):
    # both backward layouts on several CTAs with a partial last one (D = 200: 3 x 64 + 8)
    run_case(gen.workload(2, B=3, T=300, D=200, io=io, h0_std=0.1), K=64, ghT=True, bwd_kd=bwd_kd)


def test_workload2_two_channel_backward():
    run_case(gen.workload(2), K=256, bwd_kd=2)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,K", [(230, 50), (512, 256), (33, 16)])
def test_chunk_parallel_backward(io, T, K):
    # one CTA per (channel block, batch, chunk), adjoint entering each chunk from the carries
    run_case(gen.workload(2, B=2, T=T, D=40, io=io, h0_std=0.1), K=K, ghT=True, bwd_tpar=1)


def test_chunk_parallel_backward_rebuild_and_fallback():
    import torch
    w = gen.workload(2, B=3, T=300, D=72, h0_std=0.1)
    # checkpoints rebuilt in the workspace behind the carries
    run_case(w, K=64, ghT=True, ckpt_to_bwd=False, bwd_tpar=1)
    # no room for the carries: the same call sweeps each chain in one CTA
    run_case(w, K=64, ghT=True, bwd_tpar=1, bwd_workspace=torch.empty(0, dtype=torch.uint8, device="cuda:0"))


def test_workload2_sequential_backward():
    run_case(gen.workload(2), K=256, bwd_tpar=0)


@pytest.mark.parametrize("layout", ["kd1", "kd2", "chunk_parallel"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_deterministic_backward(layout, io):
    import torch
    env = {"kd1": dict(bwd_kd=1, bwd_tpar=0), "kd2": dict(bwd_kd=2, bwd_tpar=0),
           "chunk_parallel": dict(bwd_kd=1, bwd_tpar=1)}[layout]
    w = gen.workload(2, B=3, T=300, D=680, io=io, h0_std=0.1)    # 11-22 channel blocks sum into gb, gc
    # against the oracle
    run_case(w, K=64, ghT=True, deterministic=True, **env)
    # bitwise the same on every run
    inp = gen.make_inputs(w, seed=1, with_grad_inputs=True, with_ghT=True)
    t = dev_inputs(inp)
    _, _, ck = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=64)
    runs = []
    with forced(SSM_SCAN_FORCE_BWD_KD=env["bwd_kd"], SSM_SCAN_FORCE_BWD_TPAR=env["bwd_tpar"]):
        for _ in range(3):
            runs.append(ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck, t["dy"],
                                           t["ghT"], ckpt_interval=64, deterministic=True))
    torch.cuda.synchronize()
    for k in GRADS:
        assert torch.equal(runs[0][k], runs[1][k]) and torch.equal(runs[0][k], runs[2][k]), k


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("bwd_kd", [1, 2])
def test_unaligned_channel_count(io, bwd_kd):
    # D * sizeof(io) not a multiple of 16 bytes: element-wise staging path
    D = 37 if io == "f32" else 20
    run_case(gen.workload(2, B=2, T=77, D=D, io=io, h0_std=0.1), K=24, ghT=True, bwd_kd=bwd_kd)
    if bwd_kd == 2:
        run_case(gen.workload(2, B=2, T=77, D=D, io=io, h0_std=0.1), K=24, chunk_len=-1, fwd_layout="4x2",
                 bwd=False)
        return
    run_case(gen.workload(2, B=2, T=77, D=D, io=io, h0_std=0.1), K=24, chunk_len=20, bwd=False)
    run_case(gen.workload(2, B=2, T=77, D=D, io=io, h0_std=0.1), K=24, chunk_len=-1, lanes=2, bwd=False)


@pytest.mark.parametrize("T,K", [(1, 1), (15, 16), (33, 16), (20, 64), (230, 50), (255, 256), (257, 256)])
@pytest.mark.parametrize("bwd_kd", [1, 2])
def test_ragged_lengths_and_intervals(T, K, bwd_kd):
    run_case(gen.workload(2, B=2, T=T, D=40, h0_std=0.1), K=K, ghT=True, bwd_kd=bwd_kd)


CHUNK_LAYOUTS = ["4x1", "4x2", "2x2"]      # lanes per chain x channels per lane of the chunk passes


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk_layout", CHUNK_LAYOUTS)
@pytest.mark.parametrize("chunk_len", [32, 50, 129])
def test_chunked_ragged_chunks(chunk_len, chunk_layout, io):
    run_case(gen.workload(2, B=2, T=230, D=48, io=io, h0_std=0.1), K=64, chunk_len=chunk_len, bwd=False,
             chunk_layout=chunk_layout)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk_layout", ["4x2", "2x2"])
def test_chunked_two_channels_per_lane_unaligned(io, chunk_layout):
    # an odd channel count leaves the last lane's second channel empty; bf16 rows of 20
    # channels are not whole 16-byte chunks
    D = 37 if io == "f32" else 20
    run_case(gen.workload(2, B=3, T=300, D=D, io=io, h0_std=0.1), K=32, chunk_len=64, bwd=False,
             chunk_layout=chunk_layout)


@pytest.mark.parametrize("T,chunk_len,scan", [(230, 64, 1), (700, 16, None), (700, 16, 0), (1000, 16, 1),
                                              (16 * 40 + 5, 16, None),
                                              # 32 and 64 carries: one and two per lane of the scan
                                              (33 * 16, 16, 1), (65 * 16, 16, 1)])
@pytest.mark.parametrize("chunk_layout", CHUNK_LAYOUTS)
def test_chunked_carry_scan(T, chunk_len, scan, chunk_layout):
    # the middle pass that folds the chunk carries once per chain (on by default above 48
    # carries; forced on or off here) against the oracle: y, hT and checkpoints, ragged last chunk
    w = gen.workload(2, B=2, T=T, D=40, h0_std=0.1, io="bf16" if chunk_layout == "2x2" else "f32")
    with forced(SSM_SCAN_FORCE_CARRY_SCAN=scan):
        run_case(w, K=32, chunk_len=chunk_len, bwd=False, chunk_layout=chunk_layout)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_chunked_layout_chosen_by_the_library(io):
    # 12288 chains over 4096 steps: the library picks 8 chunks of 512 steps with 2 lanes per chain
    # (the workload-3 shape); sampled chains against the oracle, all of them against the one-pass
    # scan
    import torch
    w = gen.workload(3, io=io)
    inp = gen.make_inputs(w, seed=3, with_grad_inputs=False)
    t = dev_inputs(inp)
    y, hT, _ = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"])
    y1, hT1, _ = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], chunk_len=-1)
    torch.cuda.synchronize()
    bsel, dsel = np.array([0, 7]), sample_indices(w.D, 12, 9)
    sub = sub_inputs(inp, bsel, dsel)
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"])
    bi, di = torch.as_tensor(bsel, device=y.device), torch.as_tensor(dsel, device=y.device)
    assert_close(to_host(y[bi][:, :, di]), ref["y"], w.io, "fwd", "y")
    assert_close(to_host(hT[bi][:, di]), ref["hT"], w.io, "fwd", "hT")
    assert_close(to_host(y), to_host(y1), w.io, "fwd", "y")
    assert_close(to_host(hT), to_host(hT1), w.io, "fwd", "hT")


def test_backward_rebuilds_checkpoints():
    # no checkpoints passed: the backward rebuilds them in its workspace
    run_case(gen.workload(2, B=2, T=300, D=40, h0_std=0.1), K=64, ghT=True, ckpt_to_bwd=False)
    run_case(gen.workload(2, B=2, T=300, D=40, h0_std=0.1), K=64, ghT=True, ckpt_to_bwd=False, bwd_kd=2)
    # interval longer than the backward reads directly
    run_case(gen.workload(2, B=2, T=700, D=40, h0_std=0.1), K=512, ghT=True)


def test_chained_calls_match_one_long_scan():
    import torch
    w = gen.workload(4, T=4 * 200, D=96)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    h = t["h0"]
    ys = []
    for k in range(4):
        sl = slice(200 * k, 200 * (k + 1))
        y, h, _ = ssm().ssm_scan_fwd(t["x"][:, sl].contiguous(), t["delta"][:, sl].contiguous(), t["A"],
                                     t["b"][:, sl].contiguous(), t["c"][:, sl].contiguous(), h)
        ys.append(y)
    torch.cuda.synchronize()
    ref = oracle.fwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"])
    assert_close(to_host(torch.cat(ys, 1)), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(h), ref["hT"], "f32", "fwd", "hT")


def test_empty_sizes():
    import torch
    m = ssm()
    dev = "cuda:0"
    for B, T, D in ((2, 0, 8), (0, 5, 8), (2, 5, 0)):
        x = torch.zeros(B, T, D, device=dev)
        A = -torch.ones(D, 16, device=dev)
        bc = torch.zeros(B, T, 16, device=dev)
        h0 = torch.randn(B, D, 16, device=dev)
        y, hT, _ = m.ssm_scan_fwd(x, x, A, bc, bc, h0)
        ghT = torch.randn(B, D, 16, device=dev)
        g = m.ssm_scan_bwd(x, x, A, bc, bc, h0, None, x, ghT)
        torch.cuda.synchronize()
        assert torch.equal(hT, h0)
        assert torch.equal(g["gh0"], ghT)
        assert torch.all(g["gA"] == 0)
        assert torch.all(g["gb"] == 0) and torch.all(g["gc"] == 0)


@pytest.mark.parametrize("bwd_kd", [1, 2])
def test_outputs_stay_in_bounds_and_forward_is_deterministic(bwd_kd):
    import torch
    m = ssm()
    w = gen.workload(2, B=2, T=70, D=36, h0_std=0.1)
    inp = gen.make_inputs(w, with_grad_inputs=True, with_ghT=True)
    t = dev_inputs(inp)
    B, T, D = 2, 70, 36
    pad = 64
    canary = 12345.0

    def guarded(n):
        buf = torch.full((n + 2 * pad,), canary, device="cuda:0")
        return buf, buf[pad:pad + n]

    yb, y = guarded(B * T * D)
    hb, hT = guarded(B * D * 16)
    cb, ck = guarded(3 * B * D * 16)
    m.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=32,
                   y=y.view(B, T, D), hT=hT.view(B, D, 16), ckpt=ck.view(3, B, D, 16))
    grads = {}
    bufs = []
    for k, n in (("gx", B * T * D), ("gdelta", B * T * D), ("gA", D * 16), ("gb", B * T * 16),
                 ("gc", B * T * 16), ("gh0", B * D * 16)):
        full, inner = guarded(n)
        bufs.append(full)
        grads[k] = inner
    shapes = {"gx": (B, T, D), "gdelta": (B, T, D), "gA": (D, 16), "gb": (B, T, 16), "gc": (B, T, 16),
              "gh0": (B, D, 16)}
    with forced(SSM_SCAN_FORCE_BWD_KD=bwd_kd):
        m.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck.view(3, B, D, 16), t["dy"],
                       t["ghT"], ckpt_interval=32, grads={k: v.view(shapes[k]) for k, v in grads.items()})
    torch.cuda.synchronize()
    for full in [yb, hb, cb] + bufs:
        assert torch.all(full[:pad] == canary) and torch.all(full[-pad:] == canary)
    y2, _, _ = m.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=32)
    torch.cuda.synchronize()
    assert torch.equal(y2, y.view(B, T, D))


def test_autograd_wrapper():
    import torch
    w = gen.workload(2, B=2, T=64, D=16, h0_std=0.1)
    inp = gen.make_inputs(w, with_grad_inputs=True, with_ghT=True)
    t = dev_inputs(inp)
    leaves = {k: t[k].clone().requires_grad_(True) for k in ("x", "delta", "A", "b", "c", "h0")}
    y, hT = ssm().selective_scan(leaves["x"], leaves["delta"], leaves["A"], leaves["b"], leaves["c"],
                                 leaves["h0"], ckpt_interval=16)
    ((y * t["dy"]).sum() + (hT * t["ghT"]).sum()).backward()
    gref = oracle.bwd(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp["dy"], inp["ghT"])
    for k, gk in zip(("x", "delta", "A", "b", "c", "h0"), GRADS):
        assert_close(to_host(leaves[k].grad), gref[gk], "f32", "grad", gk)


# ---------------------------------------------------------------- full benchmark workloads, sampled

def test_workload3_full_size_sampled():
    import torch
    w = gen.workload(3)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    y, hT, _ = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"])
    torch.cuda.synchronize()
    bsel = sample_indices(w.B, 2, 1)
    dsel = sample_indices(w.D, 24, 2)
    sub = sub_inputs(inp, bsel, dsel)
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"])
    ys = to_host(y[torch.as_tensor(bsel)][:, :, torch.as_tensor(dsel)])
    assert_close(ys, ref["y"], "bf16", "fwd", "y")
    assert_close(to_host(hT[torch.as_tensor(bsel)][:, torch.as_tensor(dsel)]), ref["hT"], "bf16", "fwd", "hT")


def test_workload4_full_size_chained_sampled():
    import torch
    w = gen.workload(4)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    L = w.chunk_T
    h = t["h0"]
    y = torch.empty_like(t["x"])
    for k in range(w.T // L):
        sl = slice(L * k, L * (k + 1))
        yk, h, _ = ssm().ssm_scan_fwd(t["x"][:, sl].contiguous(), t["delta"][:, sl].contiguous(), t["A"],
                                      t["b"][:, sl].contiguous(), t["c"][:, sl].contiguous(), h)
        y[:, sl] = yk
    torch.cuda.synchronize()
    dsel = sample_indices(w.D, 12, 3)
    sub = sub_inputs(inp, np.array([0]), dsel)
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"])
    assert_close(to_host(y[:, :, torch.as_tensor(dsel)]), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(h[:, torch.as_tensor(dsel)]), ref["hT"], "f32", "fwd", "hT")


def test_workload5_full_size_sampled_and_identities():
    import torch
    w = gen.workload(5)
    inp = gen.make_inputs(w)
    t = dev_inputs(inp)
    K = w.ckpt_interval
    y, hT, ckpt = ssm().ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K)
    g = ssm().ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt, t["dy"], None,
                           ckpt_interval=K)
    torch.cuda.synchronize()
    # chains: y, hT, gx, gdelta, gh0
    bsel = sample_indices(w.B, 3, 4)
    dsel = sample_indices(w.D, 10, 5)
    sub = sub_inputs(inp, bsel, dsel)
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"])
    gref = oracle.bwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], sub["dy"])
    bi, di = torch.as_tensor(bsel), torch.as_tensor(dsel)
    assert_close(to_host(y[bi][:, :, di]), ref["y"], "bf16", "fwd", "y")
    assert_close(to_host(hT[bi][:, di]), ref["hT"], "bf16", "fwd", "hT")
    for k in ("gx", "gdelta"):
        assert_close(to_host(g[k][bi][:, :, di]), gref[k], "bf16", "grad", k)
    assert_close(to_host(g["gh0"][bi][:, di]), gref["gh0"], "bf16", "grad", "gh0")
    # gA: all batches, sampled channels
    sub = sub_inputs(inp, np.arange(w.B), dsel[:4])
    gref = oracle.bwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], sub["dy"])
    assert_close(to_host(g["gA"][torch.as_tensor(dsel[:4])]), gref["gA"], "bf16", "grad", "gA")
    # gb, gc: one batch, all channels
    sub = sub_inputs(inp, np.array([bsel[1]]), np.arange(w.D))
    gref = oracle.bwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], sub["dy"])
    for k in ("gb", "gc"):
        assert_close(to_host(g[k][int(bsel[1])][None]), gref[k], "bf16", "grad", k)
    # Euler identities on the full GPU outputs (float64 sums on the host):
    # I1 sum_s c gc = sum_d dy y per (b, t); I4 sum delta gdelta = sum_s A gA + sum x gx per d
    c64, dy64 = oracle.to_f64(inp["c"]), oracle.to_f64(inp["dy"])
    y64 = to_host(y)
    i1l = np.einsum("bts,bts->bt", c64, to_host(g["gc"]))
    i1r = np.einsum("btd,btd->bt", dy64, y64)
    scale = np.einsum("btd,btd->bt", np.abs(dy64), np.abs(y64)) + 1.0
    assert np.max(np.abs(i1l - i1r) / scale) < 1e-2
    del y64
    x64, d64 = oracle.to_f64(inp["x"]), oracle.to_f64(inp["delta"])
    gx, gd = to_host(g["gx"]), to_host(g["gdelta"])
    i4l = np.einsum("btd,btd->d", d64, gd)
    i4r = np.einsum("ds,ds->d", inp["A"].astype(np.float64), to_host(g["gA"])) + np.einsum("btd,btd->d", x64, gx)
    scale4 = np.einsum("btd,btd->d", np.abs(d64), np.abs(gd)) + 1.0
    assert np.max(np.abs(i4l - i4r) / scale4) < 1e-3
