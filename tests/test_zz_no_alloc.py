"""ssm_scan_fwd_noalloc: the forward that allocates nothing.

Some callers cannot allocate device memory while they run (code hosted in
another runtime that owns all device memory, or services that keep cudaMalloc
off the hot path because it synchronises the device and can fail under memory
pressure). For them the library keeps the chunked forward's scratch in a fixed
device array. These tests call that entry point through the C ABI (ctypes)
and compare it with the float64 oracle and with ssm_scan_fwd on the same
inputs and chunk length, on two calls in a row (the second reuses the array
the first one wrote), including the one-chunk case (no scratch) and a problem
that fills the array to just under its size. The file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import gen
from gpu_util import assert_close, dev_inputs, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_03_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    import selective_state_space_03_gb300 as ssm
    lib = ssm.lib()
    lib.ssm_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ssm.ssm_scan_desc)] + [ctypes.c_void_p] * 10
    lib.ssm_scan_fwd_noalloc.restype = ctypes.c_int
    return lib


def call_noalloc(L, t, w, K, chunk_len):
    import torch
    import selective_state_space_03_gb300 as ssm
    B, T, D = w.B, w.T, w.D
    io = ssm.SSM_IO_BF16 if w.io == "bf16" else ssm.SSM_IO_F32
    desc = ssm.make_desc(B, T, D, 16, io, K, chunk_len)
    y = torch.empty_like(t["x"])
    hT = torch.empty((B, D, 16), dtype=torch.float32, device="cuda:0")
    ck = torch.empty((-(-T // K), B, D, 16), dtype=torch.float32, device="cuda:0")
    p = lambda v: None if v is None else ctypes.c_void_p(v.data_ptr())  # noqa: E731
    st = L.ssm_scan_fwd_noalloc(ctypes.byref(desc), p(t["x"]), p(t["delta"]), p(t["A"]), p(t["b"]), p(t["c"]),
                                p(t["h0"]), p(y), p(hT), p(ck), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return y, hT, ck


def check_against_oracle(inp, K, y, hT, ck, io, bsel=None, dsel=None):
    import oracle
    import torch
    from gpu_util import sub_inputs
    if bsel is None:
        sub = inp
        pick = lambda v, chan_axis: v  # noqa: E731
    else:
        sub = sub_inputs(inp, bsel, dsel)
        bi, di = torch.as_tensor(bsel, device=y.device), torch.as_tensor(dsel, device=y.device)
        pick = lambda v, chan_axis: v[bi].index_select(chan_axis, di)  # noqa: E731
    ref = oracle.fwd(sub["x"], sub["delta"], sub["A"], sub["b"], sub["c"], sub["h0"], ckpt_interval=K)
    assert_close(to_host(pick(y, 2)), ref["y"], io, "fwd", "y")
    assert_close(to_host(pick(hT, 1)), ref["hT"], io, "fwd", "hT")
    if ck is None:
        return
    if bsel is None:
        assert_close(to_host(ck), ref["ckpt"], io, "fwd", "ckpt")
    else:
        bi, di = torch.as_tensor(bsel, device=ck.device), torch.as_tensor(dsel, device=ck.device)
        assert_close(to_host(ck[:, bi][:, :, di]), ref["ckpt"], io, "fwd", "ckpt")


def test_noalloc_matches_workspace_forward_two_calls(L):
    # each case twice in a row (the second call reuses the array the first one wrote), against
    # the oracle and against ssm_scan_fwd with the caller's workspace
    import torch
    import selective_state_space_03_gb300 as ssm
    cases = [(gen.workload(2, B=2, T=700, D=96, h0_std=0.1), 128, 100, 0),
             (gen.workload(5, B=3, T=513, D=64), 64, 96, 1),
             # one chunk (chunk_len >= T): the one-pass scan, no scratch
             (gen.workload(2, B=2, T=200, D=40, h0_std=0.1), 50, 256, 2)]
    for w, K, chunk_len, seed in cases:
        inp = gen.make_inputs(w, seed=seed, with_grad_inputs=False)
        t = dev_inputs(inp)
        y0, h0, c0 = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K,
                                      chunk_len=chunk_len)
        for _ in range(2):
            y1, h1, c1 = call_noalloc(L, t, w, K, chunk_len)
            torch.cuda.synchronize()
            check_against_oracle(inp, K, y1, h1, c1, w.io)
            assert_close(to_host(y1), to_host(y0), w.io, "fwd", "y")
            assert_close(to_host(h1), to_host(h0), w.io, "fwd", "hT")
            assert_close(to_host(c1), to_host(c0), w.io, "fwd", "ckpt")


def test_noalloc_at_its_scratch_limit(L):
    # B = 1, D = 4096, 31 chunks of 64 steps: 30 carries take 30*4096*64 + 30*4096*4 = 8,355,840
    # bytes, just under the 8 MiB array; sampled channels against the oracle, all of them
    # against ssm_scan_fwd
    import torch
    import selective_state_space_03_gb300 as ssm
    from gpu_util import sample_indices
    w = gen.workload(2, B=1, T=31 * 64, D=4096, h0_std=0.1)
    assert 30 * 4096 * 68 <= (8 << 20) < 31 * 4096 * 68
    inp = gen.make_inputs(w, seed=4, with_grad_inputs=False)
    t = dev_inputs(inp)
    y0, h0, c0 = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=256,
                                  chunk_len=64)
    y1, h1, c1 = call_noalloc(L, t, w, 256, 64)
    torch.cuda.synchronize()
    check_against_oracle(inp, 256, y1, h1, c1, w.io, bsel=np.array([0]), dsel=sample_indices(w.D, 24, 5))
    assert_close(to_host(y1), to_host(y0), w.io, "fwd", "y")
    assert_close(to_host(h1), to_host(h0), w.io, "fwd", "hT")
    # one chunk more does not fit
    desc = ssm.make_desc(1, 32 * 64, 4096, 16, ssm.SSM_IO_F32, 0, 64)
    fake = ctypes.c_void_p(0x7F0000000000)
    st = L.ssm_scan_fwd_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, None, fake, None, None, None)
    assert st == 4


def test_noalloc_library_chunks_grow_to_fit_its_scratch(L):
    # B = 2, D = 4096, T = 16384 with the chunk length left to the library: its 256-step chunks
    # would need 63 carries of 8192 chains (35 MB) and 512-step ones 31 (17.3 MB), so it takes 16
    # chunks of 1024 (8,355,840 bytes); sampled channels against the oracle
    import torch
    import selective_state_space_03_gb300 as ssm
    from gpu_util import sample_indices
    w = gen.workload(5, B=2, T=16384, D=4096)
    assert 63 * 8192 * 68 > 31 * 8192 * 68 > (8 << 20) >= 15 * 8192 * 68
    inp = gen.make_inputs(w, seed=7, with_grad_inputs=False)
    t = dev_inputs(inp)
    y, hT, _ = ssm.ssm_scan_fwd_noalloc(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"])
    torch.cuda.synchronize()
    check_against_oracle(inp, 0, y, hT, None, w.io, bsel=np.array([0, 1]), dsel=sample_indices(w.D, 16, 8))


def test_noalloc_rejects_problems_beyond_its_scratch(L):
    import selective_state_space_03_gb300 as ssm
    fake = ctypes.c_void_p(0x7F0000000000)      # aligned, never dereferenced: the call fails its size check
    # 2 * 99 carries of 8192 channels: 2*99*8192*68 bytes > the fixed scratch
    desc = ssm.make_desc(2, 100 * 64, 8192, 16, ssm.SSM_IO_F32, 0, 64)
    st = L.ssm_scan_fwd_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, None, fake, None, None, None)
    assert st == 4
    assert np.int64(2 * 99 * 8192 * 68) > (8 << 20)


def test_noalloc_with_softplus_on_delta(L):
    import torch
    import oracle
    import selective_state_space_03_gb300 as ssm
    w = gen.workload(2, B=2, T=300, D=48, h0_std=0.1)
    inp = gen.make_inputs(w, seed=6, with_grad_inputs=False, raw_delta=True)
    t = dev_inputs(inp)
    y, hT, _ = ssm.ssm_scan_fwd_noalloc(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], chunk_len=64,
                                        delta_softplus=True)
    torch.cuda.synchronize()
    ref = oracle.fwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], delta_softplus=True)
    assert_close(to_host(y), ref["y"], "f32", "fwd", "y")
    assert_close(to_host(hT), ref["hT"], "f32", "fwd", "hT")
