"""Seeded random sweep of small problems through every option of the C ABI.

Each case draws a shape (B, T, D), an I/O dtype, a checkpoint interval, a
forward schedule (automatic, one pass in a forced lane layout, or chunked with
a random chunk length), a backward layout (automatic, one or two channels per
lane, chunk-parallel or not), the deterministic flag, the fused softplus and
skip, and whether the backward gets the forward's checkpoints or rebuilds
them; it then compares every output with the float64 oracle at the usual
tolerances. The draws are fixed by the seed, so a failure names a
reproducible case.
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




def draw_case(seed):
    r = np.random.default_rng(1000 + seed)
    case = {
        "B": int(r.integers(1, 4)), "T": int(r.integers(1, 300)), "D": int(r.integers(1, 150)),
        "io": str(r.choice(["f32", "bf16"])), "K": int(r.choice([1, 7, 16, 48, 64, 100, 256])),
        "fwd": str(r.choice(["auto", "2x2", "4x2", "4x1", "chunked"])), "chunk_len": int(r.integers(16, 120)),
        "kd": r.choice([None, 1, 2]), "tpar": r.choice([None, 0, 1]), "det": bool(r.integers(0, 2)),
        "softplus": bool(r.integers(0, 2)), "skip": bool(r.integers(0, 2)), "rebuild": bool(r.integers(0, 4) == 0),
        "h0": bool(r.integers(0, 2)), "ghT": bool(r.integers(0, 2)),
    }
    if case["io"] == "bf16" and case["D"] % 8 and r.integers(0, 2):
        case["D"] += 8 - case["D"] % 8           # both aligned and unaligned rows for bf16
    case["chunk_kd"] = r.choice([None, 1, 2])    # channels per lane of the chunked forward
    case["lookback"] = bool(r.integers(0, 2))    # chunked forward in one launch with look-back
    case["chunk_layout"] = r.choice([None, "2x2"])   # 2 lanes x 2 channels in the chunk passes
    return case


@pytest.mark.parametrize("seed", range(160))
def test_random_case(seed):
    import torch
    import selective_state_space_03_gb300 as ssm
    cs = draw_case(seed)
    w = gen.workload(2, B=cs["B"], T=cs["T"], D=cs["D"], io=cs["io"], h0_std=0.1 if cs["h0"] else 0.0)
    inp = gen.make_inputs(w, seed=seed, with_grad_inputs=True, with_ghT=cs["ghT"], raw_delta=cs["softplus"],
                          with_skip=cs["skip"])
    t = dev_inputs(inp)
    Ds = to_dev(inp["D_skip"]) if cs["skip"] else None
    K = cs["K"]
    layout = cs["fwd"] if cs["fwd"] in ("2x2", "4x2", "4x1") else None
    chunk_len = cs["chunk_len"] if cs["fwd"] == "chunked" else (-1 if layout else 0)
    with forced(SSM_SCAN_FORCE_FWD_LAYOUT=layout, SSM_SCAN_FORCE_CHUNK_KD=cs["chunk_kd"],
                SSM_SCAN_FORCE_CHUNK_LAYOUT=cs["chunk_layout"]):
        y, hT, ck = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K,
                                     chunk_len=chunk_len, D_skip=Ds, delta_softplus=cs["softplus"],
                                     lookback=cs["lookback"])
        if cs["lookback"]:
            ssm.lookback_status()
    with forced(SSM_SCAN_FORCE_BWD_KD=cs["kd"], SSM_SCAN_FORCE_BWD_TPAR=cs["tpar"]):
        g = ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], None if cs["rebuild"] else ck,
                             t["dy"], t.get("ghT"), ckpt_interval=K, D_skip=Ds, delta_softplus=cs["softplus"],
                             deterministic=cs["det"])
    torch.cuda.synchronize()
    ref = oracle.fwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp.get("D_skip"),
                           delta_softplus=cs["softplus"], ckpt_interval=K)
    gref = oracle.bwd_fused(inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"], inp["dy"],
                            inp.get("ghT"), inp.get("D_skip"), delta_softplus=cs["softplus"])
    where = f"case {seed}: {cs}"
    for name, got, want in (("y", y, ref["y"]), ("hT", hT, ref["hT"]), ("ckpt", ck, ref["ckpt"])):
        try:
            assert_close(to_host(got), want, cs["io"], "fwd", name)
        except AssertionError as e:
            raise AssertionError(f"{where}: {e}") from None
    for k in GRADS + (("gD_skip",) if cs["skip"] else ()):
        try:
            assert_close(to_host(g[k]), gref[k], cs["io"], "grad", k)
        except AssertionError as e:
            raise AssertionError(f"{where}: {e}") from None
