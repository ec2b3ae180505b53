"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any launch.

The pointers passed here are fake (never dereferenced): every call below fails
validation, which happens before anything is enqueued.
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from selective_state_space_03_gb300 import build
    build.build()
    import selective_state_space_03_gb300 as ssm
    return ssm.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(ssm_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("ssm_scan_fwd", "ssm_scan_bwd", "ssm_scan_ckpt_bytes", "ssm_scan_fwd_workspace_bytes",
              "ssm_scan_bwd_workspace_bytes", "ssm_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"


def desc(**kw):
    import selective_state_space_03_gb300 as ssm
    base = dict(B=2, T=64, D=32, DS=16, io=0, ckpt_interval=0, chunk_len=0, flags=0)
    base.update(kw)
    return ssm.make_desc(**base)


FAKE = 0x7f0000000000      # 16-byte aligned, never dereferenced


def fwd(L, d, x=FAKE, delta=FAKE, A=FAKE, b=FAKE, c=FAKE, h0=None, y=FAKE, hT=None, ckpt=None, ws=None,
        wsb=0):
    P = ctypes.c_void_p
    return L.ssm_scan_fwd(ctypes.byref(d) if d is not None else None, P(x), P(delta), P(A), P(b), P(c), P(h0),
                          P(y), P(hT), P(ckpt), P(ws), wsb, None)


def bwd(L, d, ckpt=FAKE, ws=None, wsb=0, **kw):
    P = ctypes.c_void_p
    a = dict(x=FAKE, delta=FAKE, A=FAKE, b=FAKE, c=FAKE, h0=None, dy=FAKE, ghT=None, gx=FAKE, gdelta=FAKE,
             gA=FAKE, gb=FAKE, gc=FAKE, gh0=FAKE)
    a.update(kw)
    return L.ssm_scan_bwd(ctypes.byref(d), P(a["x"]), P(a["delta"]), P(a["A"]), P(a["b"]), P(a["c"]), P(a["h0"]),
                          P(ckpt), P(a["dy"]), P(a["ghT"]), P(a["gx"]), P(a["gdelta"]), P(a["gA"]), P(a["gb"]),
                          P(a["gc"]), P(a["gh0"]), P(ws), wsb, None)


def test_status_strings(L):
    for s in range(7):
        assert L.ssm_status_str(s)
    assert b"look-back" in L.ssm_status_str(6)
    assert b"DS" in L.ssm_status_str(2)


def test_invalid_descriptors(L):
    assert fwd(L, None) == 1
    assert fwd(L, desc(B=-1)) == 1
    assert fwd(L, desc(T=-5)) == 1
    assert fwd(L, desc(io=7)) == 1
    assert fwd(L, desc(ckpt_interval=-1)) == 1
    assert fwd(L, desc(B=70000)) == 1
    d = desc()
    d.flags = 16            # the first bit no entry point defines
    assert fwd(L, d) == 1
    assert fwd(L, desc(DS=8)) == 2
    assert fwd(L, desc(DS=32)) == 2
    assert fwd(L, desc(D=(1 << 27) + 1)) == 2        # past the kernels' 32-bit in-tile offsets
    assert fwd(L, desc(B=65536)) == 1
    assert bwd(L, desc(DS=8)) == 2


def test_null_and_misaligned_pointers(L):
    assert fwd(L, desc(), x=None) == 1
    assert fwd(L, desc(), y=None) == 1
    assert fwd(L, desc(), A=None) == 1
    assert fwd(L, desc(), delta=FAKE + 4) == 3
    assert fwd(L, desc(), hT=FAKE + 8) == 3
    assert bwd(L, desc(), gx=None) == 1
    assert bwd(L, desc(), gA=None) == 1
    assert bwd(L, desc(), gb=FAKE + 2) == 3


def test_workspace_checks(L):
    d = desc(T=1024, chunk_len=64)                       # forced chunked schedule needs scratch
    need = L.ssm_scan_fwd_workspace_bytes(ctypes.byref(d))
    nch = 1024 // 64
    assert need >= 2 * (nch - 1) * 32 * 16 * 4
    assert fwd(L, d) == 4
    assert fwd(L, d, ws=FAKE, wsb=need - 1) == 4
    assert L.ssm_scan_fwd_workspace_bytes(ctypes.byref(desc(chunk_len=-1))) == 0
    # backward without checkpoints rebuilds them in the workspace
    db = desc(T=1000, ckpt_interval=100)
    needb = L.ssm_scan_bwd_workspace_bytes(ctypes.byref(db))
    assert needb >= 10 * 2 * 32 * 16 * 4
    assert bwd(L, db, ckpt=None) == 4
    # checkpoints further apart than the backward reads directly are rebuilt too
    dk = desc(T=2048, ckpt_interval=1024)
    assert bwd(L, dk, ckpt=FAKE) == 4


def test_size_queries(L):
    d = desc(B=3, T=1000, D=40, ckpt_interval=256)
    assert L.ssm_scan_ckpt_bytes(ctypes.byref(d)) == 4 * 3 * 40 * 16 * 4
    assert L.ssm_scan_ckpt_bytes(ctypes.byref(desc(ckpt_interval=0))) == 0
    assert L.ssm_scan_fwd_workspace_bytes(ctypes.byref(desc(T=0))) == 0
    assert L.ssm_scan_bwd_workspace_bytes(ctypes.byref(desc(B=0))) == 0
    assert L.ssm_scan_ckpt_bytes(None) == 0


def step(L, d, x=FAKE, delta=FAKE, A=FAKE, b=FAKE, c=FAKE, h=FAKE, y=FAKE):
    P = ctypes.c_void_p
    return L.ssm_scan_step(ctypes.byref(d), P(x), P(delta), P(A), P(b), P(c), P(h), P(y), None)


def test_step_argument_checks(L):
    assert step(L, desc(T=2)) == 1                       # one step per call
    assert step(L, desc(T=1, DS=8)) == 2
    assert step(L, desc(T=1, io=5)) == 1
    assert step(L, desc(T=1), h=None) == 1
    assert step(L, desc(T=1), x=None) == 1
    assert step(L, desc(T=1), h=FAKE + 4) == 3
    assert step(L, desc(T=1), y=FAKE + 2) == 3
    assert step(L, desc(T=1, io=1), x=FAKE + 1) == 3     # bf16 x, y: 2-byte alignment
    assert step(L, desc(T=1), c=FAKE + 8) == 3           # b, c, A, h: 16-byte loads
    assert step(L, desc(T=1, B=0)) == 0                  # nothing to do, nothing launched
    assert step(L, desc(T=1, D=0)) == 0


def test_backward_carry_workspace(L):
    # few chains and ten checkpoint chunks: the chunk-parallel schedule's carries
    d = desc(B=2, T=1000, D=32, ckpt_interval=100)
    carry = L.ssm_scan_bwd_ckpt_workspace_bytes(ctypes.byref(d))
    assert carry >= 10 * 2 * 32 * (16 + 1) * 4
    assert L.ssm_scan_bwd_workspace_bytes(ctypes.byref(d)) >= carry + 10 * 2 * 32 * 16 * 4
    # one chunk: nothing to carry
    assert L.ssm_scan_bwd_ckpt_workspace_bytes(ctypes.byref(desc(B=2, T=100, D=32, ckpt_interval=100))) == 0
    # with checkpoints the carries are optional: a misaligned workspace is still rejected
    assert bwd(L, d, ws=FAKE + 8, wsb=carry) == 3


def test_deterministic_flag_workspace(L):
    # one chunk, many channel blocks: partials of gb/gc per block and of gA per batch
    d = desc(B=2, T=100, D=320, ckpt_interval=100, flags=1)
    need = L.ssm_scan_bwd_ckpt_workspace_bytes(ctypes.byref(d))
    assert need >= 10 * 2 * 100 * 32 * 4 + 2 * 320 * 16 * 4
    assert bwd(L, d) == 4                                # the partials are required
    assert bwd(L, d, ws=FAKE, wsb=need - 1) == 4
    assert L.ssm_scan_bwd_workspace_bytes(ctypes.byref(d)) >= need + 2 * 320 * 16 * 4
    # without the flag the same shape needs no workspace
    assert L.ssm_scan_bwd_ckpt_workspace_bytes(ctypes.byref(desc(B=2, T=100, D=320, ckpt_interval=100))) == 0
    # unknown flag bits are rejected
    assert bwd(L, desc(flags=16)) == 1
    assert step(L, desc(T=1, flags=16)) == 1


def test_fused_entry_point_checks(L):
    P = ctypes.c_void_p
    d = desc(flags=2)                                    # softplus on delta is a valid flag

    def fwdf(D_skip=FAKE, y=FAKE, dd=d):
        return L.ssm_scan_fwd_fused(ctypes.byref(dd), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(D_skip),
                                    P(None), P(y), P(None), P(None), P(None), 0, None)

    def bwdf(D_skip=FAKE, gD=FAKE, dd=d):
        g = [P(FAKE)] * 6
        return L.ssm_scan_bwd_fused(ctypes.byref(dd), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(D_skip),
                                    P(None), P(FAKE), P(FAKE), P(None), *g, P(gD), P(None), 0, None)

    assert fwdf(D_skip=FAKE + 4) == 3
    assert fwdf(y=None) == 1
    assert bwdf(gD=None) == 1                            # the skip weights' gradient is required
    assert bwdf(gD=FAKE + 8) == 3
    assert bwdf(dd=desc(flags=16)) == 1


def test_lookback_flag_workspace_and_status(L):
    # a chunked schedule with SSM_SCAN_LOOKBACK keeps every chunk's map and end state
    d_lb = desc(B=1, T=4096, D=64, chunk_len=256, flags=4)
    d_2p = desc(B=1, T=4096, D=64, chunk_len=256)
    need_lb = L.ssm_scan_fwd_workspace_bytes(ctypes.byref(d_lb))
    need_2p = L.ssm_scan_fwd_workspace_bytes(ctypes.byref(d_2p))
    nch = 4096 // 256
    assert need_lb >= 2 * nch * 64 * 16 * 4 + nch * 64 * 4 + nch * (64 // 8) * 4 + 16
    assert need_lb > need_2p > 0
    assert fwd(L, d_lb) == 4                                      # workspace required
    assert fwd(L, d_lb, ws=FAKE, wsb=need_lb - 1) == 4
    status = L.ssm_scan_fwd_lookback_status
    assert status(ctypes.byref(d_lb), None, 0, None) == 4
    assert status(ctypes.byref(d_lb), ctypes.c_void_p(FAKE), 2 * nch * 64 * 16 * 4, None) == 4
    assert status(ctypes.byref(d_lb), ctypes.c_void_p(FAKE + 8), need_lb, None) == 3
    # nothing waits in the one-pass schedule, or without the flag: no workspace needed
    assert status(ctypes.byref(desc(B=1, T=4096, D=64, chunk_len=-1, flags=4)), None, 0, None) == 0
    assert status(ctypes.byref(d_2p), None, 0, None) == 0
    assert status(ctypes.byref(desc(flags=16)), None, 0, None) == 1
    # the one-pass schedule ignores the flag
    assert L.ssm_scan_fwd_workspace_bytes(ctypes.byref(desc(T=4096, chunk_len=-1, flags=4))) == 0


def test_too_many_chunks_is_unsupported(L):
    # a chunk length that would need more than 65535 chunks is rejected before any launch
    d = desc(T=70000 * 16, chunk_len=16)
    need = L.ssm_scan_fwd_workspace_bytes(ctypes.byref(d))
    assert fwd(L, d, ws=FAKE, wsb=need) == 2


def test_product_path_does_not_import_the_oracle(L):
    # a fresh interpreter: importing the package and loading the library pulls in no oracle module
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); import selective_state_space_03_gb300 as m; m.lib(); "
            "bad = [k for k in sys.modules if k == 'oracle' or k.startswith('oracle.')]; "
            "print('ORACLE' if bad else 'CLEAN')") % ROOT
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert out.stdout.strip().endswith("CLEAN"), out.stdout + out.stderr


def test_missing_library_raises_instead_of_falling_back(monkeypatch):
    import selective_state_space_03_gb300 as m
    monkeypatch.setattr(m, "_libs", {})
    monkeypatch.setattr(m, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libssm_scan.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        m.lib()


def test_schedule_overrides_exist_only_in_the_testing_build(L):
    # the release library compiles none of the SSM_SCAN_FORCE_* / test-only names, so a stray
    # variable in a user's environment cannot change its schedule or results; the testing build
    # (used by the GPU tests that pin every schedule) has them all
    import selective_state_space_03_gb300 as ssm
    names = [b"SSM_SCAN_FORCE_LANES", b"SSM_SCAN_FORCE_FWD_LAYOUT", b"SSM_SCAN_FORCE_CHUNK_KD",
             b"SSM_SCAN_FORCE_CHUNK_LAYOUT", b"SSM_SCAN_FORCE_CARRY_SCAN",
             b"SSM_SCAN_FORCE_BWD_KD", b"SSM_SCAN_FORCE_BWD_TPAR", b"SSM_SCAN_LOOKBACK_POLLS",
             b"SSM_SCAN_TEST_LOOKBACK_DROP"]
    release = open(ssm.LIB_PATH, "rb").read()
    testing = open(ssm.TESTING_LIB_PATH, "rb").read()
    for n in names:
        assert n not in release, n
        assert n in testing, n
    with ssm.testing_library():
        T = ssm.lib()
    assert T is not L and ssm.lib() is L
    for name in declared_functions():
        assert hasattr(T, name), name


# The schedule the library chooses, computed on the host by the testing build for a GB300's 152
# SMs (no device needed): each workload's forward (mode 0 one pass / 2 chunked / 4 chunked in one
# launch, lanes per chain, channels per lane, chunk length, chunks) and backward (channels per
# lane, chunk-parallel, its chunk length), as measured and documented for each shape.
SCHEDULES = [
    # (B, T, D, io, K, chunk_len, flags) -> forward, backward
    ((16, 2048, 5120, 1, 256, 0, 0), (0, 2, 2, 2048, 1), (2, 0, 256)),   # workload 5
    ((8, 4096, 1536, 1, 0, 0, 0), (2, 2, 2, 256, 16), (1, 1, 256)),      # workload 3
    ((1, 4096, 2048, 0, 0, 0, 0), (2, 4, 2, 192, 22), (1, 1, 256)),      # one call of workload 4
    ((8, 1024, 256, 0, 256, 0, 0), (2, 4, 2, 128, 8), (1, 1, 256)),      # workload 2
    ((2, 64, 32, 0, 16, 0, 0), (0, 4, 1, 64, 1), (1, 1, 16)),            # workload 1
    ((8, 4096, 2048, 1, 0, 0, 0), (0, 4, 2, 4096, 1), (1, 1, 256)),      # 16384 chains: one pass
    ((8, 4096, 1536, 1, 0, -1, 0), (0, 4, 2, 4096, 1), (1, 1, 256)),     # one pass asked for
    ((8, 4096, 1536, 1, 0, 100, 0), (2, 2, 2, 100, 41), (1, 1, 256)),    # chunk length given
    ((1, 4096, 2048, 0, 0, 0, 4), (4, 4, 2, 192, 22), (1, 1, 256)),      # look-back flag
]


@pytest.mark.parametrize("case,fwd_plan,bwd_plan", SCHEDULES)
def test_schedule_choices(L, case, fwd_plan, bwd_plan):
    import selective_state_space_03_gb300 as ssm
    B, T, D, io, K, chunk_len, flags = case
    d = ssm.make_desc(B, T, D, 16, io, K, chunk_len, flags)
    out = (ctypes.c_int64 * 8)()
    with ssm.testing_library():
        T_lib = ssm.lib()
        T_lib.ssm_testing_schedule.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        T_lib.ssm_testing_schedule.restype = ctypes.c_int
        assert T_lib.ssm_testing_schedule(ctypes.byref(d), 152, out) == 0
    assert tuple(out[:5]) == fwd_plan, tuple(out[:5])
    assert tuple(out[5:]) == bwd_plan, tuple(out[5:])

