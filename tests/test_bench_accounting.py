"""The byte and work accounting behind the bench's roofline numbers (CPU only).

The HBM fractions divide compulsory bytes by the measured copy bandwidth, and the
compute fractions divide per-element work by the unit peaks; these checks restate
the compulsory bytes of workload 5 term by term from the tensors the step must read
and write once (the layouts in include/ssm_scan.h), and check the config both arms
print.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import gen  # noqa: E402


def test_compulsory_bytes_of_workload5():
    w = gen.workload(5)
    B, T, D, DS = w.B, w.T, w.D, w.DS
    s = 2                                   # bf16 I/O
    state = B * D * DS * 4                  # one float32 state
    nck = -(-T // w.ckpt_interval)          # checkpoint slots
    fwd = (B * T * D * s * 2                # x, delta read
           + B * T * D * s                  # y written
           + B * T * DS * s * 2             # b, c read
           + D * DS * 4                     # A read
           + state                          # hT written (h0 = 0 is not read)
           + nck * state)                   # checkpoints written
    bwd = (B * T * D * s * 3                # x, delta, dy read
           + B * T * D * 4 * 2              # gx, gdelta written (float32)
           + B * T * DS * s * 2             # b, c read
           + B * T * DS * 4 * 2             # gb, gc written
           + D * DS * 4 * 2                 # A read, gA written
           + nck * state                    # checkpoints read
           + state)                         # gh0 written
    assert bench.compulsory_bytes(w, "fwd") == fwd
    assert bench.compulsory_bytes(w, "bwd") == bwd
    # per element (b, t, d, s): 0.39 B forward and 0.90 B backward, as the roofline analysis uses
    el = B * T * D * DS
    assert abs(fwd / el - 0.393) < 0.001
    assert abs(bwd / el - 0.895) < 0.001


def test_config_names_the_workload_by_its_shape():
    w = gen.workload(5)
    c = bench.workload_config(w, 1)
    assert c["workload"] == w.name == "fwdbwd_bf16_B16_T2048_D5120"
    assert (c["B"], c["T"], c["D"], c["DS"], c["io"], c["ckpt_interval"]) == (16, 2048, 5120, 16, "bf16", 256)
    assert c["parallelism"] == "replicas x1"
    assert "model" not in c


def test_work_constants_match_the_method():
    # algorithmic counts: forward one exp per element; backward one recompute of the state from
    # its checkpoint and the decay again in the reverse sweep (the kernel executes a third for
    # its second recompute level, reported separately)
    assert bench.FWD_EX2_PER_ELEM == 1
    assert bench.BWD_EX2_PER_ELEM == 2
    assert bench.BWD_EX2_EXECUTED_PER_ELEM == 3
    assert bench.BWD_OPS_PER_ELEM == 12
    # the measured per-SM rates the peaks use (bench.py --rates on a GB300: 31.98 ex2, 125.2 FFMA)
    assert bench.EX2_PER_SM_CLK == 32 and bench.FP32_PER_SM_CLK == 128
