"""The measurement arithmetic of bench.py, on the CPU: the algorithmic bytes
and flops of one call (the numerators of the roofline fractions) against
counts written out by hand for the Mamba-2 2.7B shape, and the error metrics
of the parity report on a case whose answers are known."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_algorithmic_counts_of_the_2p7b_shape():
    import bench
    import ssd_inputs as si
    a = bench.algorithmic(si.CONFIGS["mamba2_2p7b"])
    # batch 8, seqlen 4096, 80 heads, headdim 64, dstate 128, 1 group, bf16:
    # x, z and out are 8*4096*80*64 elements of 2 bytes each, B and C
    # 8*4096*128, dt 8*4096*80, and A, D, dt_bias 80 fp32 values each
    x = 8 * 4096 * 80 * 64 * 2          # 335 544 320
    bc = 8 * 4096 * 128 * 2             # 8 388 608
    dt = 8 * 4096 * 80 * 2              # 5 242 880
    assert (a["x"], a["bc"], a["dt"]) == (x, bc, dt)
    assert a["io_bytes"] == 3 * x + 2 * bc + dt + 3 * 80 * 4 == 1_028_654_016
    # the call also writes the final states, 8*80*64*128 fp32
    fin = bench.algorithmic(si.CONFIGS["mamba2_2p7b"], final=True)
    assert fin["io_bytes"] == 1_028_654_016 + 8 * 80 * 64 * 128 * 4 == 1_049_625_536
    # causal flops per (batch row, 256-token chunk): C B^T over the 256*257/2
    # pairs j <= i once for the group (dstate 128), then per head the masked
    # product with x over the same pairs (headdim 64), C h and B^T x over all
    # 256 tokens (128 x 64 each), two flops per multiply-add; 16 chunks
    pairs = 256 * 257 // 2
    per_chunk = pairs * 128 * 2 + 80 * (pairs * 64 * 2 + 2 * 256 * 128 * 64 * 2)
    assert a["nc"] == 16 and a["tri"] == pairs
    assert a["flops"] == 8 * 16 * per_chunk == 130_094_727_168


def test_algorithmic_counts_follow_the_options():
    import dataclasses

    import bench
    import ssd_inputs as si
    cfg = si.CONFIGS["mamba2_2p7b"]
    base = bench.algorithmic(cfg)["io_bytes"]
    state = 8 * 80 * 64 * 128 * 4
    assert bench.algorithmic(cfg, init=True, final=True)["io_bytes"] == base + 2 * state
    assert bench.algorithmic(cfg, seq=True)["io_bytes"] == base + 8 * 4096 * 4   # seq_idx
    no_z = dataclasses.replace(cfg, has_z=False)
    assert bench.algorithmic(no_z)["io_bytes"] == base - 8 * 4096 * 80 * 64 * 2
    f32 = dataclasses.replace(cfg, dtype="f32")
    a32 = bench.algorithmic(f32)
    assert a32["io_bytes"] == 2 * (base - 3 * 80 * 4) + 3 * 80 * 4
    # a ragged last chunk counts as a whole one in the causal flops
    assert bench.algorithmic(cfg, seqlen=4097)["nc"] == 17


def test_error_metrics_on_known_errors():
    import bench
    ref = [np.array([[1.0, -2.0, 4.0, 0.0]]), np.array([[2.0, 2.0, -8.0, 1.0]])]
    err = [np.array([[0.5, 0.0, 0.0, 0.0]]), np.array([[0.0, -1.0, 0.0, 0.25]])]
    m = bench.error_metrics([(r + e, r) for r, e in zip(ref, err)])
    assert m["elements"] == 8
    assert m["max_rel"] == pytest.approx(1.0 / 8.0)          # max|err| 1 over max|ref| 8
    assert m["mean_rel"] == pytest.approx(1.75 / 20.0)       # sum|err| over sum|ref|
    assert m["mean_diff"] == pytest.approx((0.5 - 1.0 + 0.25) / 8)
    # 99.9th percentile of |err| per row: close to each row's largest error
    q0 = np.quantile([0.5, 0.0, 0.0, 0.0], 0.999)
    q1 = np.quantile([0.0, 1.0, 0.0, 0.25], 0.999)
    assert m["p999_rel"] == pytest.approx(max(q0, q1) / 8.0)
