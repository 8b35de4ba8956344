"""The seeded input recipe shared by the oracle tests, the GPU parity tests and
bench.py: determinism, shapes and dtypes of the workloads, and the stated
distributions (dt_bias so that softplus(dt_bias) ~ U[1e-3, 1e-1], A_h =
-exp(U[log 1, log 16]), D, x / B / C scales, initial-state spread, the
Dirichlet document split)."""
import math

import numpy as np
import pytest
import torch

import ssd_inputs as si


@pytest.mark.parametrize("name", sorted(si.CONFIGS))
def test_shapes_and_dtypes(name):
    cfg = si.CONFIGS[name]
    L = min(cfg.seqlen, 64)
    d = si.make_inputs(cfg, 5, seqlen=L)
    B, H, P, N, G = cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    dt = si.torch_dtype(cfg.dtype)
    assert d["x"].shape == (B, L, H, P) and d["x"].dtype == dt
    assert d["dt"].shape == (B, L, H) and d["dt"].dtype == dt
    assert d["B"].shape == (B, L, G, N) and d["B"].dtype == dt
    assert d["C"].shape == (B, L, G, N) and d["C"].dtype == dt
    for k in ("dt_bias", "A"):
        assert d[k].shape == (H,) and d[k].dtype == torch.float32
    assert (d["z"] is not None) == cfg.has_z
    if d["z"] is not None:
        assert d["z"].shape == (B, L, H, P) and d["z"].dtype == dt
    assert (d["initial_states"] is not None) == (cfg.init_std > 0)
    if d["initial_states"] is not None:
        assert d["initial_states"].shape == (B, H, P, N)
        assert d["initial_states"].dtype == torch.float32
    assert (d["seq_idx"] is not None) == (cfg.ndocs > 1)
    assert d["chunk_size"] == cfg.chunk_size and d["ngroups"] == G


def test_same_seed_same_inputs_other_seed_other_inputs():
    cfg = si.CONFIGS["tiny"]
    a, b, c = si.make_inputs(cfg, 11), si.make_inputs(cfg, 11), si.make_inputs(cfg, 12)
    for k in ("x", "dt", "dt_bias", "A", "B", "C", "D"):
        assert torch.equal(a[k], b[k]), k
        assert not torch.equal(a[k], c[k]), k


def test_dt_bias_and_A_ranges():
    # many heads, so that the ranges are filled out
    cfg = si.CONFIGS["tiny"].with_(nheads=4096)
    d = si.make_inputs(cfg, 3, seqlen=1)
    sp = torch.nn.functional.softplus(d["dt_bias"].double())
    assert sp.min() >= 1e-3 * (1 - 1e-5) and sp.max() <= 1e-1 * (1 + 1e-5)
    assert sp.min() < 2e-3 and sp.max() > 9.8e-2          # spans the interval
    A = d["A"].double()
    assert A.max() <= -1.0 * (1 - 1e-6) and A.min() >= -16.0 * (1 + 1e-6)
    # log(-A) ~ U[0, log 16]: its mean is log(16) / 2
    assert abs(torch.log(-A).mean().item() - math.log(16.0) / 2) < 0.05


def test_scales_D_and_initial_states():
    g = si.make_inputs(si.CONFIGS["grouped_g2"], 4, seqlen=64)
    assert torch.equal(g["D"], torch.arange(32, dtype=torch.float32) * 1000.0)
    assert abs(g["x"].std().item() - 0.5) < 0.01
    assert abs(g["B"].std().item() - 0.5) < 0.02
    m = si.make_inputs(si.CONFIGS["mamba2_2p7b"], 4, seqlen=64)
    assert abs(m["x"].float().std().item() - 1.0) < 0.01
    assert m["D"].shape == (80,) and abs(m["D"].std().item() - 1.0) < 0.3
    c = si.make_inputs(si.CONFIGS["chained"], 4, seqlen=8)
    assert abs(c["initial_states"].std().item() - 0.1) < 0.002


def test_bf16_values_are_rounded_once():
    """Both sides read the same bf16 values: the tensors are bf16 already."""
    d = si.make_inputs(si.CONFIGS["mamba2_2p7b"], 6, seqlen=32)
    x = d["x"]
    assert x.dtype == torch.bfloat16
    assert torch.equal(x.float().to(torch.bfloat16), x)


@pytest.mark.parametrize("total,ndocs,seed", [(131072, 8, 1004), (100, 8, 1), (9, 8, 2),
                                              (8, 8, 3), (1000, 1, 4)])
def test_dirichlet_lengths(total, ndocs, seed):
    lens = si.dirichlet_lengths(total, ndocs, seed)
    assert len(lens) == ndocs and sum(lens) == total and min(lens) >= 1
    assert lens == si.dirichlet_lengths(total, ndocs, seed)


def test_packed_seq_idx_marks_the_split():
    cfg = si.CONFIGS["packed"]
    L = 4096
    d = si.make_inputs(cfg, 1004, seqlen=L)
    s = d["seq_idx"]
    assert s.shape == (1, L) and s.dtype == torch.int32
    lens = si.dirichlet_lengths(L, cfg.ndocs, 1004)
    ids = s[0].numpy()
    assert np.all(np.diff(ids) >= 0) and ids[0] == 0 and ids[-1] == cfg.ndocs - 1
    assert np.bincount(ids, minlength=cfg.ndocs).tolist() == lens


def test_random_small_options():
    d = si.random_small(7, seqlen=20, seq_idx_lengths=[5, 15], dt_bias=False, has_D=False,
                        has_z=False, init_std=0.2)
    assert d["dt_bias"] is None and d["D"] is None and d["z"] is None
    assert d["initial_states"] is not None
    assert d["seq_idx"][0].tolist() == [0] * 5 + [1] * 15
    with pytest.raises(AssertionError):
        si.random_small(7, seqlen=20, seq_idx_lengths=[5, 14])
