"""The backward of the scan on the GPU (ssd_scan_bwd, fp32) against the
oracle's gradients: reverse-mode differentiation, in fp64, of the plain
token-by-token recurrence.  Every gradient is compared element by element:
x, the raw dt, dt_bias, A, B, C, D, z and the initial states.

Tolerance.  Gradients with one value per input element (x, dt, B, C, z, the
initial states): max|err| / max|ref| <= 1e-4, the forward's fp32 bound.
Each is a sum of fp32 products over at most one chunk's tokens times dstate
(or headdim) terms per scan, plus a sum over the chunks through the state
chain; with fp32's 6e-8 unit roundoff and sums of random sign that stays
near 1e-6 relative, and 1e-4 leaves the margin the forward's tests leave.
The per-head gradients (dt_bias, A, D) are sums of terms t (ddt per token;
dy x per element; for dA the elementary products of its pair form, each
pair of tokens j < i of a document contributing L_ij dt_j C_in B_jn
dy_ip x_jp over n and p, times the dt it spans), so the bound that the
elementwise one implies is |err_h| <= 1e-4 sum |t_h|: a sum of terms each
within a relative 1e-4.  (The per-token decay gradient is not such a term:
it is itself a sum over the pairs around a token, and those cancel, as do
the dot products inside a pair.)

Cases span several chunks with a ragged tail, grouped B/C, documents
(seq_idx, a one-token document among them), clamps that bite, dt without
softplus (signed), no optional inputs at all (with the strong decays that
unbiased dt gives), one token, and the per-head shape of the Mamba-2 2.7B
workload."""
import math

import numpy as np
import pytest
import torch

from oracle import ssd_oracle as so
import ssd_inputs as si
from ssd_testutil import PARITY_REPORT, TOL, assert_close, errors, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("x", "dt", "dt_bias", "A", "B", "C", "D", "z", "initial_states")
OUT = {"x": "dx", "dt": "ddt", "dt_bias": "d_dt_bias", "A": "dA", "B": "dB", "C": "dC",
       "D": "dD", "z": "dz", "initial_states": "d_initial_states"}

CASES = [
    # (id, random_small kwargs)
    ("ragged_groups_init", dict(batch=2, seqlen=300, nheads=4, headdim=32, dstate=64,
                                ngroups=2, chunk_size=64, init_std=0.3)),
    ("docs_init", dict(batch=2, seqlen=300, nheads=4, headdim=32, dstate=64, ngroups=2,
                       chunk_size=64, init_std=0.3, seq_idx_lengths=[100, 1, 199])),
    ("clamp_softplus", dict(batch=1, seqlen=257, nheads=6, headdim=16, dstate=32, ngroups=3,
                            chunk_size=32, dt_limit=(0.3, 1.0), init_std=0.2)),
    ("signed_dt_no_softplus", dict(batch=2, seqlen=200, nheads=2, headdim=64, dstate=16,
                                   ngroups=1, chunk_size=64, dt_softplus=False, dt_bias=False,
                                   a_log_range=(math.log(0.01), math.log(0.1)))),
    ("no_optionals", dict(batch=1, seqlen=130, nheads=4, headdim=128, dstate=16, ngroups=4,
                          chunk_size=16, has_z=False, has_D=False, dt_bias=False)),
    ("one_token", dict(batch=3, seqlen=1, nheads=2, headdim=16, dstate=16, ngroups=1,
                       chunk_size=16, init_std=0.5)),
    ("mamba2_2p7b_heads", dict(batch=1, seqlen=700, nheads=2, headdim=64, dstate=128,
                               ngroups=1, chunk_size=256, init_std=0.1,
                               seq_idx_lengths=[300, 400])),
    ("hd128_ds128", dict(batch=1, seqlen=300, nheads=4, headdim=128, dstate=128, ngroups=2,
                         chunk_size=128, init_std=0.2, seq_idx_lengths=[129, 171])),
    ("hd128_ds64", dict(batch=2, seqlen=200, nheads=2, headdim=128, dstate=64, ngroups=1,
                        chunk_size=128, init_std=0.2)),
]


def _run(d, dout):
    import selective_state_space_05_gb300 as ssd
    g = to_dev(d)
    res = ssd.ssd_scan_bwd(dout.cuda(), g["x"], g["dt"], g["A"], g["B"], g["C"],
                           chunk_size=d["chunk_size"], dt_bias=g["dt_bias"],
                           dt_softplus=d["dt_softplus"], dt_limit=d["dt_limit"], D=g["D"],
                           z=g["z"], initial_states=g["initial_states"], seq_idx=g["seq_idx"])
    torch.cuda.synchronize()
    return res


def _head_terms(d, dout, ref):
    """The scale of each per-head gradient, [H]: the sum of the absolute
    values of the terms it adds up -- d_dt_bias: ddt per token; dD: dy x per
    element; dA: the elementary products of its pair form (oracle
    decay_gradient_pairs), each times the dt it spans."""
    x = d["x"].double().numpy()
    dy = dout.double().numpy()
    if d["z"] is not None:
        z = d["z"].double().numpy()
        dy = dy * z / (1.0 + np.exp(-z))
    return {"dt_bias": np.abs(ref["dt"]).sum(axis=(0, 1)),
            "A": so.decay_gradient_pairs(d, dout)[1],
            "D": np.abs(dy * x).sum(axis=(0, 1, 3))}


def _check(name, d, dout, got, ref):
    scale = _head_terms(d, dout, ref)
    bad, checked = [], 0
    report = PARITY_REPORT.setdefault(f"backward {name}", {"tol": TOL["f32"]})
    for k in NAMES:
        if k in scale:
            want = ref.get(k)
            if want is None:   # not an input: its gradient is still defined
                want = (ref["dt"].sum(axis=(0, 1)) if k == "dt_bias" else
                        (dout.double().numpy() * d["x"].double().numpy()).sum(axis=(0, 1, 3)))
            err = np.abs(got[OUT[k]].double().cpu().numpy() - want)
            sc = scale[k]
            ratio = np.where(sc > 0, err / np.where(sc > 0, sc, 1.0), np.where(err > 0, np.inf, 0.0))
            worst = float(ratio.max())
            report[f"d{k}"] = {"max_err_over_sum_abs_terms": worst}
            if worst > TOL["f32"]:
                bad.append(f"d{k}: max |err| / sum|terms| = {worst:.2e}")
            checked += 1
            continue
        if d.get(k) is None:
            assert got[OUT[k]] is None
            continue
        e = errors(got[OUT[k]].double().cpu().numpy(), ref[k])
        report[f"d{k}"] = e
        if e["max_rel"] > TOL["f32"]:
            bad.append(f"d{k}: {e}")
        checked += 1
    assert not bad, f"{name}: " + "; ".join(bad)
    assert checked >= 6


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(case):
    name, kw = case
    d = si.random_small(500 + len(name), **kw)
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(len(name)))
    ref = so.scan_backward(d, dout)
    _check(name, d, dout, _run(d, dout), ref)


def test_clamped_tokens_get_no_dt_gradient():
    """Where the clamp bites (softplus(dt + bias) outside [lo, hi]) the raw
    dt's gradient is exactly zero; elsewhere it is not."""
    d = si.random_small(77, batch=1, seqlen=100, nheads=2, headdim=16, dstate=16, ngroups=1,
                        chunk_size=32, dt_limit=(0.5, 0.9))
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(1))
    got = _run(d, dout)["ddt"].cpu()
    v = torch.nn.functional.softplus(d["dt"] + d["dt_bias"])
    out = (v < 0.5) | (v > 0.9)
    assert out.any() and (~out).any()
    assert torch.all(got[out] == 0)
    assert torch.count_nonzero(got[~out]) == int((~out).sum())


def test_backward_is_linear_in_dout():
    """The gradients are linear in dout: bwd(a u + b v) = a bwd(u) + b bwd(v)."""
    d = si.random_small(78, batch=1, seqlen=200, nheads=2, headdim=32, dstate=32, ngroups=1,
                        chunk_size=64, init_std=0.2, has_z=False)
    gen = torch.Generator().manual_seed(2)
    u, v = torch.randn(d["x"].shape, generator=gen), torch.randn(d["x"].shape, generator=gen)
    gu, gv, gw = _run(d, u), _run(d, v), _run(d, 2.0 * u - 0.5 * v)
    for k, t in gw.items():
        if t is None:
            continue
        want = (2.0 * gu[k].double() - 0.5 * gv[k].double()).cpu().numpy()
        assert_close(t.double().cpu().numpy(), want, 1e-5, k)


def test_backward_rejects_bad_arguments():
    import selective_state_space_05_gb300 as ssd
    from selective_state_space_05_gb300._lib import SSDError
    d = to_dev(si.random_small(79, batch=1, seqlen=40, nheads=2, headdim=16, dstate=48,
                               ngroups=1, chunk_size=16))
    with pytest.raises(SSDError):   # dstate 48 is not one of 16, 32, 64, 128
        ssd.ssd_scan_bwd(torch.ones_like(d["x"]), d["x"], d["dt"], d["A"], d["B"], d["C"],
                         chunk_size=16)
    assert ssd.bwd_workspace_bytes(1, 40, 2, 16, 48, 1, 16) == 0
    assert ssd.bwd_workspace_bytes(1, 40, 2, 16, 32, 1, 16) > 0


def test_backward_full_size_sampled_pairs():
    """The Mamba-2 2.7B shape in fp32 (batch 8, seqlen 4096, 80 heads,
    headdim 64, dstate 128, one group, chunk 256), the launch the benchmark
    times: the per-element gradients of sampled (batch, head) pairs (dx, ddt,
    dz, d_initial_states) against the oracle run on that pair alone (a head's
    recurrence depends only on its own inputs and the shared B, C)."""
    import selective_state_space_05_gb300 as ssd
    cfg = si.CONFIGS["mamba2_2p7b"].with_(dtype="f32", init_std=0.1)
    d = si.make_inputs(cfg, 95)
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(96))
    got = _run(d, dout)
    for b, h in [(0, 0), (5, 47), (7, 79)]:
        sub = {k: v for k, v in d.items()}
        for k in ("x", "z"):
            sub[k] = d[k][b:b + 1, :, h:h + 1].contiguous()
        sub["dt"] = d["dt"][b:b + 1, :, h:h + 1].contiguous()
        for k in ("B", "C"):
            sub[k] = d[k][b:b + 1].contiguous()
        for k in ("A", "D", "dt_bias"):
            sub[k] = d[k][h:h + 1].contiguous()
        sub["initial_states"] = d["initial_states"][b:b + 1, h:h + 1].contiguous()
        sub["ngroups"] = 1
        ref = so.scan_backward(sub, dout[b:b + 1, :, h:h + 1],
                               names=("x", "dt", "z", "initial_states"))
        rep = PARITY_REPORT.setdefault(f"backward mamba2_2p7b fp32 pair ({b},{h})",
                                       {"tol": TOL["f32"]})
        for k, gk in (("x", "dx"), ("dt", "ddt"), ("z", "dz")):
            g = got[gk][b:b + 1, :, h:h + 1].double().cpu().numpy()
            rep[f"d{k}"] = assert_close(g, ref[k], TOL["f32"], f"({b},{h}) d{k}")
        g = got["d_initial_states"][b:b + 1, h:h + 1].double().cpu().numpy()
        rep["dinitial_states"] = assert_close(g, ref["initial_states"], TOL["f32"],
                                              f"({b},{h}) dh0")


def test_bf16_backward_is_the_fp32_backward_rounded():
    """bf16 inputs (ssd_scan_bwd_ex): the gradients are the fp32 backward's on
    the same values, rounded to bf16 (bit for bit) for the element-wise ones,
    the same for the fp32 ones (up to the order of the per-head atomic sums);
    and against the oracle within the bf16
    bound (element-wise) and the fp32 bound (per-head sums, initial states)."""
    d = si.random_small(520, batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2,
                        chunk_size=256, dtype="bf16", init_std=0.3, seq_idx_lengths=[150, 150])
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(21)).bfloat16()
    gb = _run(d, dout)
    d32 = {k: (v.float() if torch.is_tensor(v) and v.dtype == torch.bfloat16 else v)
           for k, v in d.items()}
    g32 = _run(d32, dout.float())
    for k in ("dx", "ddt", "dB", "dC", "dz"):
        assert gb[k].dtype == torch.bfloat16
        assert torch.equal(gb[k], g32[k].bfloat16()), k
    for k in ("dA", "d_dt_bias", "dD", "d_initial_states"):
        assert gb[k].dtype == torch.float32
    assert torch.equal(gb["d_initial_states"], g32["d_initial_states"])
    # the per-head sums add warps' partial sums with atomics, in no fixed order
    for k in ("dA", "d_dt_bias", "dD"):
        assert torch.allclose(gb[k], g32[k], rtol=1e-5, atol=0.0), k
    ref = so.scan_backward(d32, dout.float())
    scale = _head_terms(d32, dout.float(), ref)
    for name, k in (("x", "dx"), ("dt", "ddt"), ("B", "dB"), ("C", "dC"), ("z", "dz")):
        assert_close(gb[k].double().cpu().numpy(), ref[name], TOL["bf16"], k)
    assert_close(gb["d_initial_states"].double().cpu().numpy(), ref["initial_states"],
                 TOL["f32"], "dh0")
    for name, k in (("A", "dA"), ("dt_bias", "d_dt_bias"), ("D", "dD")):
        err = np.abs(gb[k].double().cpu().numpy() - ref[name])
        assert (err <= TOL["f32"] * scale[name] + 1e-30).all(), k
