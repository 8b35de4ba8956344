"""Pins for the CPU fp64 oracle (no GPU).

Each check ties the oracle to something other than itself: printed values on
the pages, closed forms, a library routine, brute force on tiny inputs and the
invariants the method must satisfy (chunk-size independence, chaining through
final/initial states, group replication, document packing).  The last test
plants mistakes in the C oracle and shows that these pins catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from oracle import ssd_oracle as so

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TIGHT = 1e-11


def rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den > 0 else 1.0))


# --------------------------------------------------------------------------
# worked example printed on the "ngroups > 1" issue page
# --------------------------------------------------------------------------

def _p1_block_out(G: int, grouped: bool, mutation: int = 0) -> float:
    """out[0,0,0] of the page's block at t = 0, built around the oracle.

    At t = 0 the causal width-4 conv sees only its last tap: every conv
    channel is 0.1*0.1 + 0.1 = 0.11, then SiLU; so x, B and C all equal
    s = silu(0.11).  z = dt_raw = 0.1.  The oracle runs the scan (D-skip and
    silu(z) gate included; the page's block applies the gate before the norm,
    norm_before_gate=False).  The rest is the page's RMSNorm (weight 0.1,
    eps 1e-5, over dim/ngroups channels when grouped) and out-projection
    (weight 0.1, bias 0.1), written here as test-side glue.
    """
    H, P, N = 32, 64, 128
    dim = H * P
    s = 0.11 / (1.0 + math.exp(-0.11))
    f = torch.float64
    d = dict(x=torch.full((1, 1, H, P), s, dtype=f),
             dt=torch.full((1, 1, H), 0.1, dtype=f),
             dt_bias=torch.full((H,), 0.1, dtype=f),
             A=-torch.exp(torch.zeros(H, dtype=f)),
             B=torch.full((1, 1, G, N), s, dtype=f),
             C=torch.full((1, 1, G, N), s, dtype=f),
             D=torch.arange(H, dtype=f) * 1000.0,
             z=torch.full((1, 1, H, P), 0.1, dtype=f),
             dt_softplus=True, dt_limit=(0.0, float("inf")))
    y, _ = so.scan_sequential(d, mutation=mutation)
    y = y.reshape(dim)                       # channel = h * headdim + p
    gs = dim // G if grouped else dim
    yg = y.reshape(-1, gs)
    yn = (yg / np.sqrt((yg ** 2).mean(axis=1, keepdims=True) + 1e-5)).reshape(dim) * 0.1
    return float(0.1 * yn.sum() + 0.1)


def test_p1_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "p1_worked_example.json")))
    for G in (1, 2, 4):
        assert abs(_p1_block_out(G, True) - g["printed"]["combined"][str(G)]) < 1.5e-4
        assert abs(_p1_block_out(G, False) - g["printed"]["ref"][str(G)]) < 1.5e-4


def _p1_block_full(G: int, grouped: bool, L: int = 5) -> np.ndarray:
    """The page's whole block over the first L tokens, in fp64, from the
    oracle's conv, scan and group norm (the out-projection, weight 0.1 and
    bias 0.1 as on the page, is test-side glue): out[0, :, 0]."""
    H, P, N, Wc = 32, 64, 128, 4
    dim = H * P
    conv_dim = dim + 2 * G * N
    zx = np.full((1, L, 2 * dim + 2 * G * N + H), 0.1)
    xbc = oracle.causal_conv1d(zx[:, :, dim:dim + conv_dim], np.full((conv_dim, Wc), 0.1),
                               np.full(conv_dim, 0.1), silu=True)
    f = torch.float64
    d = dict(x=torch.from_numpy(xbc[:, :, :dim].reshape(1, L, H, P).copy()),
             B=torch.from_numpy(xbc[:, :, dim:dim + G * N].reshape(1, L, G, N).copy()),
             C=torch.from_numpy(xbc[:, :, dim + G * N:].reshape(1, L, G, N).copy()),
             dt=torch.from_numpy(zx[:, :, -H:].copy()),
             dt_bias=torch.full((H,), 0.1, dtype=f), A=-torch.ones(H, dtype=f),
             D=torch.arange(H, dtype=f) * 1000.0,
             z=torch.from_numpy(zx[:, :, :dim].reshape(1, L, H, P).copy()),
             dt_softplus=True, dt_limit=(0.0, float("inf")))
    y, _ = so.scan_sequential(d)
    yn = oracle.group_rmsnorm(y.reshape(1, L, dim), np.full(dim, 0.1), 1e-5,
                              dim // G if grouped else dim)
    return 0.1 * yn.sum(axis=-1)[0] + 0.1


def test_p1_worked_example_through_block_oracle():
    """The printed values again, now through the oracle's conv and group
    norm over a short sequence (token 0 is the printed one); later tokens
    see more conv taps and the recurrence, and must differ from token 0."""
    g = json.load(open(os.path.join(GOLDEN, "p1_worked_example.json")))
    for G in (1, 2, 4):
        out = _p1_block_full(G, True)
        assert abs(out[0] - g["printed"]["combined"][str(G)]) < 1.5e-4
        assert abs(out[0] - _p1_block_out(G, True)) < 1e-9
        assert abs(out[1] - out[0]) > 1e-6   # (the norm and the D skip keep it small)
        ref = _p1_block_full(G, False)
        assert abs(ref[0] - g["printed"]["ref"][str(G)]) < 1.5e-4


def test_causal_conv1d_is_numpy_convolve():
    """Per channel, the causal conv is numpy's full convolution with the
    reversed filter, truncated to the sequence (a library routine)."""
    rng = np.random.default_rng(3)
    for W in (1, 2, 4, 7):
        x = rng.normal(size=(2, 23, 5))
        w = rng.normal(size=(5, W))
        b = rng.normal(size=5)
        out = oracle.causal_conv1d(x, w, b, silu=False)
        for bi in range(2):
            for c in range(5):
                ref = np.convolve(x[bi, :, c], w[c, ::-1])[:23] + b[c]
                assert rel(out[bi, :, c], ref) < 1e-14
        s = oracle.causal_conv1d(x, w, b, silu=True)
        assert rel(s, out / (1 + np.exp(-out))) < 1e-14


def test_causal_conv1d_impulse_and_documents():
    """A unit impulse at token t0 gives the filter reversed over t0..t0+W-1;
    with seq_idx every document is convolved on its own (the result equals
    the concatenation of the separate convolutions)."""
    W = 4
    w = np.arange(1.0, 1 + 3 * W).reshape(3, W)
    x = np.zeros((1, 12, 3))
    x[0, 5, :] = 1.0
    out = oracle.causal_conv1d(x, w, None, silu=False)
    for c in range(3):
        want = np.zeros(12)
        want[5:5 + W] = w[c, ::-1]
        assert np.array_equal(out[0, :, c], want)
    rng = np.random.default_rng(4)
    lens = [7, 1, 3, 9]
    x = rng.normal(size=(2, sum(lens), 3))
    sq = torch.cat([torch.full((n,), i, dtype=torch.int32) for i, n in enumerate(lens)])
    sq = sq.unsqueeze(0).expand(2, -1).contiguous()
    packed = oracle.causal_conv1d(x, w, np.ones(3), seq_idx=sq, silu=True)
    parts, t = [], 0
    for n in lens:
        parts.append(oracle.causal_conv1d(x[:, t:t + n], w, np.ones(3), silu=True))
        t += n
    assert rel(packed, np.concatenate(parts, axis=1)) < 1e-15


def test_group_rmsnorm_closed_forms_and_library():
    rng = np.random.default_rng(5)
    y = rng.normal(size=(3, 4, 48))
    w = rng.normal(size=48)
    for gs in (48, 16, 8):
        out = oracle.group_rmsnorm(y, w, 1e-5, gs)
        # torch's own RMSNorm over each group (a library routine)
        t = torch.nn.functional.rms_norm(torch.from_numpy(y).reshape(3, 4, 48 // gs, gs), (gs,),
                                         eps=1e-5).reshape(3, 4, 48).numpy() * w
        assert rel(out, t) < 1e-13
    # a constant group: y / sqrt(y^2 + eps), times the weight
    c = np.full((1, 1, 16), -2.0)
    out = oracle.group_rmsnorm(c, np.full(16, 0.5), 1e-3, 8)
    assert np.allclose(out, 0.5 * -2.0 / math.sqrt(4.0 + 1e-3), rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# dt preprocessing
# --------------------------------------------------------------------------

def test_dt_processing_matches_library_softplus():
    rng = np.random.default_rng(0)
    raw = rng.normal(size=(2, 9, 3)) * 30
    bias = rng.normal(size=3)
    # softplus(v) = log(1 + e^v) = numpy's logaddexp(0, v)
    ref = np.logaddexp(0.0, raw + bias)
    assert rel(oracle.dt_process_c(raw, bias, True, 0.0, math.inf), ref) < 1e-15
    assert rel(oracle.dt_process(raw, bias, True, 0.0, math.inf), ref) < 1e-15
    # clamp after softplus
    ref_c = np.clip(ref, 0.05, 2.0)
    assert rel(oracle.dt_process_c(raw, bias, True, 0.05, 2.0), ref_c) < 1e-15
    # no softplus, default limit: untouched (negative values stay)
    assert np.array_equal(oracle.dt_process_c(raw, None, False, 0.0, math.inf), raw)
    # known values: softplus(0) = ln 2
    z = np.zeros((1, 1, 1))
    assert abs(oracle.dt_process_c(z, None, True, 0.0, math.inf)[0, 0, 0] - math.log(2)) < 1e-16


# --------------------------------------------------------------------------
# brute force: sequential recurrence == materialised quadratic form
# --------------------------------------------------------------------------

CASES = [
    dict(),
    dict(init_std=0.5),
    dict(seq_idx_lengths=[5, 1, 20, 11]),
    dict(seq_idx_lengths=[1, 35, 1], init_std=0.2),
    dict(has_z=False, has_D=False, dt_bias=False),
    dict(ngroups=1, nheads=3),
    dict(ngroups=4, nheads=4, init_std=1.0, seq_idx_lengths=[16, 16, 5]),
    dict(dt_softplus=False, a_log_range=(-3.0, 0.0)),
    dict(dt_limit=(0.02, 0.3)),
    dict(a_log_range=(math.log(1e-3), math.log(1e-1)), seqlen=60, init_std=0.3),
]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_sequential_equals_quadratic(kw):
    d = si.random_small(11, **kw)
    y1, f1 = so.scan_sequential(d)
    y2, f2 = so.scan_quadratic(d)
    assert rel(y1, y2) < TIGHT
    assert rel(f1, f2) < TIGHT


# --------------------------------------------------------------------------
# chunked form: any chunk length gives the recurrence's result
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Q", [1, 7, 16, 64, 37, 50])
def test_chunk_size_invariance(Q):
    d = si.random_small(3, seqlen=37, init_std=0.4, seq_idx_lengths=[9, 7, 1, 20])
    y1, f1 = so.scan_sequential(d)
    y2, f2 = so.scan_chunked(d, Q)
    assert rel(y1, y2) < TIGHT
    assert rel(f1, f2) < TIGHT


def test_chunked_intermediates_shapes_and_states():
    d = si.random_small(4, seqlen=40, init_std=0.4)
    y, f, im = so.scan_chunked(d, 16, return_intermediates=True)
    assert im["cs"].shape == (2, 4, 3, 16)
    assert im["states"].shape == (2, 3, 4, 8, 6)
    # state entering chunk 0 is the initial state
    assert np.array_equal(im["prev_states"][:, 0], so.f64(d["initial_states"]))


# --------------------------------------------------------------------------
# chaining: final_states fed back as initial_states == one whole run
# --------------------------------------------------------------------------

def _slice(d, t0, t1, init):
    e = dict(d)
    for k in ("x", "dt", "B", "C", "z", "seq_idx"):
        if e.get(k) is not None:
            e[k] = e[k][:, t0:t1].contiguous()
    e["initial_states"] = None if init is None else torch.from_numpy(init)
    return e


@pytest.mark.parametrize("nseg,docs", [(2, None), (4, None), (3, [10, 30, 8])])
def test_chaining(nseg, docs):
    L = 48
    d = si.random_small(5, seqlen=L, init_std=0.3, seq_idx_lengths=docs)
    y_all, f_all = so.scan_sequential(d)
    cuts = np.linspace(0, L, nseg + 1).astype(int)
    st = so.f64(d["initial_states"])
    ys = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        y, st = so.scan_sequential(_slice(d, a, b, st))
        ys.append(y)
    assert rel(np.concatenate(ys, axis=1), y_all) < TIGHT
    assert rel(st, f_all) < TIGHT


# --------------------------------------------------------------------------
# head -> group mapping: G > 1 == G' = H with each head's B/C replicated
# --------------------------------------------------------------------------

@pytest.mark.parametrize("G", [2, 4])
def test_group_replication(G):
    H = 8
    d = si.random_small(6, nheads=H, ngroups=G, init_std=0.2)
    y1, f1 = so.scan_sequential(d)
    e = dict(d)
    idx = torch.arange(H) // (H // G)            # head h reads group h / (H/G)
    e["B"] = d["B"][:, :, idx].contiguous()
    e["C"] = d["C"][:, :, idx].contiguous()
    y2, f2 = so.scan_sequential(e)
    assert rel(y1, y2) < 1e-15 and rel(f1, f2) < 1e-15
    # and the mapping is not the interleaved one h % G
    e2 = dict(d)
    idx2 = torch.arange(H) % G
    e2["B"] = d["B"][:, :, idx2].contiguous()
    e2["C"] = d["C"][:, :, idx2].contiguous()
    y3, _ = so.scan_sequential(e2)
    assert rel(y1, y3) > 1e-3


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_closed_form_linear_attention():
    """A = 0, dt = 1 (no softplus, no bias): no decay, unit step, so
    y_t = C_t . sum_{s<=t} x_s (outer) B_s -- causal linear attention, here a
    cumulative sum of outer products."""
    d = si.random_small(7, has_z=False, has_D=False, dt_bias=False, dt_softplus=False)
    d["dt"] = torch.ones_like(d["dt"])
    d["A"] = torch.zeros_like(d["A"])
    x, Bm, Cm = (so.f64(d[k]) for k in ("x", "B", "C"))
    H, G = x.shape[2], Bm.shape[2]
    gi = np.arange(H) // (H // G)
    kv = np.cumsum(np.einsum("blhp,blhn->blhpn", x, Bm[:, :, gi]), axis=1)
    ref = np.einsum("blhpn,blhn->blhp", kv, Cm[:, :, gi])
    y, f = so.scan_sequential(d)
    assert rel(y, ref) < TIGHT
    assert rel(f, kv[:, -1]) < TIGHT


def test_closed_form_constant_inputs():
    """Constant dt, x, B, C: h_t = dt x B^T (1 - r^(t+1)) / (1 - r), r = e^{dt A}
    (a geometric series); y_t = (C . B) dt x (1 - r^(t+1)) / (1 - r)."""
    L, H, P, N = 50, 3, 2, 5
    f = torch.float64
    A = torch.tensor([-0.3, -1.0, -4.0], dtype=f)
    dtv, xv, bv, cv = 0.7, 1.3, -0.4, 0.9
    d = dict(x=torch.full((1, L, H, P), xv, dtype=f), dt=torch.full((1, L, H), dtv, dtype=f),
             dt_bias=None, A=A, B=torch.full((1, L, 1, N), bv, dtype=f),
             C=torch.full((1, L, 1, N), cv, dtype=f), D=None, z=None,
             dt_softplus=False)
    y, fin = so.scan_sequential(d)
    t = np.arange(L)
    for h in range(H):
        r = math.exp(dtv * float(A[h]))
        geo = (1 - r ** (t + 1)) / (1 - r)
        ref = N * cv * bv * dtv * xv * geo
        assert rel(y[0, :, h, 0], ref) < 1e-13
        assert abs(fin[0, h, 0, 0] - dtv * xv * bv * geo[-1]) < 1e-13


def test_closed_form_decay_of_initial_state():
    """x = 0: the state only decays, h_t = exp(dt A (t+1)) h0 for constant dt,
    and y_t = exp(dt A (t+1)) h0 C_t."""
    L, H, P, N = 20, 2, 3, 4
    rng = np.random.default_rng(1)
    h0 = rng.normal(size=(1, H, P, N))
    Cm = rng.normal(size=(1, L, 1, N))
    f = torch.float64
    A = torch.tensor([-0.5, -2.0], dtype=f)
    d = dict(x=torch.zeros(1, L, H, P, dtype=f), dt=torch.full((1, L, H), 0.25, dtype=f),
             A=A, B=torch.ones(1, L, 1, N, dtype=f), C=torch.from_numpy(Cm),
             initial_states=torch.from_numpy(h0), dt_softplus=False)
    y, fin = so.scan_sequential(d)
    for h in range(H):
        e = np.exp(0.25 * float(A[h]) * (np.arange(L) + 1))
        ref = e[:, None] * (Cm[0, :, 0, :] @ h0[0, h].T)
        assert rel(y[0, :, h, :], ref) < 1e-13
        assert rel(fin[0, h], e[-1] * h0[0, h]) < 1e-13


def test_closed_form_single_token():
    """L = 1 from a zero state: y = dt (C . B) x + D x."""
    d = si.random_small(8, seqlen=1, has_z=False)
    dt = oracle.dt_process(d["dt"], d["dt_bias"], True, 0.0, math.inf)
    x, Bm, Cm, D = (so.f64(d[k]) for k in ("x", "B", "C", "D"))
    H, G = x.shape[2], Bm.shape[2]
    gi = np.arange(H) // (H // G)
    cb = np.einsum("bln,bln->bl", Cm[:, :, gi].reshape(-1, H, Bm.shape[-1]),
                   Bm[:, :, gi].reshape(-1, H, Bm.shape[-1])).reshape(x.shape[0], 1, H)
    ref = (dt * cb)[..., None] * x + D[None, None, :, None] * x
    y, _ = so.scan_sequential(d)
    assert rel(y, ref) < 1e-14


def test_scalar_case_matches_iir_filter():
    """P = N = H = 1 with constant dt: h_t = r h_{t-1} + dt B_t x_t is a
    first-order IIR filter; scipy.signal.lfilter computes it independently."""
    signal = pytest.importorskip("scipy.signal")
    L = 300
    rng = np.random.default_rng(2)
    x, Bv, Cv = rng.normal(size=L), rng.normal(size=L), rng.normal(size=L)
    dtv, A = 0.3, -0.8
    f = torch.float64
    d = dict(x=torch.tensor(x, dtype=f).view(1, L, 1, 1),
             dt=torch.full((1, L, 1), dtv, dtype=f), A=torch.tensor([A], dtype=f),
             B=torch.tensor(Bv, dtype=f).view(1, L, 1, 1),
             C=torch.tensor(Cv, dtype=f).view(1, L, 1, 1), dt_softplus=False)
    y, _ = so.scan_sequential(d)
    r = math.exp(dtv * A)
    h = signal.lfilter([1.0], [1.0, -r], dtv * Bv * x)
    assert rel(y[0, :, 0, 0], Cv * h) < 1e-13


# --------------------------------------------------------------------------
# document packing: seq_idx resets == separate runs from zero state
# --------------------------------------------------------------------------

def test_packed_documents_equal_separate_runs():
    lens = [7, 1, 13, 19]
    L = sum(lens)
    d = si.random_small(9, seqlen=L, seq_idx_lengths=lens, init_std=0.5)
    y, fin = so.scan_sequential(d)
    t0 = 0
    for i, n in enumerate(lens):
        e = _slice(d, t0, t0 + n, so.f64(d["initial_states"]) if i == 0 else None)
        e["seq_idx"] = None
        ye, fe = so.scan_sequential(e)
        assert rel(y[:, t0:t0 + n], ye) < TIGHT
        t0 += n
    assert rel(fin, fe) < TIGHT   # final state belongs to the last document


def test_head_subset_matches_full_run():
    d = si.random_small(10, nheads=8, ngroups=2, init_std=0.1, seq_idx_lengths=[20, 17])
    y, f = so.scan_sequential(d)
    ys, fs = so.scan_sequential(d, heads=[1, 6], batches=[1])
    assert np.array_equal(ys[0], y[1][:, [1, 6]])
    assert np.array_equal(fs[0], f[1][[1, 6]])


# --------------------------------------------------------------------------
# planted mistakes: every mutation of the C oracle fails at least one pin
# --------------------------------------------------------------------------

MUTATIONS = {1: "decay sign flipped", 2: "dt dropped from the input term",
             3: "B and C swapped", 4: "head->group map h % G",
             5: "seq_idx resets ignored", 6: "D skip dropped",
             7: "gate without sigmoid"}


@pytest.mark.parametrize("k", sorted(MUTATIONS), ids=[MUTATIONS[k] for k in sorted(MUTATIONS)])
def test_planted_mistakes_are_caught(k):
    failures = 0
    # pin A: brute-force quadratic form on a case with every option on
    d = si.random_small(12, nheads=4, ngroups=2, init_std=0.3,
                        seq_idx_lengths=[10, 1, 26])
    y_m, f_m = so.scan_sequential(d, mutation=k)
    y_q, f_q = so.scan_quadratic(d)
    failures += rel(y_m, y_q) > 1e-9 or rel(f_m, f_q) > 1e-9
    # pin B: the page's printed worked example
    g = json.load(open(os.path.join(GOLDEN, "p1_worked_example.json")))
    for G in (1, 2, 4):
        failures += abs(_p1_block_out(G, True, mutation=k) - g["printed"]["combined"][str(G)]) > 1.5e-4
    assert failures > 0, f"mutation {k} ({MUTATIONS[k]}) not caught"


# --------------------------------------------------------------------------
# backward: the torch form of the recurrence and its reverse-mode gradients
# --------------------------------------------------------------------------

def test_torch_recurrence_equals_c_oracle():
    for kw in (dict(init_std=0.5, seq_idx_lengths=[10, 1, 26]),
               dict(has_z=False, dt_limit=(0.02, 0.3)),
               dict(dt_softplus=False, dt_bias=False, a_log_range=(-3.0, 0.0))):
        d = si.random_small(70, **kw)
        if not kw.get("dt_softplus", True):
            d["dt"] = d["dt"].abs() * 0.2
        t = {k: (torch.as_tensor(v).to(torch.float64) if torch.is_tensor(v) and
                 v.dtype != torch.int32 else v) for k, v in d.items()}
        out, fin = so.scan_torch(t["x"], t["dt"], t["A"], t["B"], t["C"], dt_bias=t["dt_bias"],
                                 D=t["D"], z=t["z"], initial_states=t["initial_states"],
                                 seq_idx=t["seq_idx"], dt_softplus=d["dt_softplus"],
                                 dt_limit=d["dt_limit"])
        ry, rf = so.scan_sequential(d)
        assert rel(out.numpy(), ry) < TIGHT and rel(fin.numpy(), rf) < TIGHT


def test_backward_oracle_passes_gradcheck():
    """The reverse-mode gradients the backward oracle returns agree with
    central finite differences of the forward (torch's gradcheck), on a tiny
    case with every input, a reset and a clamp."""
    d = si.random_small(71, batch=1, seqlen=6, nheads=2, ngroups=1, headdim=2, dstate=3,
                        init_std=0.5, seq_idx_lengths=[4, 2], dt_limit=(0.0, 3.0))
    t = {k: torch.as_tensor(v).to(torch.float64).requires_grad_(True)
         for k, v in d.items() if torch.is_tensor(v) and v.dtype != torch.int32}
    sq = d["seq_idx"]

    def f(x, dt, A, B, C, dt_bias, D, z, h0):
        return so.scan_torch(x, dt, A, B, C, dt_bias=dt_bias, D=D, z=z, initial_states=h0,
                             seq_idx=sq, dt_limit=(0.0, 3.0))[0]
    args = (t["x"], t["dt"], t["A"], t["B"], t["C"], t["dt_bias"], t["D"], t["z"],
            t["initial_states"])
    assert torch.autograd.gradcheck(f, args, eps=1e-6, atol=1e-7, rtol=1e-6)
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(3))
    g = so.scan_backward(d, dout)
    out = f(*args)
    grads = torch.autograd.grad((out * dout.double()).sum(), args)
    for k, gr in zip(("x", "dt", "A", "B", "C", "dt_bias", "D", "z", "initial_states"), grads):
        assert rel(g[k], gr.numpy()) < TIGHT, k


def test_decay_gradient_by_finite_differences_and_chain_rule():
    """decay_gradient (d loss / d a_t, a_t = dt_t A) matches central finite
    differences of the loss in each a_t, and, since A enters the forward only
    through a = dt A, summing it times dt over the tokens gives the
    backward oracle's dA."""
    d = si.random_small(72, batch=2, seqlen=7, nheads=2, ngroups=1, headdim=3, dstate=2,
                        init_std=0.5, seq_idx_lengths=[3, 4], dt_limit=(0.0, 3.0))
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(4)).double()
    da, dtp = so.decay_gradient(d, dout)
    t = {k: (None if d.get(k) is None else torch.as_tensor(d[k]).double())
         for k in ("x", "dt", "A", "B", "C", "dt_bias", "D", "z", "initial_states")}

    def loss(a):
        out, _ = so.scan_torch(t["x"], t["dt"], t["A"], t["B"], t["C"], dt_bias=t["dt_bias"],
                               D=t["D"], z=t["z"], initial_states=t["initial_states"],
                               seq_idx=d["seq_idx"], dt_limit=(0.0, 3.0), a=a)
        return float((out * dout).sum())
    a0 = torch.from_numpy(dtp) * t["A"]
    eps = 1e-6
    for idx in [(0, 0, 0), (0, 2, 1), (0, 3, 0), (1, 6, 1), (1, 4, 0)]:
        ap, am = a0.clone(), a0.clone()
        ap[idx] += eps
        am[idx] -= eps
        fd = (loss(ap) - loss(am)) / (2 * eps)
        assert abs(fd - da[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, da[idx])
    g = so.scan_backward(d, dout)
    assert rel((da * dtp).sum(axis=(0, 1)), g["A"]) < TIGHT


@pytest.mark.parametrize("kw", [
    dict(batch=2, seqlen=40, nheads=4, ngroups=2, headdim=3, dstate=5, init_std=0.5,
         seq_idx_lengths=[10, 1, 29]),
    dict(batch=1, seqlen=30, nheads=2, ngroups=1, headdim=4, dstate=3, dt_limit=(0.0, 0.5),
         init_std=0.3),
    dict(batch=1, seqlen=25, nheads=2, ngroups=2, headdim=4, dstate=3, has_z=False,
         dt_bias=False),
])
def test_decay_gradient_pairs_sum_to_autograd_dA(kw):
    """dA written as its sum over token pairs (and initial-state terms), each
    term times the dt it spans, equals the autograd oracle's dA; the scale
    (absolute terms) bounds it."""
    d = si.random_small(73, **kw)
    dout = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(5))
    dA, scale = so.decay_gradient_pairs(d, dout)
    ref = so.scan_backward(d, dout)["A"]
    assert rel(dA, ref) < TIGHT
    assert (scale >= np.abs(ref) * (1 - 1e-12)).all()
