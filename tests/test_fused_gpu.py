"""GPU parity of the fused tensor-core path (bf16, headdim 64, dstate 128,
chunk 128 / 256, an even number of heads per group): ssd_scan_fwd routes
these shapes to the fused tcgen05 kernel, which also runs stage 1.
Compared with the fp64 oracle (max|err|/max|ref| <= 2e-2) and with the four
SIMT stage kernels; the kernel's error word must stay 0."""
import math

import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from ssd_testutil import TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _run_fused(d, chunk, check_error_word=True):
    import selective_state_space_05_gb300 as ssd
    g = to_dev(d)
    Bsz, L, H, P = g["x"].shape
    G, N = g["B"].shape[2], g["B"].shape[3]
    ws = torch.empty(ssd.workspace_bytes(Bsz, L, H, P, N, G, chunk), dtype=torch.uint8,
                     device="cuda")
    out, fin = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=chunk,
                                dt_bias=g["dt_bias"], dt_softplus=d.get("dt_softplus", True),
                                dt_limit=d.get("dt_limit", (0.0, math.inf)), D=g["D"], z=g["z"],
                                initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                                return_final_states=True, workspace=ws)
    torch.cuda.synchronize()
    if check_error_word:
        assert int(ws[4:8].view(torch.int32).item()) == 0, "fused kernel gave up a wait"
    return out.double().cpu().numpy(), fin.double().cpu().numpy()


def _small(seed, **kw):
    base = dict(batch=2, nheads=4, ngroups=2, headdim=64, dstate=128, dtype="bf16")
    base.update(kw)
    return si.random_small(seed, **base)


CASES = [
    ("L1_q128", dict(seqlen=1, chunk_size=128)),
    ("L100_q128", dict(seqlen=100, chunk_size=128)),
    ("L128_q128", dict(seqlen=128, chunk_size=128)),
    ("L129_q128", dict(seqlen=129, chunk_size=128)),
    ("L255_q256", dict(seqlen=255, chunk_size=256)),
    ("L256_q256", dict(seqlen=256, chunk_size=256)),
    ("L257_q256", dict(seqlen=257, chunk_size=256)),
    ("L700_q256_init", dict(seqlen=700, chunk_size=256, init_std=0.5)),
    ("L1000_q128_init_G1", dict(seqlen=1000, chunk_size=128, ngroups=1, init_std=0.5)),
    ("docs_on_sub_edges", dict(seqlen=640, chunk_size=256, init_std=0.3,
                               seq_idx_lengths=[128, 128, 1, 127, 256])),
    ("docs_inside_subs", dict(seqlen=600, chunk_size=256, init_std=0.3,
                              seq_idx_lengths=[5, 200, 1, 1, 300, 93])),
    ("no_z_no_D", dict(seqlen=300, chunk_size=256, has_z=False, has_D=False)),
    ("slow_decay", dict(seqlen=1024, chunk_size=128, init_std=0.5,
                        a_log_range=(math.log(1e-3), math.log(1e-1)))),
    ("many_heads", dict(seqlen=512, chunk_size=256, nheads=16, ngroups=4, batch=3)),
    # without dt_bias dt is about 0.7: a 32-token block decays by 2^40 to 2^600,
    # so the diagonal blocks take both the factored and the per-element form
    ("strong_decay_mixed", dict(seqlen=600, chunk_size=256, dt_bias=False, init_std=0.3,
                                a_log_range=(0.0, math.log(4.0)),
                                seq_idx_lengths=[250, 1, 349])),
    ("strong_decay", dict(seqlen=300, chunk_size=128, dt_bias=False, init_std=0.3)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_oracle(case):
    _, kw = case
    d = _small(3000 + len(case[0]), **kw)
    y, f = _run_fused(d, kw["chunk_size"])
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["bf16"], "out")
    assert_close(f, rf, TOL["bf16"], "final")


def test_fused_matches_simt_stages():
    """Same inputs through the fused kernel and through the four SIMT stage
    kernels (which the fp32 path uses)."""
    import selective_state_space_05_gb300 as ssd
    Q = 256
    d = _small(41, seqlen=1500, chunk_size=Q, init_std=0.3, seq_idx_lengths=[700, 800])
    y_f, f_f = _run_fused(d, Q)
    g = to_dev(d)
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"],
                                        seq_idx=g["seq_idx"])
    st = ssd.ssd_chunk_state(g["x"], g["B"], dt_out, cs, seg, chunk_size=Q)
    fin = ssd.ssd_state_passing(st, cs, seg, seqlen=1500, chunk_size=Q,
                                initial_states=g["initial_states"])
    y_s = ssd.ssd_chunk_scan(g["x"], g["B"], g["C"], dt_out, cs, seg, st, chunk_size=Q,
                             D=g["D"], z=g["z"])
    torch.cuda.synchronize()
    assert_close(y_f, y_s.double().cpu().numpy(), TOL["bf16"], "out fused vs SIMT")
    assert_close(f_f, fin.double().cpu().numpy(), TOL["bf16"], "final fused vs SIMT")


def test_fused_stage_entry_point():
    """ssd_chunk_fused called on its own after ssd_dt_cumsum."""
    import selective_state_space_05_gb300 as ssd
    Q = 128
    d = _small(42, seqlen=777, chunk_size=Q, init_std=0.2)
    g = to_dev(d)
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"])
    ws = torch.empty(ssd.workspace_bytes(2, 777, 4, 64, 128, 2, Q), dtype=torch.uint8,
                     device="cuda")
    y, f = ssd.ssd_chunk_fused(g["x"], g["B"], g["C"], dt_out, cs, seg, chunk_size=Q,
                               workspace=ws, D=g["D"], z=g["z"],
                               initial_states=g["initial_states"], return_final_states=True)
    torch.cuda.synchronize()
    ry, rf = oracle.scan_sequential(d)
    assert_close(y.double().cpu().numpy(), ry, TOL["bf16"], "out")
    assert_close(f.double().cpu().numpy(), rf, TOL["bf16"], "final")


def test_fused_long_lookback_chain():
    """Many chunks per sequence and more work items than resident CTAs."""
    d = _small(43, batch=4, seqlen=8192, nheads=32, ngroups=4, chunk_size=256, init_std=0.2)
    y, f = _run_fused(d, 256)
    heads = [0, 9, 31]
    ry, rf = oracle.scan_sequential(d, heads=heads, batches=[0, 3])
    assert_close(y[[0, 3]][:, :, heads], ry, TOL["bf16"], "out (sampled)")
    assert_close(f[[0, 3]][:, heads], rf, TOL["bf16"], "final (sampled)")


def test_fused_rejects_other_shapes():
    import selective_state_space_05_gb300 as ssd
    from selective_state_space_05_gb300._lib import SSDError
    d = to_dev(si.random_small(44, headdim=32, dstate=128, dtype="bf16", seqlen=64,
                               chunk_size=128))
    dt_out, cs, seg = ssd.ssd_dt_cumsum(d["dt"], d["A"], chunk_size=128)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(SSDError, match="headdim 64"):
        ssd.ssd_chunk_fused(d["x"], d["B"], d["C"], dt_out, cs, seg, chunk_size=128, workspace=ws)


def test_fused_rejects_odd_heads_per_group():
    """The kernel pairs the heads of a group; an odd count is refused."""
    import selective_state_space_05_gb300 as ssd
    from selective_state_space_05_gb300._lib import SSDError
    d = to_dev(si.random_small(45, nheads=3, ngroups=1, headdim=64, dstate=128, dtype="bf16",
                               seqlen=200, chunk_size=128))
    dt_out, cs, seg = ssd.ssd_dt_cumsum(d["dt"], d["A"], chunk_size=128)
    ws = torch.empty(ssd.workspace_bytes(2, 200, 3, 64, 128, 1, 128), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(SSDError, match="even number of heads"):
        ssd.ssd_chunk_fused(d["x"], d["B"], d["C"], dt_out, cs, seg, chunk_size=128, workspace=ws)


def test_scan_fwd_odd_heads_per_group_takes_stage_kernels():
    """ssd_scan_fwd still serves such shapes, through the four stage kernels."""
    d = _small(46, seqlen=300, chunk_size=256, nheads=3, ngroups=1, init_std=0.3)
    y, f = _run_fused(d, 256, check_error_word=False)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["bf16"], "out")
    assert_close(f, rf, TOL["bf16"], "final")


@pytest.mark.parametrize("seg", [1, 2, 3, 4])
def test_fused_segments(seg, monkeypatch):
    """The state stays on chip across a segment of chunks and is handed on
    between segments; every segment length (ragged last segment included)
    gives the same result."""
    monkeypatch.setenv("SSD_FUSED_SEGMENT_CHUNKS", str(seg))
    d = _small(47, batch=2, seqlen=1800, nheads=4, ngroups=2, chunk_size=128, init_std=0.3,
               seq_idx_lengths=[700, 1100])
    y, f = _run_fused(d, 128)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["bf16"], f"out (segments of {seg})")
    assert_close(f, rf, TOL["bf16"], f"final (segments of {seg})")


def _run_raw(g, chunk):
    """The fused path on device inputs; out and final states as device tensors."""
    import selective_state_space_05_gb300 as ssd
    Bsz, L, H, P = g["x"].shape
    G, N = g["B"].shape[2], g["B"].shape[3]
    ws = torch.empty(ssd.workspace_bytes(Bsz, L, H, P, N, G, chunk), dtype=torch.uint8,
                     device="cuda")
    out, fin = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=chunk,
                                dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                                initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                                return_final_states=True, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[4:8].view(torch.int32).item()) == 0, "fused kernel gave up a wait"
    return out, fin


@pytest.mark.parametrize("shape", [
    dict(batch=2, seqlen=1800, nheads=4, ngroups=2, chunk_size=128,
         seq_idx_lengths=[700, 1100]),
    dict(batch=4, seqlen=8192, nheads=32, ngroups=4, chunk_size=256),
    dict(batch=8, seqlen=1000, nheads=40, ngroups=4, chunk_size=256,
         seq_idx_lengths=[300, 1, 699]),
], ids=["docs_15_chunks", "32_chunks", "160_pairs_ragged"])
def test_fused_segment_lengths_bit_identical(shape, monkeypatch):
    """The hand-off between segments is an exact fp32 copy of the state
    (TMEM -> slot -> TMEM), so the segment length changes nothing in the
    result, bit for bit, down to one segment per sequence (no hand-off at
    all); the result also matches the oracle on sampled heads."""
    d = _small(48, init_std=0.3, **shape)
    g = to_dev(d)
    Q = shape["chunk_size"]
    nc = -(-shape["seqlen"] // Q)
    monkeypatch.setenv("SSD_FUSED_PREPASS", "0")   # the hand-off between segments
    monkeypatch.setenv("SSD_FUSED_SEGMENT_CHUNKS", "1")
    y_1, f_1 = _run_raw(g, Q)
    for seg in sorted({2, 3, nc} - {1}):
        if seg > nc:
            continue
        monkeypatch.setenv("SSD_FUSED_SEGMENT_CHUNKS", str(seg))
        y_s, f_s = _run_raw(g, Q)
        assert torch.equal(y_1, y_s), f"out: segments of 1 vs {seg}"
        assert torch.equal(f_1, f_s), f"final: segments of 1 vs {seg}"
    H = shape["nheads"]
    heads, batches = sorted({0, H // 2 + 1, H - 1}), sorted({0, shape["batch"] - 1})
    ry, rf = oracle.scan_sequential(d, heads=heads, batches=batches)
    y = y_1.double().cpu().numpy()[batches][:, :, heads]
    f = f_1.double().cpu().numpy()[batches][:, heads]
    assert_close(y, ry, TOL["bf16"], "out (sampled)")
    assert_close(f, rf, TOL["bf16"], "final (sampled)")


# --------------------------------------------------------------------------
# stage-1 options on the fused path: the dt clamp and softplus off (dt used
# as given, which may be negative; the kernel then runs its signed-dt form)
# --------------------------------------------------------------------------

def _signed_dt(d, scale, seed):
    g = torch.Generator().manual_seed(seed)
    d["dt"] = (torch.randn(d["dt"].shape, generator=g) * scale).to(d["dt"].dtype)
    return d


DT_OPTION_CASES = [
    # (id, random_small kwargs, dt rewrite)
    ("limit_0.02_0.3", dict(seqlen=700, chunk_size=256, init_std=0.3, dt_limit=(0.02, 0.3),
                            seq_idx_lengths=[300, 400]), None),
    # the ceiling binds on most tokens (softplus of the biased dt is about 0.7 without bias)
    ("limit_0_0.05_mostly_clamped", dict(seqlen=600, chunk_size=128, dt_bias=False,
                                         dt_limit=(0.0, 0.05), init_std=0.3), None),
    # softplus off, default limit: dt used as given (here non-negative), signed form
    ("no_softplus_nonneg", dict(seqlen=500, chunk_size=256, dt_softplus=False, dt_bias=False,
                                init_std=0.3), "abs"),
    # softplus off with a non-negative clamp floor: the unsigned form
    ("no_softplus_clamped", dict(seqlen=500, chunk_size=128, dt_softplus=False, dt_bias=False,
                                 dt_limit=(0.0, 1.0), seq_idx_lengths=[200, 1, 299]), "signed"),
    # softplus off, negative dt on about half the tokens: the state grows there
    ("no_softplus_signed", dict(seqlen=640, chunk_size=256, dt_softplus=False, dt_bias=False,
                                init_std=0.3, a_log_range=(0.0, math.log(4.0)),
                                seq_idx_lengths=[128, 300, 212]), "signed"),
    ("no_softplus_signed_q128", dict(seqlen=1000, chunk_size=128, dt_softplus=False,
                                     dt_bias=False, ngroups=1, nheads=4,
                                     a_log_range=(0.0, math.log(2.0))), "signed"),
]


@pytest.mark.parametrize("case", DT_OPTION_CASES, ids=[c[0] for c in DT_OPTION_CASES])
def test_fused_dt_options(case):
    name, kw, rewrite = case
    d = _small(3100 + len(name), **kw)
    if rewrite == "abs":
        d["dt"] = (d["dt"].float().abs() * 0.2).to(d["dt"].dtype)
    elif rewrite == "signed":
        d = _signed_dt(d, 0.05, 3200 + len(name))
    y, f = _run_fused(d, kw["chunk_size"])
    ry, rf = oracle.scan_sequential(d)
    assert np.isfinite(ry).all() and np.abs(ry).max() < 1e30
    assert_close(y, ry, TOL["bf16"], "out")
    assert_close(f, rf, TOL["bf16"], "final")


def test_fused_stage_entry_point_signed_dt():
    """ssd_chunk_fused takes caller-given stage-1 outputs as possibly negative."""
    import selective_state_space_05_gb300 as ssd
    Q = 256
    d = _signed_dt(_small(49, seqlen=700, chunk_size=Q, dt_softplus=False, dt_bias=False,
                          init_std=0.2), 0.05, 50)
    g = to_dev(d)
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_softplus=False)
    ws = torch.empty(ssd.workspace_bytes(2, 700, 4, 64, 128, 2, Q), dtype=torch.uint8,
                     device="cuda")
    y, f = ssd.ssd_chunk_fused(g["x"], g["B"], g["C"], dt_out, cs, seg, chunk_size=Q,
                               workspace=ws, D=g["D"], z=g["z"],
                               initial_states=g["initial_states"], return_final_states=True)
    ssd.scan_status(reset=True)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y.double().cpu().numpy(), ry, TOL["bf16"], "out")
    assert_close(f.double().cpu().numpy(), rf, TOL["bf16"], "final")


# --------------------------------------------------------------------------
# a wait that gives up: reported through the status word, context still usable
# --------------------------------------------------------------------------

def test_fused_timeout_is_reported(monkeypatch):
    """A hand-off flag value that nothing ever writes (a test-only launch
    option) makes the look-back wait of every later segment run out after
    the shortened limit of 0.2 s; the kernel then stops every role, lets its
    copies and MMAs in flight finish and ends.  The status word says so, and
    the next normal launch is correct again."""
    import selective_state_space_05_gb300 as ssd
    from selective_state_space_05_gb300._lib import SSD_ERR_TIMEOUT, SSDError
    d = _small(51, batch=2, seqlen=1024, nheads=4, ngroups=2, chunk_size=128, init_std=0.3)
    g = to_dev(d)
    ws = torch.empty(ssd.workspace_bytes(2, 1024, 4, 64, 128, 2, 128), dtype=torch.uint8,
                     device="cuda")
    ssd.scan_status(reset=True)
    monkeypatch.setenv("SSD_FUSED_PREPASS", "0")   # segments wait for their predecessors
    monkeypatch.setenv("SSD_FUSED_SEGMENT_CHUNKS", "1")
    monkeypatch.setenv("SSD_FUSED_WAIT_NS", "200000000")
    monkeypatch.setenv("SSD_FUSED_TEST_STALL", "1")
    ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=128,
                     dt_bias=g["dt_bias"], D=g["D"], z=g["z"], workspace=ws)
    with pytest.raises(SSDError) as ei:
        ssd.scan_status(reset=False)
    assert ei.value.code == SSD_ERR_TIMEOUT
    assert int(ws[4:8].view(torch.int32).item()) & 2, "the hand-off wait should have given up"
    with pytest.raises(SSDError):
        ssd.scan_status(reset=True)                  # still set, then cleared
    ssd.scan_status(reset=True)                      # clear
    monkeypatch.delenv("SSD_FUSED_TEST_STALL")
    monkeypatch.delenv("SSD_FUSED_WAIT_NS")
    y, f = _run_fused(d, 128)
    ssd.scan_status(reset=True)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["bf16"], "out after the time-out")
    assert_close(f, rf, TOL["bf16"], "final after the time-out")


# --------------------------------------------------------------------------
# state pre-pass (few head pairs, many chunks): segment states first, then
# the states entering each segment, then the main kernel without hand-off
# --------------------------------------------------------------------------

PREPASS_CASES = [
    ("docs_init_q128", dict(batch=1, nheads=4, ngroups=2, seqlen=3000, chunk_size=128,
                            init_std=0.3, seq_idx_lengths=[1000, 1, 1200, 799]), None),
    ("docs_on_chunk_edges", dict(batch=1, nheads=2, ngroups=1, seqlen=2500, chunk_size=128,
                                 init_std=0.3, seq_idx_lengths=[256, 1024, 128, 1092]), None),
    ("two_rows_q256", dict(batch=2, nheads=8, ngroups=1, seqlen=4096, chunk_size=256,
                           init_std=0.2), None),
    ("slow_decay", dict(batch=1, nheads=4, ngroups=2, seqlen=2048, chunk_size=128,
                        init_std=0.5, a_log_range=(math.log(1e-3), math.log(1e-1))), None),
    ("signed_dt", dict(batch=1, nheads=4, ngroups=1, seqlen=2048, chunk_size=256,
                       dt_softplus=False, dt_bias=False, init_std=0.3,
                       a_log_range=(0.0, math.log(2.0)), seq_idx_lengths=[900, 1148]), "signed"),
]


@pytest.mark.parametrize("seg", ["auto", "3", "5"])
@pytest.mark.parametrize("case", PREPASS_CASES, ids=[c[0] for c in PREPASS_CASES])
def test_fused_prepass_matches_oracle(case, seg, monkeypatch):
    name, kw, rewrite = case
    monkeypatch.setenv("SSD_FUSED_PREPASS", "1")
    if seg != "auto":
        monkeypatch.setenv("SSD_FUSED_SEGMENT_CHUNKS", seg)
    d = _small(3300 + len(name), **kw)
    if rewrite == "signed":
        d = _signed_dt(d, 0.05, 3400 + len(name))
    y, f = _run_fused(d, kw["chunk_size"])
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["bf16"], f"out ({seg})")
    assert_close(f, rf, TOL["bf16"], f"final ({seg})")


def test_fused_prepass_agrees_with_handoff(monkeypatch):
    """The two ways of carrying the state between segments give the same
    result up to the rounding of the state sums."""
    d = _small(52, batch=1, nheads=8, ngroups=2, seqlen=4000, chunk_size=256, init_std=0.3,
               seq_idx_lengths=[1500, 2500])
    monkeypatch.setenv("SSD_FUSED_SEGMENT_CHUNKS", "4")
    monkeypatch.setenv("SSD_FUSED_PREPASS", "0")
    y0, f0 = _run_fused(d, 256)
    monkeypatch.setenv("SSD_FUSED_PREPASS", "1")
    y1, f1 = _run_fused(d, 256)
    assert_close(y1, y0, 5e-3, "out: pre-pass vs hand-off")
    assert_close(f1, f0, 5e-3, "final: pre-pass vs hand-off")


@pytest.mark.parametrize("Q", [128, 256])
def test_chunk_state_stage_on_tensor_cores(Q):
    """ssd_chunk_state routes the bf16 headdim-64 / dstate-128 shapes to the
    tensor-core segment-state kernel (one chunk per segment)."""
    import selective_state_space_05_gb300 as ssd
    from oracle import ssd_oracle as so
    d = _small(53 + Q, batch=2, nheads=4, ngroups=2, seqlen=700, chunk_size=Q,
               seq_idx_lengths=[300, 1, 399])
    g = to_dev(d)
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"],
                                        seq_idx=g["seq_idx"])
    st = ssd.ssd_chunk_state(g["x"], g["B"], dt_out, cs, seg, chunk_size=Q)
    torch.cuda.synchronize()
    _, _, im = so.scan_chunked(d, Q, return_intermediates=True)
    assert_close(st.double().cpu().numpy(), im["states"], TOL["bf16"], "chunk states")


@pytest.mark.parametrize("Q", [128, 256])
def test_four_stage_exports_on_tensor_cores(Q):
    """The four stage calls one by one on the Mamba-2 shape: chunk_state and
    chunk_scan run on tensor cores (the segment-state kernel with one chunk
    per segment; the fused kernel reading stage 3's prev_states), state
    passing on CUDA cores; each intermediate against the oracle's chunked
    form and the result against the recurrence."""
    import selective_state_space_05_gb300 as ssd
    from oracle import ssd_oracle as so
    d = _small(60 + Q, batch=2, nheads=4, ngroups=2, seqlen=900, chunk_size=Q, init_std=0.3,
               seq_idx_lengths=[256, 1, 400, 243])
    g = to_dev(d)
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"],
                                        seq_idx=g["seq_idx"])
    st = ssd.ssd_chunk_state(g["x"], g["B"], dt_out, cs, seg, chunk_size=Q)
    ry, rf, im = so.scan_chunked(d, Q, return_intermediates=True)
    assert_close(st.double().cpu().numpy(), im["states"], TOL["bf16"], "chunk states")
    fin = ssd.ssd_state_passing(st, cs, seg, seqlen=900, chunk_size=Q,
                                initial_states=g["initial_states"])
    assert_close(st.double().cpu().numpy(), im["prev_states"], TOL["bf16"], "prev states")
    y = ssd.ssd_chunk_scan(g["x"], g["B"], g["C"], dt_out, cs, seg, st, chunk_size=Q,
                           D=g["D"], z=g["z"])
    torch.cuda.synchronize()
    ssd.scan_status(reset=True)
    assert_close(y.double().cpu().numpy(), ry, TOL["bf16"], "out")
    assert_close(fin.double().cpu().numpy(), rf, TOL["bf16"], "final")
