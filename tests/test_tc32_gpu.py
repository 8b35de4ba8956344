"""The fp32 stages on the tensor cores (3xTF32 tcgen05, 128-token chunks):
chunk_state and chunk_scan through the forward call and through the stage
exports, against the oracle, for every headdim / dstate combination they
take (and the ones where only chunk_scan does), with documents, initial
states, ragged tails, strided views and the optional inputs missing; and
bf16 inputs of the shapes the fused kernel does not take, which run the same
stages on fp32 copies.  Tolerance: the forward's fp32 bound, max|err| /
max|ref| <= 1e-4 (the 3xTF32 products are within about 2^-22 of fp32 ones),
and the bf16 bound for bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from oracle import ssd_oracle as so
import ssd_inputs as si
from ssd_testutil import TOL, assert_close, run_gpu, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    # (id, headdim, dstate): the first three take both stages on tensor
    # cores, the others chunk_scan only
    ("p64_n128", 64, 128),
    ("p128_n64", 128, 64),
    ("p128_n128", 128, 128),
    ("p64_n64", 64, 64),
    ("p64_n96", 64, 96),
    # two dstate slices: the first token slice loads in the pipeline's first step
    ("p64_n32", 64, 32),
    # the largest dstate chunk_scan takes: 16 slices of C B^T and of the
    # inter-chunk term
    ("p64_n256", 64, 256),
    ("p128_n256", 128, 256),
]

CASES = [
    ("ragged_init_docs", dict(batch=2, seqlen=300, nheads=4, ngroups=2, init_std=0.3,
                              seq_idx_lengths=[130, 1, 169])),
    ("one_chunk_tail", dict(batch=1, seqlen=77, nheads=2, ngroups=1)),
    ("no_optionals", dict(batch=2, seqlen=256, nheads=2, ngroups=2, has_z=False, has_D=False,
                          dt_bias=False)),
    ("docs_on_edges", dict(batch=1, seqlen=512, nheads=2, ngroups=1, init_std=0.5,
                           seq_idx_lengths=[128, 127, 1, 256])),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_forward_fp32_chunk128_matches_oracle(shape, case):
    _, P, N = shape
    name, kw = case
    d = si.random_small(3000 + P + N + len(name), headdim=P, dstate=N, chunk_size=128,
                        dtype="f32", **kw)
    y, f = run_gpu(d)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["f32"], "out")
    assert_close(f, rf, TOL["f32"], "final")


def test_forward_fp32_chunk128_strided_views():
    """x, B, C, z as slices of one projection row per token (strides that
    keep 16-byte rows) take the tensor-core stages and agree with the
    oracle."""
    import selective_state_space_05_gb300 as ssd
    B_, L, H, P, N = 2, 200, 2, 64, 128
    d = si.random_small(3100, batch=B_, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=1,
                        chunk_size=128, dtype="f32", init_std=0.2)
    W = 2 * H * P + 2 * N + 8
    proj = torch.zeros(B_, L, W)
    proj[:, :, :H * P] = d["z"].reshape(B_, L, -1)
    proj[:, :, H * P:2 * H * P] = d["x"].reshape(B_, L, -1)
    proj[:, :, 2 * H * P:2 * H * P + N] = d["B"].reshape(B_, L, -1)
    proj[:, :, 2 * H * P + N:2 * H * P + 2 * N] = d["C"].reshape(B_, L, -1)
    pg = proj.cuda()
    g = to_dev(d)
    z = pg[:, :, :H * P].unflatten(2, (H, P))
    x = pg[:, :, H * P:2 * H * P].unflatten(2, (H, P))
    Bm = pg[:, :, 2 * H * P:2 * H * P + N].unflatten(2, (1, N))
    Cm = pg[:, :, 2 * H * P + N:2 * H * P + 2 * N].unflatten(2, (1, N))
    y, f = ssd.ssd_scan_fwd(x, g["dt"], g["A"], Bm, Cm, chunk_size=128, dt_bias=g["dt_bias"],
                            D=g["D"], z=z, initial_states=g["initial_states"],
                            return_final_states=True, check=True)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y.double().cpu().numpy(), ry, TOL["f32"], "out")
    assert_close(f.double().cpu().numpy(), rf, TOL["f32"], "final")


# the stage exports compute C B^T inside chunk_scan (dstate 256: 40 slices)
STAGE_SHAPES = SHAPES[:3] + [("p64_n256", 64, 256)]


@pytest.mark.parametrize("shape", STAGE_SHAPES, ids=[s[0] for s in STAGE_SHAPES])
def test_stage_exports_fp32_chunk128_match_chunked_oracle(shape):
    """ssd_chunk_state and ssd_chunk_scan at chunk 128 in fp32 (the
    tensor-core kernels; chunk_state on the SIMT kernel for dstate 256)
    against the chunked oracle's intermediates."""
    import selective_state_space_05_gb300 as ssd
    _, P, N = shape
    Q = 128
    d = si.random_small(3200 + P + N, batch=2, seqlen=333, nheads=4, ngroups=2, headdim=P,
                        dstate=N, chunk_size=Q, dtype="f32", init_std=0.3,
                        seq_idx_lengths=[100, 1, 232])
    ry, rf, im = so.scan_chunked(d, Q, return_intermediates=True)
    g = to_dev(d)
    L = d["x"].shape[1]
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"],
                                        seq_idx=g["seq_idx"])
    states = ssd.ssd_chunk_state(g["x"], g["B"], dt_out, cs, seg, chunk_size=Q)
    assert_close(states.double().cpu().numpy(), im["states"], TOL["f32"], "chunk states")
    fin = ssd.ssd_state_passing(states, cs, seg, seqlen=L, chunk_size=Q,
                                initial_states=g["initial_states"])
    out = ssd.ssd_chunk_scan(g["x"], g["B"], g["C"], dt_out, cs, seg, states, chunk_size=Q,
                             D=g["D"], z=g["z"])
    torch.cuda.synchronize()
    assert_close(out.double().cpu().numpy(), ry, TOL["f32"], "out")
    assert_close(fin.double().cpu().numpy(), rf, TOL["f32"], "final")


def test_forward_fp32_tc_status_clean():
    """A tensor-core fp32 launch leaves the status word clear (no wait gave up)."""
    import selective_state_space_05_gb300 as ssd
    d = si.random_small(3300, batch=1, seqlen=256, nheads=2, headdim=64, dstate=128, ngroups=1,
                        chunk_size=128, dtype="f32")
    g = to_dev(d)
    ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=128,
                     dt_bias=g["dt_bias"], D=g["D"], z=g["z"], check=True)
    ssd.scan_status()


def test_tc32_timeout_is_reported(monkeypatch):
    """A test-only launch option leaves the first slice of the first CTA
    uncommitted, so that its buffer's mbarrier never completes: the bounded
    wait (shortened to 0.2 s) gives up, the CTA ends without touching the
    accumulators, and ssd_scan_status reports SSD_ERR_TIMEOUT.  The next
    normal launch is correct again."""
    import selective_state_space_05_gb300 as ssd
    from selective_state_space_05_gb300._lib import SSD_ERR_TIMEOUT, SSDError
    d = si.random_small(3400, batch=1, seqlen=256, nheads=2, headdim=64, dstate=128, ngroups=1,
                        chunk_size=128, dtype="f32")
    g = to_dev(d)
    ssd.scan_status(reset=True)
    monkeypatch.setenv("SSD_TC32_WAIT_NS", "200000000")
    monkeypatch.setenv("SSD_TC32_TEST_STALL", "1")
    ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=128,
                     dt_bias=g["dt_bias"], D=g["D"], z=g["z"])
    with pytest.raises(SSDError) as ei:
        ssd.scan_status(reset=True)
    assert ei.value.code == SSD_ERR_TIMEOUT
    assert "8 fp32 tensor-core stage" in str(ei.value)
    ssd.scan_status(reset=True)                      # cleared
    monkeypatch.delenv("SSD_TC32_TEST_STALL")
    monkeypatch.delenv("SSD_TC32_WAIT_NS")
    y, f = run_gpu(d)
    ssd.scan_status(reset=True)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["f32"], "out after the time-out")
    assert_close(f, rf, TOL["f32"], "final after the time-out")


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_forward_bf16_through_fp32_stages(shape, case):
    """bf16 shapes the fused kernel does not take (headdim 128, dstate other
    than 128, an odd number of heads per group) run the fp32 tensor-core
    stages on exact fp32 copies of their inputs, out rounded to bf16 once
    (chunk 256, run at 128); the others run the fused kernel.  bf16 bound."""
    _, P, N = shape
    name, kw = case
    d = si.random_small(3500 + P + N + len(name), headdim=P, dstate=N, chunk_size=256,
                        dtype="bf16", **kw)
    y, f = run_gpu(d)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["bf16"], "out")
    assert_close(f, rf, TOL["bf16"], "final")


def _proj_views(d, H, P, N, extra):
    """x, z, B, C of d as slices of one projection row per token, the row
    `extra` elements longer than the four (a token stride of any length)."""
    B_, L = d["x"].shape[:2]
    W = 2 * H * P + 2 * N + extra
    proj = torch.zeros(B_, L, W, dtype=d["x"].dtype)
    proj[:, :, :H * P] = d["z"].reshape(B_, L, -1)
    proj[:, :, H * P:2 * H * P] = d["x"].reshape(B_, L, -1)
    proj[:, :, 2 * H * P:2 * H * P + N] = d["B"].reshape(B_, L, -1)
    proj[:, :, 2 * H * P + N:2 * H * P + 2 * N] = d["C"].reshape(B_, L, -1)
    pg = proj.cuda()
    return (pg[:, :, H * P:2 * H * P].unflatten(2, (H, P)), pg[:, :, :H * P].unflatten(2, (H, P)),
            pg[:, :, 2 * H * P:2 * H * P + N].unflatten(2, (1, N)),
            pg[:, :, 2 * H * P + N:2 * H * P + 2 * N].unflatten(2, (1, N)))


@pytest.mark.parametrize("extra", [8, 3], ids=["stride_x8", "stride_odd"])
def test_forward_bf16_through_fp32_stages_strided(extra):
    """Strided bf16 views (slices of a projection row) into the fp32 copies:
    16-byte loads when the token stride is a multiple of 8 elements, one
    element at a time otherwise."""
    import selective_state_space_05_gb300 as ssd
    H, P, N = 2, 128, 64
    d = si.random_small(3600 + extra, batch=2, seqlen=200, nheads=H, headdim=P, dstate=N,
                        ngroups=1, chunk_size=256, dtype="bf16", init_std=0.2)
    x, z, Bm, Cm = _proj_views(d, H, P, N, extra)
    g = to_dev(d)
    y, f = ssd.ssd_scan_fwd(x, g["dt"], g["A"], Bm, Cm, chunk_size=256, dt_bias=g["dt_bias"],
                            D=g["D"], z=z, initial_states=g["initial_states"],
                            return_final_states=True, check=True)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y.double().cpu().numpy(), ry, TOL["bf16"], "out")
    assert_close(f.double().cpu().numpy(), rf, TOL["bf16"], "final")


def test_forward_bf16_least_workspace_runs_stage_kernels():
    """A workspace of ssd_scan_workspace_bytes_min has no room for the fp32
    copies: the same bf16 call then runs the bf16 stage kernels, and agrees
    with the oracle (and, to bf16 rounding, with the call on the full
    workspace)."""
    import selective_state_space_05_gb300 as ssd
    H, P, N, Q = 4, 128, 64, 256
    d = si.random_small(3700, batch=2, seqlen=300, nheads=H, headdim=P, dstate=N, ngroups=2,
                        chunk_size=Q, dtype="bf16", init_std=0.3, seq_idx_lengths=[120, 180])
    g = to_dev(d)
    full = ssd.workspace_bytes(2, 300, H, P, N, 2, Q, torch.bfloat16)
    least = ssd.workspace_bytes(2, 300, H, P, N, 2, Q, torch.bfloat16, least=True)
    assert 0 < least < full
    outs = []
    for nbytes in (least, full):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        y, f = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=Q,
                                dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                                initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                                return_final_states=True, workspace=ws, check=True)
        outs.append((y.double().cpu().numpy(), f.double().cpu().numpy()))
    ry, rf = oracle.scan_sequential(d)
    for y, f in outs:
        assert_close(y, ry, TOL["bf16"], "out")
        assert_close(f, rf, TOL["bf16"], "final")
