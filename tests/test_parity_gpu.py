"""GPU parity: the CUDA path (called through the C ABI) against the fp64 CPU
oracle on the same seeded inputs.

Bar: max|err| / max|ref| <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs
(fp32 accumulation and state); mean errors are reported with every failure,
because SSD kernel errors can be heavy-tailed.  Integer work (the per-chunk
segment counts) is compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from oracle import ssd_oracle as so
from ssd_testutil import (PARITY_REPORT, TOL, ErrorStats, assert_close, errors, run_gpu,
                          to_dev)

pytestmark = pytest.mark.gpu


# --------------------------------------------------------------------------
# small and medium workloads: whole outputs against the oracle
# --------------------------------------------------------------------------

def test_tiny_fp32():
    cfg = si.CONFIGS["tiny"]
    d = si.make_inputs(cfg, 1000)
    y, f = run_gpu(d)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["f32"], "out")
    assert_close(f, rf, TOL["f32"], "final")


@pytest.mark.parametrize("name", ["grouped_g1", "grouped_g2", "grouped_g4"])
@pytest.mark.parametrize("with_D", [True, False])
def test_grouped_fp32(name, with_D):
    """D_h = 1000 h dominates max|ref| and could hide scan errors, so the same
    inputs are also checked with D absent."""
    d = si.make_inputs(si.CONFIGS[name], 1001)
    if not with_D:
        d["D"] = None
    y, f = run_gpu(d)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["f32"], "out")
    assert_close(f, rf, TOL["f32"], "final")


EDGE = [
    # (id, kwargs for random_small)
    ("ragged_tail", dict(seqlen=200, chunk_size=64)),
    ("len1", dict(seqlen=1, chunk_size=16)),
    ("shorter_than_chunk", dict(seqlen=50, chunk_size=256)),
    ("docs_on_chunk_edges", dict(seqlen=192, chunk_size=64, seq_idx_lengths=[64, 63, 1, 64])),
    ("docs_off_edges", dict(seqlen=192, chunk_size=64, seq_idx_lengths=[65, 1, 1, 60, 65])),
    ("many_len1_docs", dict(seqlen=40, chunk_size=16, seq_idx_lengths=[1] * 20 + [20])),
    ("init_and_docs", dict(seqlen=300, chunk_size=128, init_std=0.5,
                           seq_idx_lengths=[130, 1, 169])),
    ("slow_decay", dict(seqlen=512, chunk_size=64, init_std=0.5,
                        a_log_range=(math.log(1e-3), math.log(1e-1)))),
    ("no_z_no_D_no_bias", dict(has_z=False, has_D=False, dt_bias=False, seqlen=100)),
    # without softplus dt is used as given: keep it non-negative so that the
    # state decays (a negative dt makes it grow like e^(hundreds), beyond fp32)
    ("no_softplus", dict(dt_softplus=False, dt_bias=False, a_log_range=(-3.0, 0.0),
                         seqlen=100)),
    ("dt_limit", dict(dt_limit=(0.02, 0.3), seqlen=100)),
    ("groups_8", dict(nheads=16, ngroups=8, seqlen=130, chunk_size=32)),
    ("hd16_ds16", dict(headdim=16, dstate=16, seqlen=77)),
    ("hd32_ds48", dict(headdim=32, dstate=48, seqlen=77, chunk_size=32)),
    ("hd128_ds256", dict(headdim=128, dstate=256, seqlen=150, chunk_size=64, nheads=2,
                         ngroups=1)),
    ("hd64_ds128_q256", dict(headdim=64, dstate=128, seqlen=700, chunk_size=256, init_std=0.3,
                             seq_idx_lengths=[300, 400])),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_edge_cases(case, dtype):
    _, kw = case
    kw = dict(kw)
    kw.setdefault("headdim", 16)
    kw.setdefault("dstate", 32)
    d = si.random_small(2000 + len(case[0]), dtype=dtype, **kw)
    if not kw.get("dt_softplus", True):
        d["dt"] = (d["dt"].float().abs() * 0.2).to(d["dt"].dtype)
    y, f = run_gpu(d)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL[dtype], "out")
    assert_close(f, rf, TOL[dtype], "final")


@pytest.mark.parametrize("Q", [16, 32, 64, 128, 256])
def test_chunk_size_invariance_on_gpu(Q):
    d = si.random_small(77, seqlen=333, headdim=32, dstate=64, init_std=0.3,
                        seq_idx_lengths=[100, 33, 200])
    y, f = run_gpu(d, chunk_size=Q)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["f32"], "out")
    assert_close(f, rf, TOL["f32"], "final")


def test_no_writes_outside_out():
    """out placed inside a larger buffer filled with a sentinel: a ragged tail
    must not write past the last token."""
    d = si.random_small(5, seqlen=131, chunk_size=64, headdim=16, dstate=16)
    n = d["x"].numel()
    buf = torch.full((n + 4096,), float("nan"), device="cuda")
    out = buf[1024:1024 + n].view(d["x"].shape)
    y, _ = run_gpu(d, out=out, final=False)
    assert torch.isnan(buf[:1024]).all() and torch.isnan(buf[1024 + n:]).all()
    ry, _ = oracle.scan_sequential(d)
    assert_close(y, ry, TOL["f32"], "out")


def test_repeat_calls_identical():
    d = si.random_small(6, seqlen=257, headdim=64, dstate=128, dtype="bf16", chunk_size=128)
    y1, f1 = run_gpu(d)
    y2, f2 = run_gpu(d)
    assert np.array_equal(y1, y2) and np.array_equal(f1, f2)


def test_binding_rejects_bad_sizes():
    import selective_state_space_05_gb300 as ssd
    from selective_state_space_05_gb300._lib import SSDError
    d = to_dev(si.random_small(7, seqlen=64))
    with pytest.raises(SSDError, match="chunk_size"):
        ssd.ssd_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk_size=48)


# --------------------------------------------------------------------------
# stage by stage, against the oracle's chunked form
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_stages_match_chunked_oracle(dtype):
    import selective_state_space_05_gb300 as ssd
    Q = 64
    d = si.random_small(8, batch=2, seqlen=300, nheads=4, ngroups=2, headdim=32, dstate=64,
                        chunk_size=Q, dtype=dtype, init_std=0.3,
                        seq_idx_lengths=[64, 100, 1, 135])
    ry, rf, im = so.scan_chunked(d, Q, return_intermediates=True)
    g = to_dev(d)
    L = d["x"].shape[1]
    dt_out, cs, seg = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"],
                                        seq_idx=g["seq_idx"])
    # stage 1: dt and cumsum over the valid positions
    nc = cs.shape[2]
    valid = np.zeros((nc, Q), dtype=bool)
    valid.reshape(-1)[:L] = True
    dt_ref = np.zeros((2, 4, nc * Q))
    dt_ref[:, :, :L] = im["dt"].transpose(0, 2, 1)
    assert_close(dt_out.double().cpu().numpy()[:, :, valid], dt_ref.reshape(2, 4, nc, Q)[:, :, valid],
                 1e-5, "dt")
    assert_close(cs.double().cpu().numpy()[:, :, valid], im["cs"][:, :, valid], 1e-5, "cumsum")
    # segment counts: integer, bit-exact against their definition
    sidx = d["seq_idx"].numpy()
    want = np.zeros((2, nc, Q), dtype=np.int32)
    for b in range(2):
        for c in range(nc):
            cnt = 0
            for t in range(Q):
                pos = c * Q + t
                if pos < L and pos >= 1 and sidx[b, pos] != sidx[b, pos - 1]:
                    cnt += 1
                want[b, c, t] = cnt
    assert np.array_equal(seg.cpu().numpy(), want)
    # stage 2
    states = ssd.ssd_chunk_state(g["x"], g["B"], dt_out, cs, seg, chunk_size=Q)
    assert_close(states.double().cpu().numpy(), im["states"], 1e-4, "chunk states")
    # stage 3 (in place)
    fin = ssd.ssd_state_passing(states, cs, seg, seqlen=L, chunk_size=Q,
                                initial_states=g["initial_states"])
    assert_close(states.double().cpu().numpy(), im["prev_states"], 1e-4, "prev states")
    assert_close(fin.double().cpu().numpy(), rf, 1e-4, "final")
    # stage 4
    out = ssd.ssd_chunk_scan(g["x"], g["B"], g["C"], dt_out, cs, seg, states, chunk_size=Q,
                             D=g["D"], z=g["z"])
    torch.cuda.synchronize()
    assert_close(out.double().cpu().numpy(), ry, TOL[dtype], "out")


# --------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times: the
# whole GPU output against the oracle, every (batch, head) pair, in pieces;
# mean and max errors (and the 99.9th percentile) are recorded for the
# parity report because SSD kernel errors can be heavy-tailed
# --------------------------------------------------------------------------

def _full_check(name, d, y_gpu, f_gpu, tol, head_block=16):
    """Every (batch, head) recurrence of the GPU output against the oracle
    (run over the whole sequence), accumulated piece by piece."""
    Bsz, L, H, P = d["x"].shape
    yg, fg = y_gpu.cpu(), f_gpu.cpu()
    sy, sf = ErrorStats(), ErrorStats()
    for b in range(Bsz):
        for h0 in range(0, H, head_block):
            hs = list(range(h0, min(H, h0 + head_block)))
            ry, rf = so.scan_sequential(d, heads=hs, batches=[b])
            sy.add(yg[b:b + 1, :, h0:h0 + len(hs)].double().numpy(), ry)
            sf.add(fg[b:b + 1, h0:h0 + len(hs)].double().numpy(), rf)
    ey, ef = sy.result(), sf.result()
    PARITY_REPORT[name] = {"out": ey, "final_states": ef, "tol": tol,
                           "pairs": Bsz * H, "tokens": Bsz * L}
    assert ey["max_rel"] <= tol, f"{name} out: {ey}"
    assert ef["max_rel"] <= tol, f"{name} final: {ef}"


def _gpu_full(d, chunk):
    import selective_state_space_05_gb300 as ssd
    g = to_dev(d)
    y, f = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=chunk,
                            dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                            initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                            return_final_states=True, check=True)
    return y, f


def test_mamba2_2p7b_full_size():
    cfg = si.CONFIGS["mamba2_2p7b"]
    d = si.make_inputs(cfg, 1002)
    y, f = _gpu_full(d, cfg.chunk_size)
    assert torch.isfinite(y.float()).all()
    _full_check("mamba2_2p7b", d, y, f, TOL["bf16"])


def test_chained_prefill_full_size():
    """4 calls of 2048 tokens, final_states fed back as initial_states, against
    the oracle over the whole 8192 tokens."""
    import selective_state_space_05_gb300 as ssd
    cfg = si.CONFIGS["chained"]
    d = si.make_inputs(cfg, 1003)
    g = to_dev(d)
    seg_len = cfg.seqlen // cfg.segments
    y = torch.empty_like(g["x"])
    st = g["initial_states"]
    for s in range(cfg.segments):
        sl = slice(s * seg_len, (s + 1) * seg_len)
        part = {k: g[k][:, sl].contiguous() for k in ("x", "dt", "B", "C", "z")}
        ys, st = ssd.ssd_scan_fwd(part["x"], part["dt"], g["A"], part["B"], part["C"],
                                  chunk_size=cfg.chunk_size, dt_bias=g["dt_bias"], D=g["D"],
                                  z=part["z"], initial_states=st, return_final_states=True)
        y[:, sl] = ys
    ssd.scan_status(reset=True)
    del g, part
    _full_check("chained", d, y, st, TOL["bf16"])


def test_packed_documents_full_size():
    cfg = si.CONFIGS["packed"]
    d = si.make_inputs(cfg, 1004)
    y, f = _gpu_full(d, cfg.chunk_size)
    _full_check("packed", d, y, f, TOL["bf16"], head_block=8)


def test_small_workloads_report():
    """The tiny and grouped workloads whole, for the parity report; the
    grouped runs also on y - D x silu(z) (D_h = 1000 h dominates max|ref| and
    could hide scan errors; both sides lose the same exactly computed term)."""
    for name, seed in (("tiny", 1000), ("grouped_g1", 1001), ("grouped_g2", 1001),
                       ("grouped_g4", 1001)):
        cfg = si.CONFIGS[name]
        d = si.make_inputs(cfg, seed)
        y, f = run_gpu(d)
        ry, rf = oracle.scan_sequential(d)
        tol = TOL[cfg.dtype]
        entry = {"out": errors(y, ry), "final_states": errors(f, rf), "tol": tol}
        if d["D"] is not None and d["z"] is not None:
            x = d["x"].double().numpy()
            zz = d["z"].double().numpy()
            skip = d["D"].double().numpy()[None, None, :, None] * x * zz / (1 + np.exp(-zz))
            entry["out_minus_Dx"] = errors(y - skip, ry - skip)
        PARITY_REPORT[name] = entry
        assert entry["out"]["max_rel"] <= tol and entry["final_states"]["max_rel"] <= tol, entry
