"""The decode step (ssd_decode_step) on the GPU: one step equals the
oracle's recurrence at one token from the given state; a run of steps from a
prefill's final states equals the oracle over the whole sequence (chunked
prefill continued by decoding, as the initial-state page describes: PR #488
of state-spaces/mamba); options and shapes as in the scan."""
import pytest
import torch

import oracle
import ssd_inputs as si
from ssd_testutil import TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _token(d, t):
    """The inputs of token t as a one-token sequence."""
    e = dict(d)
    for k in ("x", "dt", "B", "C", "z"):
        if d[k] is not None:
            e[k] = d[k][:, t:t + 1].contiguous()
    e["seq_idx"] = None
    return e


CASES = [
    ("bf16_hd64_ds128", dict(batch=3, nheads=8, ngroups=2, headdim=64, dstate=128,
                             dtype="bf16", init_std=0.5)),
    ("f32_hd64_ds64_G1", dict(batch=2, nheads=4, ngroups=1, headdim=64, dstate=64,
                              dtype="f32", init_std=0.5, has_z=False)),
    ("f32_hd128_ds256", dict(batch=1, nheads=2, ngroups=2, headdim=128, dstate=256,
                             dtype="f32", init_std=0.3, dt_limit=(0.01, 0.2))),
    ("f32_hd16_ds16_no_softplus", dict(batch=2, nheads=4, ngroups=4, headdim=16, dstate=16,
                                       dtype="f32", init_std=0.3, dt_softplus=False,
                                       dt_bias=False, has_D=False)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_one_step_matches_oracle(case):
    import selective_state_space_05_gb300 as ssd
    _, kw = case
    d = si.random_small(900 + len(case[0]), seqlen=1, chunk_size=16, **kw)
    if not kw.get("dt_softplus", True):
        d["dt"] = (d["dt"].float().abs() * 0.2).to(d["dt"].dtype)
    g = to_dev(d)
    state = g["initial_states"].clone()
    tok = {k: (None if g[k] is None else g[k][:, 0].contiguous())
           for k in ("x", "dt", "B", "C", "z")}
    out = ssd.ssd_decode_step(tok["x"], tok["dt"], g["A"], tok["B"], tok["C"], state,
                              dt_bias=g["dt_bias"], dt_softplus=d["dt_softplus"],
                              dt_limit=d["dt_limit"], D=g["D"], z=tok["z"])
    torch.cuda.synchronize()
    ry, rf = oracle.scan_sequential(d)
    tol = TOL[kw["dtype"]]
    assert_close(out.double().cpu().numpy(), ry[:, 0], tol, "out")
    assert_close(state.double().cpu().numpy(), rf, tol, "state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_then_decode_equals_whole_sequence(dtype):
    """Prefill 300 tokens with ssd_scan_fwd, then 40 decode steps from its
    final states: the decoded outputs and the last state match the oracle run
    over all 340 tokens (and the GPU scan over all of them)."""
    import selective_state_space_05_gb300 as ssd
    L0, T = 300, 40
    d = si.random_small(950, batch=2, seqlen=L0 + T, nheads=4, ngroups=2, headdim=64,
                        dstate=128, chunk_size=128, dtype=dtype, init_std=0.3)
    g = to_dev(d)
    pre = {k: (g[k][:, :L0].contiguous() if k in ("x", "dt", "B", "C", "z") else g[k])
           for k in g}
    _, state = ssd.ssd_scan_fwd(pre["x"], pre["dt"], g["A"], pre["B"], pre["C"], chunk_size=128,
                                dt_bias=g["dt_bias"], D=g["D"], z=pre["z"],
                                initial_states=g["initial_states"], return_final_states=True)
    outs = []
    for t in range(L0, L0 + T):
        tok = {k: g[k][:, t].contiguous() for k in ("x", "dt", "B", "C", "z")}
        outs.append(ssd.ssd_decode_step(tok["x"], tok["dt"], g["A"], tok["B"], tok["C"], state,
                                        dt_bias=g["dt_bias"], D=g["D"], z=tok["z"]))
    y = torch.stack(outs, dim=1)
    whole, whole_fin = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=128,
                                        dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                                        initial_states=g["initial_states"],
                                        return_final_states=True)
    torch.cuda.synchronize()
    ry, rf = oracle.scan_sequential(d)
    tol = TOL[dtype]
    assert_close(y.double().cpu().numpy(), ry[:, L0:], tol, "decoded out")
    assert_close(state.double().cpu().numpy(), rf, tol, "state after decoding")
    assert_close(y.double().cpu().numpy(), whole[:, L0:].double().cpu().numpy(), tol,
                 "decoded vs scanned")
    assert_close(state.double().cpu().numpy(), whole_fin.double().cpu().numpy(), tol,
                 "state vs scanned")
