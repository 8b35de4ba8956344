"""Strided inputs (ssd_scan_fwd_strided): x, B, C as slices of one
convolved xBC buffer and z, dt as slices of one input-projection buffer
zxbcdt, the way the block around the scan splits its projection (repro
script of state-spaces/mamba issue #647).  Where the strided and the dense
call take the same kernels, their results must be equal bit for bit (the
kernels only address the inputs differently); odd strides leave the
tensor-core path, so that case is compared with the oracle only."""
import pytest
import torch

import oracle
import ssd_inputs as si
from ssd_testutil import TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _packed_views(g, pad_tok=0):
    """zxbcdt = [z | xBC | dt] and xBC = [x | B | C] per token (plus pad_tok
    unused elements at the end of each token's row), filled from the dense
    inputs; returns the views x, B, C, z, dt into them."""
    Bsz, L, H, P = g["x"].shape
    G, N = g["B"].shape[2], g["B"].shape[3]
    dx, dbc = H * P, G * N
    xbc_w = dx + 2 * dbc + pad_tok
    zx_w = dx + (dx + 2 * dbc) + H + pad_tok
    xbc = torch.zeros(Bsz, L, xbc_w, dtype=g["x"].dtype, device=g["x"].device)
    zx = torch.zeros(Bsz, L, zx_w, dtype=g["x"].dtype, device=g["x"].device)
    xbc[:, :, :dx] = g["x"].reshape(Bsz, L, dx)
    xbc[:, :, dx:dx + dbc] = g["B"].reshape(Bsz, L, dbc)
    xbc[:, :, dx + dbc:dx + 2 * dbc] = g["C"].reshape(Bsz, L, dbc)
    zx[:, :, :dx] = g["z"].reshape(Bsz, L, dx)
    zx[:, :, 2 * dx + 2 * dbc:2 * dx + 2 * dbc + H] = g["dt"]
    x = xbc[:, :, :dx].view(Bsz, L, H, P)
    B = xbc[:, :, dx:dx + dbc].view(Bsz, L, G, N)
    C = xbc[:, :, dx + dbc:dx + 2 * dbc].view(Bsz, L, G, N)
    z = zx[:, :, :dx].view(Bsz, L, H, P)
    dt = zx[:, :, 2 * dx + 2 * dbc:2 * dx + 2 * dbc + H]
    return x, B, C, z, dt


CASES = [
    # (id, random_small kwargs, pad elements per token, same kernels as the
    # dense call): the 2.7B block's strides are multiples of 8 and keep the
    # tensor-core path; an odd pad makes them odd and takes the stage kernels
    ("bf16_fused_strides", dict(batch=2, seqlen=700, nheads=8, headdim=64, dstate=128,
                                ngroups=2, chunk_size=256, dtype="bf16", init_std=0.3,
                                seq_idx_lengths=[300, 400]), 0, True),
    ("bf16_odd_strides", dict(batch=2, seqlen=300, nheads=4, headdim=64, dstate=128,
                              ngroups=2, chunk_size=128, dtype="bf16"), 3, False),
    ("f32_strides", dict(batch=2, seqlen=200, nheads=4, headdim=32, dstate=64, ngroups=1,
                         chunk_size=64, dtype="f32", init_std=0.2), 4, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_strided_equals_dense(case):
    import selective_state_space_05_gb300 as ssd
    name, kw, pad, same_path = case
    d = si.random_small(700 + len(name), **kw)
    g = to_dev(d)
    x, B, C, z, dt = _packed_views(g, pad)
    assert not x.is_contiguous() and not dt.is_contiguous()
    common = dict(chunk_size=kw["chunk_size"], dt_bias=g["dt_bias"], D=g["D"],
                  initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                  return_final_states=True, check=True)
    ys, fs = ssd.ssd_scan_fwd(x, dt, g["A"], B, C, z=z, **common)
    yd, fd = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], z=g["z"], **common)
    if same_path:
        assert torch.equal(ys, yd) and torch.equal(fs, fd)
    ry, rf = oracle.scan_sequential(d)
    tol = TOL[kw["dtype"]]
    assert_close(yd.double().cpu().numpy(), ry, tol, "out (dense)")
    assert_close(ys.double().cpu().numpy(), ry, tol, "out")
    assert_close(fs.double().cpu().numpy(), rf, tol, "final")
