"""The scan as a differentiable torch function (ssd_scan: ssd_scan_fwd
forward, ssd_scan_bwd backward): loss.backward() fills every input's .grad
with the oracle's gradients (tolerances as in test_bwd_gpu.py), gradients
flow through torch ops around the scan, and strided views (slices of an
input projection) work."""
import numpy as np
import pytest
import torch

from oracle import ssd_oracle as so
import ssd_inputs as si
from ssd_testutil import TOL, assert_close
from test_bwd_gpu import _head_terms

pytestmark = pytest.mark.gpu

LEAVES = ("x", "dt", "A", "B", "C", "dt_bias", "D", "z", "initial_states")


def _leaves(d):
    return {k: d[k].cuda().clone().requires_grad_(True) for k in LEAVES if d.get(k) is not None}


@pytest.mark.parametrize("Q,P,N", [(128, 64, 128), (64, 32, 64)])
def test_loss_backward_matches_oracle(Q, P, N):
    import selective_state_space_05_gb300 as ssd
    d = si.random_small(600 + P, batch=2, seqlen=300, nheads=4, headdim=P, dstate=N, ngroups=2,
                        chunk_size=Q, dtype="f32", init_std=0.3, seq_idx_lengths=[120, 1, 179])
    w = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(9))
    t = _leaves(d)
    out = ssd.ssd_scan(t["x"], t["dt"], t["A"], t["B"], t["C"], chunk_size=Q,
                       dt_bias=t["dt_bias"], D=t["D"], z=t["z"],
                       initial_states=t["initial_states"], seq_idx=d["seq_idx"].cuda())
    (out * w.cuda()).sum().backward()
    ref = so.scan_backward(d, w)
    scale = _head_terms(d, w, ref)
    for k in LEAVES:
        got = t[k].grad.double().cpu().numpy()
        if k in scale:
            assert (np.abs(got - ref[k]) <= TOL["f32"] * scale[k] + 1e-30).all(), k
        else:
            assert_close(got, ref[k], TOL["f32"], k)


def test_gradients_flow_through_surrounding_ops():
    """dt from a scaled leaf, x from a strided slice of a projection: the
    leaves' gradients are the scan's gradients pushed back through them."""
    import selective_state_space_05_gb300 as ssd
    d = si.random_small(610, batch=1, seqlen=256, nheads=2, headdim=64, dstate=128, ngroups=1,
                        chunk_size=128, dtype="f32", init_std=0.2)
    H, P = 2, 64
    raw = (d["dt"] / 3.0).cuda().requires_grad_(True)
    proj = torch.cat([d["x"].reshape(1, 256, -1), torch.zeros(1, 256, 8)], dim=2).cuda()
    proj.requires_grad_(True)
    x = proj[:, :, :H * P].unflatten(2, (H, P))
    assert not x.is_contiguous()
    g = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    out = ssd.ssd_scan(x, raw * 3.0, g["A"], g["B"], g["C"], chunk_size=128,
                       dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                       initial_states=g["initial_states"])
    w = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(10))
    (out * w.cuda()).sum().backward()
    ref = so.scan_backward(d, w, names=("x", "dt"))
    assert_close(raw.grad.double().cpu().numpy(), 3.0 * ref["dt"], TOL["f32"], "d raw")
    gx = proj.grad[:, :, :H * P].reshape(d["x"].shape).double().cpu().numpy()
    assert_close(gx, ref["x"], TOL["f32"], "d proj (x part)")
    assert float(proj.grad[:, :, H * P:].abs().max()) == 0.0


def test_bf16_training_step():
    """bf16 leaves: the forward is the bf16 path, loss.backward() gives bf16
    gradients for x, dt, B, C, z and fp32 ones for A, dt_bias, D, within the
    bf16 bound of the oracle's."""
    import selective_state_space_05_gb300 as ssd
    d = si.random_small(620, batch=1, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2,
                        chunk_size=256, dtype="bf16")
    w = torch.randn(d["x"].shape, generator=torch.Generator().manual_seed(11))
    t = _leaves(d)
    out = ssd.ssd_scan(t["x"], t["dt"], t["A"], t["B"], t["C"], chunk_size=256,
                       dt_bias=t["dt_bias"], D=t["D"], z=t["z"])
    assert out.dtype == torch.bfloat16
    (out.float() * w.cuda()).sum().backward()
    d32 = {k: (v.float() if torch.is_tensor(v) and v.dtype == torch.bfloat16 else v)
           for k, v in d.items()}
    # the upstream gradient reaching the scan is w rounded to bf16
    ref = so.scan_backward(d32, w.bfloat16().float())
    for k in ("x", "dt", "B", "C", "z"):
        assert t[k].grad.dtype == torch.bfloat16
        assert_close(t[k].grad.double().cpu().numpy(), ref[k], TOL["bf16"], k)
    for k in ("A", "dt_bias", "D"):
        assert t[k].grad.dtype == torch.float32
        assert_close(t[k].grad.double().cpu().numpy(), ref[k], TOL["bf16"], k)
