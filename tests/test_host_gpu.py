"""ssd_scan_fwd_host (tensors in host memory, pipelined batch slices) against
ssd_scan_fwd on the same inputs in device memory.  Each batch row's result
does not depend on the others, so the two must agree exactly, for the fused
kernel's shapes and for the stage kernels' shapes, with every slice size."""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from ssd_testutil import TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _host(d, pin=True):
    h = {}
    for k, v in d.items():
        if torch.is_tensor(v):
            v = v.contiguous()
            h[k] = v.pin_memory() if pin else v
        else:
            h[k] = v
    return h


def _both(d, chunk, rows, pin=True):
    import selective_state_space_05_gb300 as ssd
    g = to_dev(d)
    kw = dict(chunk_size=chunk, dt_bias=g["dt_bias"], dt_softplus=d.get("dt_softplus", True),
              D=g["D"], z=g["z"], initial_states=g["initial_states"], seq_idx=g["seq_idx"],
              return_final_states=True)
    y_d, f_d = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], **kw)
    torch.cuda.synchronize()
    h = _host(d, pin)
    kw = dict(chunk_size=chunk, dt_bias=h["dt_bias"], dt_softplus=d.get("dt_softplus", True),
              D=h["D"], z=h["z"], initial_states=h["initial_states"], seq_idx=h["seq_idx"],
              return_final_states=True, rows_per_slice=rows)
    y_h, f_h = ssd.ssd_scan_fwd_host(h["x"], h["dt"], h["A"], h["B"], h["C"], **kw)
    return y_d.cpu(), f_d.cpu(), y_h, f_h


@pytest.mark.parametrize("rows", [0, 1, 2, 5])
def test_host_equals_device_fused(rows):
    d = si.random_small(71, batch=5, seqlen=700, nheads=4, ngroups=2, headdim=64, dstate=128,
                        chunk_size=256, dtype="bf16", init_std=0.3, seq_idx_lengths=[300, 400])
    y_d, f_d, y_h, f_h = _both(d, 256, rows)
    assert torch.equal(y_d, y_h)
    assert torch.equal(f_d, f_h)
    ry, rf = oracle.scan_sequential(d)
    assert_close(y_h.double().numpy(), ry, TOL["bf16"], "out")
    assert_close(f_h.double().numpy(), rf, TOL["bf16"], "final")


def test_host_equals_device_stage_kernels_f32():
    d = si.random_small(72, batch=3, seqlen=300, nheads=3, ngroups=1, headdim=16, dstate=32,
                        chunk_size=64, dtype="f32", init_std=0.5)
    y_d, f_d, y_h, f_h = _both(d, 64, 2)
    assert torch.equal(y_d, y_h)
    assert torch.equal(f_d, f_h)


def test_host_pageable_memory_and_no_optionals():
    """Pageable host tensors work (without overlap); no z, D, dt_bias,
    initial states or seq_idx."""
    import selective_state_space_05_gb300 as ssd
    d = si.random_small(73, batch=4, seqlen=513, nheads=4, ngroups=1, headdim=64, dstate=128,
                        chunk_size=128, dtype="bf16", has_z=False, has_D=False, dt_bias=False)
    h = _host(d, pin=False)
    y = ssd.ssd_scan_fwd_host(h["x"], h["dt"], h["A"], h["B"], h["C"], chunk_size=128,
                              rows_per_slice=1)
    ry, _ = oracle.scan_sequential(d)
    assert_close(y.double().numpy(), ry, TOL["bf16"], "out")


def test_host_call_is_ordered_on_the_stream():
    """Without synchronize, reading after the stream is synchronised gives the
    result; a second call on the same workspace and stream sees the first one
    finished (same answer twice)."""
    import selective_state_space_05_gb300 as ssd
    d = si.random_small(74, batch=4, seqlen=600, nheads=4, ngroups=2, headdim=64, dstate=128,
                        chunk_size=256, dtype="bf16", init_std=0.2)
    h = _host(d)
    s = torch.cuda.Stream()
    ws = torch.empty(ssd.host_workspace_bytes(4, 600, 4, 64, 128, 2, 256, torch.bfloat16, 1),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        outs.append(ssd.ssd_scan_fwd_host(h["x"], h["dt"], h["A"], h["B"], h["C"],
                                          chunk_size=256, dt_bias=h["dt_bias"], D=h["D"],
                                          z=h["z"], initial_states=h["initial_states"],
                                          workspace=ws, rows_per_slice=1, stream=s,
                                          synchronize=False))
    s.synchronize()
    assert torch.equal(outs[0], outs[1])
    ry, _ = oracle.scan_sequential(d)
    assert_close(outs[1].double().numpy(), ry, TOL["bf16"], "out")
    assert np.isfinite(outs[1].float().numpy()).all()
