"""The block around the scan on the GPU: the causal conv1d and the group
RMSNorm against the oracle's fp64 definitions, and the whole
mamba_split_conv1d_scan_combined block of the "ngroups > 1" issue page
(state-spaces/mamba #647) end to end: conv, scan (on strided views of the
conv output and of the projection) and grouped norm all run in the CUDA
library, only the output projection is test-side glue, and out[0, 0, 0]
must reproduce the values the page prints."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import ssd_oracle as so
from ssd_testutil import TOL, assert_close

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


CONV_CASES = [
    # (id, batch, seqlen, channels, width, dtype, elements before / after the
    # channels in each token's row of the source (a strided view when > 0;
    # both keep 16-byte alignment), seq_idx document lengths)
    ("bf16_w4_strided", 2, 300, 272, 4, torch.bfloat16, (16, 24), None),
    ("bf16_w4_docs", 1, 517, 128, 4, torch.bfloat16, (0, 0), [100, 1, 2, 300, 114]),
    ("f32_w2_strided", 2, 130, 64, 2, torch.float32, (4, 4), None),
    ("f32_w7_docs", 1, 200, 40, 7, torch.float32, (4, 0), [63, 64, 73]),
    ("bf16_w1_len1", 3, 1, 16, 1, torch.bfloat16, (0, 0), None),
]


@pytest.mark.parametrize("case", CONV_CASES, ids=[c[0] for c in CONV_CASES])
def test_causal_conv1d_matches_oracle(case):
    import selective_state_space_05_gb300 as ssd
    _, B, L, C, W, dt, (before, after), lens = case
    g = torch.Generator().manual_seed(len(case[0]))
    src = torch.randn(B, L, before + C + after, generator=g).to(dt)
    x = src[:, :, before:before + C]
    w = torch.randn(C, W, generator=g) * 0.5
    b = torch.randn(C, generator=g)
    sq = None
    if lens:
        sq = torch.cat([torch.full((n,), i, dtype=torch.int32) for i, n in enumerate(lens)])
        sq = sq.unsqueeze(0).expand(B, -1).contiguous()
    xd = src.cuda()[:, :, before:before + C]
    assert xd.is_contiguous() == (before + after == 0)
    y = ssd.causal_conv1d(xd, w.cuda(), b.cuda(), seq_idx=None if sq is None else sq.cuda())
    torch.cuda.synchronize()
    ref = oracle.causal_conv1d(x, w, b, seq_idx=sq, silu=True)
    tol = 1e-5 if dt == torch.float32 else TOL["bf16"]
    assert_close(y.double().cpu().numpy(), ref, tol, "conv")


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gs_div", [1, 2, 8])
def test_group_rmsnorm_matches_oracle(dt, gs_div):
    import selective_state_space_05_gb300 as ssd
    g = torch.Generator().manual_seed(7 + gs_div)
    dim = 5120
    y = (torch.randn(3, 33, dim, generator=g) * 3).to(dt)
    w = torch.randn(dim, generator=g)
    yd = y.cuda()
    ssd.group_rmsnorm_(yd, w.cuda(), group_size=dim // gs_div, eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.group_rmsnorm(y, w, 1e-5, dim // gs_div)
    tol = 1e-5 if dt == torch.float32 else TOL["bf16"]
    assert_close(yd.double().cpu().numpy(), ref, tol, "norm")


def _p1_block_gpu(G: int, grouped: bool):
    """The page's block (batch 2, seqlen 2048, dim 2048, 32 heads of 64,
    dstate 128, conv width 4, chunk 128; every input and weight 0.1, A = -1,
    D = 1000 h, fp32) with the conv, scan and norm on the GPU; returns the
    output projection's result [B, L, dim] (fp32) and the normalised scan
    output [B, L, d_inner]."""
    import selective_state_space_05_gb300 as ssd
    B, L, H, P, N, Wc = 2, 2048, 32, 64, 128, 4
    dim = H * P
    conv_dim = dim + 2 * G * N
    dev = "cuda"
    zx = torch.full((B, L, 2 * dim + 2 * G * N + H), 0.1, device=dev)
    xbc = ssd.causal_conv1d(zx[:, :, dim:dim + conv_dim],
                            torch.full((conv_dim, Wc), 0.1, device=dev),
                            torch.full((conv_dim,), 0.1, device=dev))
    x = xbc[:, :, :dim].unflatten(2, (H, P))
    Bm = xbc[:, :, dim:dim + G * N].unflatten(2, (G, N))
    Cm = xbc[:, :, dim + G * N:].unflatten(2, (G, N))
    z = zx[:, :, :dim].unflatten(2, (H, P))
    dt = zx[:, :, -H:]
    y = ssd.ssd_scan_fwd(x, dt, -torch.ones(H, device=dev), Bm, Cm, chunk_size=128,
                         dt_bias=torch.full((H,), 0.1, device=dev),
                         D=torch.arange(H, device=dev, dtype=torch.float32) * 1000.0, z=z,
                         check=True)
    yn = ssd.group_rmsnorm_(y.view(B, L, dim), torch.full((dim,), 0.1, device=dev),
                            group_size=dim // G if grouped else dim, eps=1e-5)
    out = torch.nn.functional.linear(yn, torch.full((dim, dim), 0.1, device=dev),
                                     torch.full((dim,), 0.1, device=dev))
    torch.cuda.synchronize()
    return out, yn


@pytest.mark.parametrize("G", [1, 2, 4])
def test_p1_block_end_to_end_reproduces_printed_values(G):
    golden = json.load(open(os.path.join(GOLDEN, "p1_worked_example.json")))
    out, yn = _p1_block_gpu(G, grouped=True)
    assert abs(float(out[0, 0, 0]) - golden["printed"]["combined"][str(G)]) < 1.5e-4
    out_r, _ = _p1_block_gpu(G, grouped=False)
    assert abs(float(out_r[0, 0, 0]) - golden["printed"]["ref"][str(G)]) < 1.5e-4
    # the whole normalised scan output of the first 96 tokens against the
    # oracle's conv, scan and norm in fp64
    H, P, N, L = 32, 64, 128, 96
    dim = H * P
    conv_dim = dim + 2 * G * N
    zx = np.full((1, L, 2 * dim + 2 * G * N + H), 0.1)
    xbc = oracle.causal_conv1d(zx[:, :, dim:dim + conv_dim], np.full((conv_dim, 4), 0.1),
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
    ref = oracle.group_rmsnorm(y.reshape(1, L, dim), np.full(dim, 0.1), 1e-5, dim // G)
    assert_close(yn[:1, :L].double().cpu().numpy(), ref, TOL["f32"], "normalised scan output")
