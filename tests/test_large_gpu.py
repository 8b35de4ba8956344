"""Index arithmetic past 2^31 elements.  The benchmark shape (seqlen 4096,
80 heads, headdim 64, dstate 128, 1 group, chunk 256, z gate, D) with the
batch raised to 132 rows, so that x, z and out hold 2.77e9 elements each and
every row from index 103 on starts beyond element 2^31.  The rows are 33
copies of four rows drawn on the CPU: every copy must give the bits its
original gives, wherever it sits in memory, and the last copies must match
the oracle on sampled heads.  bf16 runs the fused kernel, fp32 the stage
kernels (their chunk_state / chunk_scan on the tensor cores)."""
import dataclasses

import pytest
import torch

import ssd_inputs as si
from oracle import ssd_oracle as so
from ssd_testutil import TOL, assert_close

pytestmark = pytest.mark.gpu

ROWS, COPIES = 4, 33
HEADS = [0, 1, 38, 79]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_beyond_2_31_elements(dtype):
    import selective_state_space_05_gb300 as ssd
    cfg = dataclasses.replace(si.CONFIGS["mamba2_2p7b"], batch=ROWS, dtype=dtype)
    d = si.make_inputs(cfg, 4242)

    def copies(t):
        return t.cuda().repeat(COPIES, *([1] * (t.dim() - 1)))

    def dev(t):
        return None if t is None else t.cuda()

    x, dt, Bm, Cm, z = (copies(d[k]) for k in ("x", "dt", "B", "C", "z"))
    assert x.numel() > 2 ** 31 and x.shape[0] == ROWS * COPIES
    y, f = ssd.ssd_scan_fwd(x, dt, dev(d["A"]), Bm, Cm, chunk_size=cfg.chunk_size,
                            dt_bias=dev(d["dt_bias"]), dt_softplus=cfg.dt_softplus,
                            dt_limit=cfg.dt_limit, D=dev(d["D"]), z=z,
                            return_final_states=True, check=True)
    del x, dt, Bm, Cm, z
    for k in range(1, COPIES):
        rows = slice(ROWS * k, ROWS * (k + 1))
        assert torch.equal(y[rows], y[:ROWS]), f"out, copy {k}"
        assert torch.equal(f[rows], f[:ROWS]), f"final, copy {k}"
    last = ROWS * (COPIES - 1)
    for b in range(ROWS):
        ry, rf = so.scan_sequential(d, heads=HEADS, batches=[b])
        assert_close(y[last + b:last + b + 1, :, HEADS].double().cpu().numpy(), ry, TOL[dtype],
                     f"out, row {last + b}")
        assert_close(f[last + b:last + b + 1, HEADS].double().cpu().numpy(), rf, TOL[dtype],
                     f"final, row {last + b}")
