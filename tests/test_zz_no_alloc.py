"""ssd_scan_fwd_noalloc, the entry point for callers that cannot allocate
device memory (a host application whose allocator owns the whole GPU, or a
latency-critical path where an allocation call is not acceptable).  It keeps
its scratch in a fixed static device array inside the library.

Checked through the C ABI against ssd_scan_fwd on two calls in a row with
different sizes and options, so that the second call runs on scratch that
still holds the first call's contents.  This file is collected last so that a
run stopping at the first failure has run every other test before it.
"""

import pytest
import torch

import ssd_inputs as si
from ssd_testutil import TOL, assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_05_gb300 import _lib, build
    build.build()
    return _lib.load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _noalloc(lib, g, d, out, fin):
    Bsz, L, H, P = g["x"].shape
    G, N = g["B"].shape[2], g["B"].shape[3]
    dtype = 1 if g["x"].dtype == torch.bfloat16 else 0
    lo, hi = d.get("dt_limit", (0.0, float("inf")))
    return lib.ssd_scan_fwd_noalloc(
        _ptr(g["x"]), _ptr(g["dt"]), _ptr(g["dt_bias"]), int(d.get("dt_softplus", True)),
        float(lo), float(hi), _ptr(g["A"]), _ptr(g["B"]), _ptr(g["C"]), _ptr(g["D"]),
        _ptr(g["z"]), _ptr(g["initial_states"]), _ptr(g["seq_idx"]), Bsz, L, H, P, N, G,
        int(d["chunk_size"]), dtype, _ptr(out), _ptr(fin),
        torch.cuda.current_stream().cuda_stream)


def _reference(g, d):
    import selective_state_space_05_gb300 as ssd
    return ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=d["chunk_size"],
                            dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                            initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                            return_final_states=True)


CALLS = [
    ("f32", dict(batch=2, seqlen=1000, nheads=8, headdim=64, dstate=128, ngroups=2,
                 chunk_size=128, dtype="f32", init_std=0.3, seq_idx_lengths=[400, 1, 599])),
    ("bf16", dict(batch=1, seqlen=777, nheads=4, headdim=64, dstate=128, ngroups=1,
                  chunk_size=256, dtype="bf16")),
]


def test_noalloc_matches_scan_fwd_on_two_calls_in_a_row(lib):
    for seed, (dtype, kw) in enumerate(CALLS):
        d = si.random_small(500 + seed, **kw)
        g = to_dev(d)
        ref_out, ref_fin = _reference(g, d)
        out = torch.full_like(g["x"], float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        rc = _noalloc(lib, g, d, out, fin)
        torch.cuda.synchronize()
        assert rc == 0, lib.ssd_last_error().decode()
        # no launch gave up a bounded wait (read without allocating either)
        st = lib.ssd_scan_status(1, torch.cuda.current_stream().cuda_stream)
        assert st == 0, lib.ssd_last_error().decode()
        assert_close(out.double().cpu().numpy(), ref_out.double().cpu().numpy(), TOL[dtype],
                     f"out, call {seed + 1}")
        assert_close(fin.double().cpu().numpy(), ref_fin.double().cpu().numpy(), TOL[dtype],
                     f"final states, call {seed + 1}")


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from selective_state_space_05_gb300._lib import SSD_NOALLOC_SCRATCH_BYTES
    cfg = si.CONFIGS["mamba2_2p7b"]
    need = lib.ssd_scan_workspace_bytes(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim,
                                        cfg.dstate, cfg.ngroups, cfg.chunk_size, 1)
    assert need > SSD_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20     # aligned, never dereferenced: the size check comes first
    rc = lib.ssd_scan_fwd_noalloc(fake, fake, None, 1, 0.0, float("inf"), fake, fake, fake,
                                  None, None, None, None, cfg.batch, cfg.seqlen, cfg.nheads,
                                  cfg.headdim, cfg.dstate, cfg.ngroups, cfg.chunk_size, 1, fake,
                                  None, None)
    assert rc == -5
    assert b"scratch" in lib.ssd_last_error()
