"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

TOL = {"f32": 1e-4, "bf16": 2e-2}   # max|err| / max|ref|


def to_dev(d: dict, dev="cuda") -> dict:
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}


def run_gpu(d: dict, chunk_size=None, final=True, out=None):
    import selective_state_space_05_gb300 as ssd
    g = to_dev(d)
    res = ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"],
                           chunk_size=chunk_size or d["chunk_size"], dt_bias=g["dt_bias"],
                           dt_softplus=d.get("dt_softplus", True),
                           dt_limit=d.get("dt_limit", (0.0, float("inf"))), D=g["D"], z=g["z"],
                           initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                           return_final_states=final, out=out)
    torch.cuda.synchronize()
    if final:
        return res[0].double().cpu().numpy(), res[1].double().cpu().numpy()
    return res.double().cpu().numpy(), None


def errors(got, ref) -> dict:
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    diff = got - ref
    den = max(np.abs(ref).max(), 1e-300)
    return dict(max_rel=float(np.abs(diff).max() / den),
                mean_rel=float(np.abs(diff).mean() / max(np.abs(ref).mean(), 1e-300)),
                mean_diff=float(diff.mean()),
                p999_rel=float(np.quantile(np.abs(diff), 0.999) / den))


def assert_close(got, ref, tol, what=""):
    e = errors(got, ref)
    assert e["max_rel"] <= tol, f"{what}: {e}"
    return e
