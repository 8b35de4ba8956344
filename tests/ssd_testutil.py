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


class ErrorStats:
    """The metrics of errors() accumulated over pieces of an output too large
    to hold in fp64 at once.  The 99.9th percentile comes from a histogram of
    |err| with bins 1 % wide (log-spaced from 1e-14 to 1e6)."""

    EDGES = np.logspace(-14, 6, 20 * 231 + 1)

    def __init__(self):
        self.max_diff = 0.0
        self.max_ref = 0.0
        self.sum_abs_diff = 0.0
        self.sum_abs_ref = 0.0
        self.sum_diff = 0.0
        self.n = 0
        self.zeros = 0
        self.hist = np.zeros(len(self.EDGES) - 1, dtype=np.int64)

    def add(self, got, ref):
        got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
        diff = got - ref
        ad = np.abs(diff).ravel()
        self.max_diff = max(self.max_diff, float(ad.max(initial=0.0)))
        self.max_ref = max(self.max_ref, float(np.abs(ref).max(initial=0.0)))
        self.sum_abs_diff += float(ad.sum())
        self.sum_abs_ref += float(np.abs(ref).sum())
        self.sum_diff += float(diff.sum())
        self.n += ad.size
        self.zeros += int((ad < self.EDGES[0]).sum())
        nz = ad[ad >= self.EDGES[0]]
        self.hist += np.histogram(np.minimum(nz, self.EDGES[-1]), self.EDGES)[0]

    def result(self) -> dict:
        den = max(self.max_ref, 1e-300)
        want = 0.999 * self.n - self.zeros
        if want <= 0:
            p999 = 0.0
        else:
            k = int(np.searchsorted(np.cumsum(self.hist), want))
            p999 = float(self.EDGES[min(k + 1, len(self.EDGES) - 1)])
        return dict(max_rel=self.max_diff / den,
                    mean_rel=self.sum_abs_diff / max(self.sum_abs_ref, 1e-300),
                    mean_diff=self.sum_diff / max(self.n, 1),
                    p999_rel=p999 / den, elements=self.n)


# parity figures of the full-size runs, written as JSON at the end of the
# session when SSD_PARITY_REPORT names a file
PARITY_REPORT = {}
