"""Seeded synthetic inputs for the SSD chunked-scan forward.

This module is shared by the oracle-based tests, the CUDA parity tests and
``bench.py``.  It only draws random numbers with the distributions of the
workloads below; it holds none of the scan's arithmetic.  Everything is drawn
on the CPU from a seeded ``torch.Generator`` so that the oracle and the GPU
path see bit-identical values (bf16 tensors are rounded once, here).

Workloads (distributions as the benchmark configurations state them):

* ``tiny``      fp32, batch 1, seqlen 256, 4 heads, headdim 16, dstate 16,
                1 group, chunk 64; no z, no initial state.
* ``grouped``   fp32, batch 2, seqlen 2048, 32 heads, headdim 64, dstate 128,
                ngroups in {1, 2, 4}, chunk 128; x, B, C ~ N(0,1)/2,
                D_h = 1000*h, z gate on.  These are the shapes of the
                ``mamba_split_conv1d_scan_combined`` repro on the
                "ngroups > 1" issue page (state-spaces/mamba #647, script).
* ``mamba2_2p7b`` bf16, batch 8, seqlen 4096, 80 heads, headdim 64
                (d_inner 5120), dstate 128, 1 group, chunk 256, z gate on.
* ``chained``   bf16, batch 16, seqlen 8192 run as 4 segments of 2048 with
                final states fed back; 128 heads, 8 groups, chunk 256,
                first-segment initial states ~ N(0, 0.1^2).
* ``packed``    bf16, batch 1, seqlen 131072 holding 8 documents whose
                lengths come from a seeded Dirichlet(1,...,1) split, marked by
                seq_idx; 128 heads, 8 groups, chunk 256.

Common to all: dt_raw ~ N(0,1) (stored in x's dtype), dt_bias =
log(expm1(U[1e-3, 1e-1])) so that softplus(dt_bias) ~ U[1e-3, 1e-1],
softplus on, A_h = -exp(U[log 1, log 16]) fp32, D ~ N(0,1) fp32 unless
stated.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class SSDConfig:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    dtype: str                 # "f32" or "bf16"
    x_scale: float = 1.0       # x, B, C ~ N(0,1) * x_scale
    d_mode: str = "normal"     # "normal": D ~ N(0,1); "ramp": D_h = 1000*h; "none"
    has_z: bool = True
    init_std: float = 0.0      # > 0: initial_states ~ N(0, init_std^2)
    ndocs: int = 1             # > 1: seq_idx with a Dirichlet split into ndocs
    segments: int = 1          # > 1: run as this many chained calls
    a_log_range: tuple = (0.0, math.log(16.0))   # A = -exp(U[lo, hi])
    dt_softplus: bool = True
    dt_limit: tuple = (0.0, float("inf"))

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def with_(self, **kw) -> "SSDConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": SSDConfig("tiny", 1, 256, 4, 16, 16, 1, 64, "f32",
                      d_mode="normal", has_z=False),
    "grouped_g1": SSDConfig("grouped_g1", 2, 2048, 32, 64, 128, 1, 128, "f32",
                            x_scale=0.5, d_mode="ramp"),
    "grouped_g2": SSDConfig("grouped_g2", 2, 2048, 32, 64, 128, 2, 128, "f32",
                            x_scale=0.5, d_mode="ramp"),
    "grouped_g4": SSDConfig("grouped_g4", 2, 2048, 32, 64, 128, 4, 128, "f32",
                            x_scale=0.5, d_mode="ramp"),
    "mamba2_2p7b": SSDConfig("mamba2_2p7b", 8, 4096, 80, 64, 128, 1, 256, "bf16"),
    "chained": SSDConfig("chained", 16, 8192, 128, 64, 128, 8, 256, "bf16",
                         init_std=0.1, segments=4),
    "packed": SSDConfig("packed", 1, 131072, 128, 64, 128, 8, 256, "bf16",
                        ndocs=8),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def dirichlet_lengths(total: int, ndocs: int, seed: int) -> list:
    """Document lengths: floor(Dirichlet(1,...,1) * total), each >= 1, the
    remainder added to the last document."""
    rng = np.random.default_rng(seed)
    w = rng.dirichlet(np.ones(ndocs))
    lens = np.maximum(np.floor(w * total).astype(np.int64), 1)
    # keep the sum exact: trim from the longest if the floors overshot, then
    # give the remainder to the last document
    while lens.sum() > total:
        lens[np.argmax(lens)] -= 1
    lens[-1] += total - lens.sum()
    assert lens.min() >= 1 and lens.sum() == total
    return [int(v) for v in lens]


def seq_idx_from_lengths(lengths, batch: int) -> torch.Tensor:
    ids = torch.cat([torch.full((n,), i, dtype=torch.int32)
                     for i, n in enumerate(lengths)])
    return ids.unsqueeze(0).expand(batch, -1).contiguous()


def make_inputs(cfg: SSDConfig, seed: int, seqlen: Optional[int] = None,
                device="cpu") -> dict:
    """Draw one set of inputs, on the CPU by default.

    Draw order is fixed: x, z, B, C, dt_raw, dt_bias, A, D, initial_states,
    then the document split.  Returns a dict of tensors keyed by the C-ABI
    argument names plus the scalar options.  With a CUDA ``device`` the same
    recipe is drawn by that device's generator (same distributions, other
    values; the benchmark uses it for workloads too large to draw on the host
    quickly, and no parity check compares against such draws).
    """
    L = cfg.seqlen if seqlen is None else seqlen
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    dt_ = torch_dtype(cfg.dtype)
    Bsz, H, P, N, G = cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups

    def normal(*shape, scale=1.0):
        t = torch.randn(*shape, generator=g, dtype=torch.float32, device=dev)
        if scale != 1.0:
            t.mul_(scale)
        return t

    x = normal(Bsz, L, H, P, scale=cfg.x_scale).to(dt_)
    z = normal(Bsz, L, H, P).to(dt_) if cfg.has_z else None
    Bm = normal(Bsz, L, G, N, scale=cfg.x_scale).to(dt_)
    Cm = normal(Bsz, L, G, N, scale=cfg.x_scale).to(dt_)
    dt = normal(Bsz, L, H).to(dt_)
    u = torch.rand(H, generator=g, dtype=torch.float64, device=dev) * (1e-1 - 1e-3) + 1e-3
    dt_bias = torch.log(torch.expm1(u)).to(torch.float32)
    lo, hi = cfg.a_log_range
    A = -torch.exp(torch.rand(H, generator=g, dtype=torch.float64, device=dev) * (hi - lo)
                   + lo).to(torch.float32)
    if cfg.d_mode == "normal":
        D = normal(H)
    elif cfg.d_mode == "ramp":
        D = torch.arange(H, dtype=torch.float32, device=dev) * 1000.0
    else:
        D = None
    init = normal(Bsz, H, P, N, scale=cfg.init_std) if cfg.init_std > 0 else None
    seq_idx = None
    if cfg.ndocs > 1:
        lens = dirichlet_lengths(L, cfg.ndocs, seed)
        seq_idx = seq_idx_from_lengths(lens, Bsz).to(dev)
    return dict(x=x, dt=dt, dt_bias=dt_bias, A=A, B=Bm, C=Cm, D=D, z=z,
                initial_states=init, seq_idx=seq_idx,
                dt_softplus=cfg.dt_softplus, dt_limit=cfg.dt_limit,
                chunk_size=cfg.chunk_size, ngroups=G)


def random_small(seed: int, *, batch=2, seqlen=37, nheads=4, headdim=8, dstate=6,
                 ngroups=2, chunk_size=16, dtype="f32", has_z=True, has_D=True,
                 init_std=0.0, seq_idx_lengths=None, dt_softplus=True,
                 dt_bias=True, dt_limit=(0.0, float("inf")),
                 a_log_range=(0.0, math.log(16.0)), x_scale=1.0) -> dict:
    """Small random inputs for edge cases and oracle self-checks."""
    cfg = SSDConfig("small", batch, seqlen, nheads, headdim, dstate, ngroups,
                    chunk_size, dtype, x_scale=x_scale,
                    d_mode="normal" if has_D else "none", has_z=has_z,
                    init_std=init_std, a_log_range=a_log_range,
                    dt_softplus=dt_softplus, dt_limit=dt_limit)
    d = make_inputs(cfg, seed)
    if not dt_bias:
        d["dt_bias"] = None
    if seq_idx_lengths is not None:
        assert sum(seq_idx_lengths) == seqlen
        d["seq_idx"] = seq_idx_from_lengths(seq_idx_lengths, batch)
    return d
