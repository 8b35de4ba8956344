"""Python binding of the SSD chunked-scan C ABI (include/ssd_scan.h).

Argument marshalling only: checks that torch tensors are CUDA, contiguous and
of the expected dtypes, allocates outputs and workspace with torch, and passes
raw device pointers plus the current CUDA stream to the library.  Every step
of the computation runs in the library's kernels.  Names and argument meaning
follow the C functions of the same names.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _lib

_DT = {torch.float32: _lib.SSD_DTYPE_F32, torch.bfloat16: _lib.SSD_DTYPE_BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _token_dense(t: torch.Tensor) -> bool:
    """Whether each token's part t[b, l] of a [batch, seqlen, ...] tensor is
    dense (row-major), so that two strides describe the whole tensor."""
    want = 1
    for n, s in zip(reversed(t.shape[2:]), reversed(t.stride()[2:])):
        if n > 1 and s != want:
            return False
        want *= n
    return True


def _need(t: Optional[torch.Tensor], name: str, dtype=None, shape=None, device=None,
          optional=False, host=False, strided=False) -> None:
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if host and t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not host and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if strided:
        if not _token_dense(t):
            raise ValueError(f"{name}: each token's [..] part must be dense")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def abi_version() -> int:
    return _lib.load().ssd_abi_version()


def scan_status(reset: bool = True, stream=None) -> None:
    """Synchronises ``stream`` and raises SSDError(SSD_ERR_TIMEOUT) if a
    tensor-core launch on this device gave up a bounded internal wait since
    the last reset (its outputs are then not valid)."""
    _lib.check(_lib.load().ssd_scan_status(int(bool(reset)), _stream(stream)))


def workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                    dtype=torch.bfloat16, least: bool = False) -> int:
    """ssd_scan_workspace_bytes, or with least=True ssd_scan_workspace_bytes_min
    (the smallest workspace ssd_scan_fwd accepts)."""
    f = (_lib.load().ssd_scan_workspace_bytes_min if least
         else _lib.load().ssd_scan_workspace_bytes)
    return int(f(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, _DT[dtype]))


def ssd_scan_fwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                 C: torch.Tensor, *, chunk_size: int = 256,
                 dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
                 dt_limit: Tuple[float, float] = (0.0, math.inf),
                 D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                 initial_states: Optional[torch.Tensor] = None,
                 seq_idx: Optional[torch.Tensor] = None, return_final_states: bool = False,
                 out: Optional[torch.Tensor] = None,
                 final_states: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, stream=None, check: bool = False):
    """SSD chunked-scan forward.  x, z, out: [batch, seqlen, nheads, headdim];
    dt: [batch, seqlen, nheads] (x dtype); B, C: [batch, seqlen, ngroups, dstate];
    dt_bias, A, D: [nheads] fp32; states [batch, nheads, headdim, dstate] fp32;
    seq_idx [batch, seqlen] int32.  x, dt, B, C and z may be strided views
    (slices of a fused projection) as long as each token's part is dense;
    they then go through ssd_scan_fwd_strided.  check=True synchronises the
    stream and raises if the launch gave up a bounded wait (ssd_scan_status).
    Returns out, or (out, final_states)."""
    if x.dtype not in _DT:
        raise ValueError(f"x must be float32 or bfloat16, got {x.dtype}")
    dev = x.device
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    xd = x.dtype
    _need(x, "x", xd, device=dev, strided=True)
    _need(dt, "dt", xd, (Bsz, L, H), dev, strided=True)
    _need(A, "A", torch.float32, (H,), dev)
    _need(B, "B", xd, (Bsz, L, G, N), dev, strided=True)
    _need(C, "C", xd, (Bsz, L, G, N), dev, strided=True)
    _need(dt_bias, "dt_bias", torch.float32, (H,), dev, optional=True)
    _need(D, "D", torch.float32, (H,), dev, optional=True)
    _need(z, "z", xd, (Bsz, L, H, P), dev, optional=True, strided=True)
    _need(initial_states, "initial_states", torch.float32, (Bsz, H, P, N), dev, optional=True)
    _need(seq_idx, "seq_idx", torch.int32, (Bsz, L), dev, optional=True)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", xd, (Bsz, L, H, P), dev)
    if return_final_states and final_states is None:
        final_states = torch.empty(Bsz, H, P, N, dtype=torch.float32, device=dev)
    _need(final_states, "final_states", torch.float32, (Bsz, H, P, N), dev, optional=True)
    lib = _lib.load()
    ws_need = int(lib.ssd_scan_workspace_bytes(Bsz, L, H, P, N, G, chunk_size, _DT[xd]))
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lo, hi = dt_limit
    ins = [x, dt, B, C] + ([z] if z is not None else [])
    if all(t.is_contiguous() for t in ins):
        _lib.check(lib.ssd_scan_fwd(
            _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)), float(lo), float(hi),
            _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(initial_states), _ptr(seq_idx),
            Bsz, L, H, P, N, G, int(chunk_size), _DT[xd], _ptr(out), _ptr(final_states),
            _ptr(workspace), ws_bytes, _stream(stream)))
    else:
        def st(t):
            return _lib.Stride(0, 0) if t is None else _lib.Stride(t.stride(0), t.stride(1))
        _lib.check(lib.ssd_scan_fwd_strided(
            _ptr(x), st(x), _ptr(dt), st(dt), _ptr(dt_bias), int(bool(dt_softplus)), float(lo),
            float(hi), _ptr(A), _ptr(B), st(B), _ptr(C), st(C), _ptr(D), _ptr(z), st(z),
            _ptr(initial_states), _ptr(seq_idx), Bsz, L, H, P, N, G, int(chunk_size), _DT[xd],
            _ptr(out), _ptr(final_states), _ptr(workspace), ws_bytes, _stream(stream)))
    if check:
        scan_status(reset=True, stream=stream)
    if return_final_states:
        return out, final_states
    return out


# --- the four stages, one call each -----------------------------------------

def ssd_dt_cumsum(dt: torch.Tensor, A: torch.Tensor, *, chunk_size: int,
                  dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
                  dt_limit: Tuple[float, float] = (0.0, math.inf),
                  seq_idx: Optional[torch.Tensor] = None, stream=None):
    """Stage 1.  Returns (dt_out, dA_cumsum, chunk_seg or None), the first two
    [batch, nheads, nchunks, chunk_size] fp32, chunk_seg
    [batch, nchunks, chunk_size] int32."""
    Bsz, L, H = dt.shape
    dev = dt.device
    _need(dt, "dt", None, device=dev)
    if dt.dtype not in _DT:
        raise ValueError("dt must be float32 or bfloat16")
    _need(A, "A", torch.float32, (H,), dev)
    _need(dt_bias, "dt_bias", torch.float32, (H,), dev, optional=True)
    _need(seq_idx, "seq_idx", torch.int32, (Bsz, L), dev, optional=True)
    nc = (L + chunk_size - 1) // chunk_size
    dt_out = torch.empty(Bsz, H, nc, chunk_size, dtype=torch.float32, device=dev)
    cs = torch.empty_like(dt_out)
    seg = (torch.empty(Bsz, nc, chunk_size, dtype=torch.int32, device=dev)
           if seq_idx is not None else None)
    lo, hi = dt_limit
    _lib.check(_lib.load().ssd_dt_cumsum(
        _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)), float(lo), float(hi), _ptr(A),
        _ptr(seq_idx), Bsz, L, H, int(chunk_size), _DT[dt.dtype], _ptr(dt_out), _ptr(cs),
        _ptr(seg), _stream(stream)))
    return dt_out, cs, seg


def ssd_chunk_state(x: torch.Tensor, B: torch.Tensor, dt_out: torch.Tensor,
                    dA_cumsum: torch.Tensor, chunk_seg: Optional[torch.Tensor], *,
                    chunk_size: int, stream=None) -> torch.Tensor:
    """Stage 2.  Returns states [batch, nchunks, nheads, headdim, dstate] fp32."""
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    nc = (L + chunk_size - 1) // chunk_size
    _need(x, "x", None, device=dev)
    _need(B, "B", x.dtype, (Bsz, L, G, N), dev)
    _need(dt_out, "dt_out", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(dA_cumsum, "dA_cumsum", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(chunk_seg, "chunk_seg", torch.int32, (Bsz, nc, chunk_size), dev, optional=True)
    states = torch.empty(Bsz, nc, H, P, N, dtype=torch.float32, device=dev)
    _lib.check(_lib.load().ssd_chunk_state(
        _ptr(x), _ptr(B), _ptr(dt_out), _ptr(dA_cumsum), _ptr(chunk_seg), Bsz, L, H, P, N, G,
        int(chunk_size), _DT[x.dtype], _ptr(states), _stream(stream)))
    return states


def ssd_state_passing(states: torch.Tensor, dA_cumsum: torch.Tensor,
                      chunk_seg: Optional[torch.Tensor], *, seqlen: int, chunk_size: int,
                      initial_states: Optional[torch.Tensor] = None,
                      return_final_states: bool = True, stream=None):
    """Stage 3, in place on ``states``.  Returns final_states (or None)."""
    Bsz, nc, H, P, N = states.shape
    dev = states.device
    _need(states, "states", torch.float32, device=dev)
    _need(dA_cumsum, "dA_cumsum", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(chunk_seg, "chunk_seg", torch.int32, (Bsz, nc, chunk_size), dev, optional=True)
    _need(initial_states, "initial_states", torch.float32, (Bsz, H, P, N), dev, optional=True)
    fin = (torch.empty(Bsz, H, P, N, dtype=torch.float32, device=dev)
           if return_final_states else None)
    _lib.check(_lib.load().ssd_state_passing(
        _ptr(states), _ptr(dA_cumsum), _ptr(chunk_seg), _ptr(initial_states), _ptr(fin),
        Bsz, int(seqlen), H, P, N, int(chunk_size), _stream(stream)))
    return fin


def ssd_chunk_scan(x: torch.Tensor, B: torch.Tensor, C: torch.Tensor, dt_out: torch.Tensor,
                   dA_cumsum: torch.Tensor, chunk_seg: Optional[torch.Tensor],
                   prev_states: torch.Tensor, *, chunk_size: int,
                   D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Stage 4.  Returns out [batch, seqlen, nheads, headdim] in x's dtype."""
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    nc = (L + chunk_size - 1) // chunk_size
    _need(x, "x", None, device=dev)
    _need(B, "B", x.dtype, (Bsz, L, G, N), dev)
    _need(C, "C", x.dtype, (Bsz, L, G, N), dev)
    _need(dt_out, "dt_out", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(dA_cumsum, "dA_cumsum", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(chunk_seg, "chunk_seg", torch.int32, (Bsz, nc, chunk_size), dev, optional=True)
    _need(prev_states, "prev_states", torch.float32, (Bsz, nc, H, P, N), dev)
    _need(D, "D", torch.float32, (H,), dev, optional=True)
    _need(z, "z", x.dtype, (Bsz, L, H, P), dev, optional=True)
    if out is None:
        out = torch.empty_like(x)
    _lib.check(_lib.load().ssd_chunk_scan(
        _ptr(x), _ptr(B), _ptr(C), _ptr(dt_out), _ptr(dA_cumsum), _ptr(chunk_seg),
        _ptr(prev_states), _ptr(D), _ptr(z), Bsz, L, H, P, N, G, int(chunk_size),
        _DT[x.dtype], _ptr(out), _stream(stream)))
    return out


def ssd_chunk_fused(x: torch.Tensor, B: torch.Tensor, C: torch.Tensor, dt_out: torch.Tensor,
                    dA_cumsum: torch.Tensor, chunk_seg: Optional[torch.Tensor], *,
                    chunk_size: int, workspace: torch.Tensor, D: Optional[torch.Tensor] = None,
                    z: Optional[torch.Tensor] = None,
                    initial_states: Optional[torch.Tensor] = None,
                    return_final_states: bool = False, out: Optional[torch.Tensor] = None,
                    final_states: Optional[torch.Tensor] = None, stream=None):
    """Stages 2-4 in one tensor-core kernel (bf16, headdim 64, dstate 128,
    chunk 128/256, an even number of heads per group).  Returns out, or
    (out, final_states)."""
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    nc = (L + chunk_size - 1) // chunk_size
    _need(x, "x", torch.bfloat16, device=dev)
    _need(B, "B", torch.bfloat16, (Bsz, L, G, N), dev)
    _need(C, "C", torch.bfloat16, (Bsz, L, G, N), dev)
    _need(dt_out, "dt_out", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(dA_cumsum, "dA_cumsum", torch.float32, (Bsz, H, nc, chunk_size), dev)
    _need(chunk_seg, "chunk_seg", torch.int32, (Bsz, nc, chunk_size), dev, optional=True)
    _need(D, "D", torch.float32, (H,), dev, optional=True)
    _need(z, "z", torch.bfloat16, (Bsz, L, H, P), dev, optional=True)
    _need(initial_states, "initial_states", torch.float32, (Bsz, H, P, N), dev, optional=True)
    _need(workspace, "workspace", torch.uint8, device=dev)
    if out is None:
        out = torch.empty_like(x)
    if return_final_states and final_states is None:
        final_states = torch.empty(Bsz, H, P, N, dtype=torch.float32, device=dev)
    _lib.check(_lib.load().ssd_chunk_fused(
        _ptr(x), _ptr(B), _ptr(C), _ptr(dt_out), _ptr(dA_cumsum), _ptr(chunk_seg), _ptr(D),
        _ptr(z), _ptr(initial_states), Bsz, L, H, P, N, G, int(chunk_size),
        _lib.SSD_DTYPE_BF16, _ptr(out), _ptr(final_states), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    if return_final_states:
        return out, final_states
    return out


# --- host-resident tensors ---------------------------------------------------

def host_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                         dtype=torch.bfloat16, rows_per_slice: int = 0) -> int:
    return int(_lib.load().ssd_scan_host_workspace_bytes(
        batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, _DT[dtype],
        rows_per_slice))


def ssd_scan_fwd_host(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                      C: torch.Tensor, *, chunk_size: int = 256,
                      dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
                      dt_limit: Tuple[float, float] = (0.0, math.inf),
                      D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                      initial_states: Optional[torch.Tensor] = None,
                      seq_idx: Optional[torch.Tensor] = None,
                      return_final_states: bool = False, out: Optional[torch.Tensor] = None,
                      final_states: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, rows_per_slice: int = 0,
                      device=None, stream=None, synchronize: bool = True):
    """ssd_scan_fwd with every tensor on the host (CPU tensors, ideally
    pinned); the library stages them through `workspace` on `device` (default
    the current CUDA device) in pipelined batch slices.  Outputs are written
    to host tensors (allocated pinned when not given).  With synchronize=False
    the call returns once the work is queued on `stream`; the outputs are
    valid after that stream is synchronised."""
    if x.dtype not in _DT:
        raise ValueError(f"x must be float32 or bfloat16, got {x.dtype}")
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    xd = x.dtype
    cpu = torch.device("cpu")
    _need(x, "x", xd, host=True)
    _need(dt, "dt", xd, (Bsz, L, H), cpu, host=True)
    _need(A, "A", torch.float32, (H,), cpu, host=True)
    _need(B, "B", xd, (Bsz, L, G, N), cpu, host=True)
    _need(C, "C", xd, (Bsz, L, G, N), cpu, host=True)
    _need(dt_bias, "dt_bias", torch.float32, (H,), cpu, optional=True, host=True)
    _need(D, "D", torch.float32, (H,), cpu, optional=True, host=True)
    _need(z, "z", xd, (Bsz, L, H, P), cpu, optional=True, host=True)
    _need(initial_states, "initial_states", torch.float32, (Bsz, H, P, N), cpu, optional=True,
          host=True)
    _need(seq_idx, "seq_idx", torch.int32, (Bsz, L), cpu, optional=True, host=True)
    if out is None:
        out = torch.empty(x.shape, dtype=xd).pin_memory()
    _need(out, "out", xd, (Bsz, L, H, P), cpu, host=True)
    if return_final_states and final_states is None:
        final_states = torch.empty(Bsz, H, P, N, dtype=torch.float32).pin_memory()
    _need(final_states, "final_states", torch.float32, (Bsz, H, P, N), cpu, optional=True,
          host=True)
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    need = int(lib.ssd_scan_host_workspace_bytes(Bsz, L, H, P, N, G, chunk_size, _DT[xd],
                                                 rows_per_slice))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    lo, hi = dt_limit
    with torch.cuda.device(dev):
        _lib.check(lib.ssd_scan_fwd_host(
            _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)), float(lo), float(hi),
            _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(initial_states), _ptr(seq_idx),
            Bsz, L, H, P, N, G, int(chunk_size), _DT[xd], _ptr(out), _ptr(final_states),
            int(rows_per_slice), _ptr(workspace), workspace.numel(), _stream(stream)))
        if synchronize:
            scan_status(reset=True, stream=stream)   # synchronises the stream
    if return_final_states:
        return out, final_states
    return out


# --- the block around the scan ----------------------------------------------

def causal_conv1d(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
                  *, seq_idx: Optional[torch.Tensor] = None, activation: Optional[str] = "silu",
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal depthwise conv1d over tokens (ssd_causal_conv1d): x [batch,
    seqlen, channels] (a strided view such as the xBC slice of zxbcdt is
    fine), weight [channels, width] fp32, bias [channels] fp32.  Returns a
    dense [batch, seqlen, channels] tensor of x's dtype."""
    if x.dtype not in _DT:
        raise ValueError("x must be float32 or bfloat16")
    if activation not in (None, "silu"):
        raise ValueError("activation must be None or 'silu'")
    Bsz, L, Cn = x.shape
    dev = x.device
    _need(x, "x", None, device=dev, strided=True)
    W = weight.shape[-1]
    _need(weight, "weight", torch.float32, (Cn, W), dev)
    _need(bias, "bias", torch.float32, (Cn,), dev, optional=True)
    _need(seq_idx, "seq_idx", torch.int32, (Bsz, L), dev, optional=True)
    if out is None:
        out = torch.empty(Bsz, L, Cn, dtype=x.dtype, device=dev)
    _need(out, "out", x.dtype, (Bsz, L, Cn), dev)
    _lib.check(_lib.load().ssd_causal_conv1d(
        _ptr(x), _lib.Stride(x.stride(0), x.stride(1)), _ptr(weight), _ptr(bias), _ptr(seq_idx),
        Bsz, L, Cn, W, int(activation == "silu"), _DT[x.dtype], _ptr(out), _stream(stream)))
    return out


def group_rmsnorm_(y: torch.Tensor, weight: torch.Tensor, *, group_size: int,
                   eps: float = 1e-5, stream=None) -> torch.Tensor:
    """In-place RMSNorm over groups of group_size consecutive channels of the
    last dimension (ssd_group_rmsnorm).  y: [..., dim] dense, e.g. the scan's
    gated out viewed as [batch, seqlen, nheads * headdim]; weight [dim] fp32."""
    if y.dtype not in _DT:
        raise ValueError("y must be float32 or bfloat16")
    dim = y.shape[-1]
    _need(y, "y", None, device=y.device)
    _need(weight, "weight", torch.float32, (dim,), y.device)
    rows = y.numel() // dim
    _lib.check(_lib.load().ssd_group_rmsnorm(_ptr(y), _ptr(weight), float(eps), rows, dim,
                                             int(group_size), _DT[y.dtype], _stream(stream)))
    return y


# --- decoding ----------------------------------------------------------------

def ssd_decode_step(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                    C: torch.Tensor, state: torch.Tensor, *,
                    dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
                    dt_limit: Tuple[float, float] = (0.0, math.inf),
                    D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One token per batch row (ssd_decode_step): x, z [batch, nheads,
    headdim]; dt [batch, nheads]; B, C [batch, ngroups, dstate]; state
    [batch, nheads, headdim, dstate] fp32, advanced in place.  Returns out
    [batch, nheads, headdim]."""
    if x.dtype not in _DT:
        raise ValueError("x must be float32 or bfloat16")
    Bsz, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    dev = x.device
    _need(x, "x", x.dtype, device=dev)
    _need(dt, "dt", x.dtype, (Bsz, H), dev)
    _need(A, "A", torch.float32, (H,), dev)
    _need(B, "B", x.dtype, (Bsz, G, N), dev)
    _need(C, "C", x.dtype, (Bsz, G, N), dev)
    _need(state, "state", torch.float32, (Bsz, H, P, N), dev)
    _need(dt_bias, "dt_bias", torch.float32, (H,), dev, optional=True)
    _need(D, "D", torch.float32, (H,), dev, optional=True)
    _need(z, "z", x.dtype, (Bsz, H, P), dev, optional=True)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", x.dtype, (Bsz, H, P), dev)
    lo, hi = dt_limit
    _lib.check(_lib.load().ssd_decode_step(
        _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)), float(lo), float(hi), _ptr(A),
        _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(state), Bsz, H, P, N, G, _DT[x.dtype],
        _ptr(out), _stream(stream)))
    return out


# --- backward -----------------------------------------------------------------

def bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                        dtype=torch.float32) -> int:
    return int(_lib.load().ssd_scan_bwd_ex_workspace_bytes(batch, seqlen, nheads, headdim,
                                                           dstate, ngroups, chunk_size,
                                                           _DT[dtype]))


def ssd_scan_bwd(dout: torch.Tensor, x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor,
                 B: torch.Tensor, C: torch.Tensor, *, chunk_size: int = 256,
                 dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
                 dt_limit: Tuple[float, float] = (0.0, math.inf),
                 D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                 initial_states: Optional[torch.Tensor] = None,
                 seq_idx: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Gradients of sum(out * dout) for the forward ssd_scan_fwd with the same
    arguments (dense tensors).  x, dt, B, C, z and dout are fp32
    (ssd_scan_bwd) or all bf16 (ssd_scan_bwd_ex: computed in fp32, the
    element-wise gradients returned in bf16); A, dt_bias, D, initial_states
    fp32.  Returns a dict with dx, ddt (w.r.t. the raw dt), dA, dB, dC,
    d_dt_bias, dD, and dz / d_initial_states when z / initial_states are
    given."""
    f32 = torch.float32
    xd = x.dtype
    if xd not in _DT:
        raise ValueError(f"x must be float32 or bfloat16, got {xd}")
    Bsz, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    _need(dout, "dout", xd, (Bsz, L, H, P), dev)
    _need(x, "x", xd, device=dev)
    _need(dt, "dt", xd, (Bsz, L, H), dev)
    _need(A, "A", f32, (H,), dev)
    _need(B, "B", xd, (Bsz, L, G, N), dev)
    _need(C, "C", xd, (Bsz, L, G, N), dev)
    _need(dt_bias, "dt_bias", f32, (H,), dev, optional=True)
    _need(D, "D", f32, (H,), dev, optional=True)
    _need(z, "z", xd, (Bsz, L, H, P), dev, optional=True)
    _need(initial_states, "initial_states", f32, (Bsz, H, P, N), dev, optional=True)
    _need(seq_idx, "seq_idx", torch.int32, (Bsz, L), dev, optional=True)
    lib = _lib.load()
    ws_need = int(lib.ssd_scan_bwd_ex_workspace_bytes(Bsz, L, H, P, N, G, chunk_size, _DT[xd]))
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    g = {"dx": torch.empty_like(x), "ddt": torch.empty_like(dt),
         "dA": torch.empty(H, dtype=f32, device=dev), "dB": torch.empty_like(B),
         "dC": torch.empty_like(C), "d_dt_bias": torch.empty(H, dtype=f32, device=dev),
         "dD": torch.empty(H, dtype=f32, device=dev),
         "dz": None if z is None else torch.empty_like(z),
         "d_initial_states": (None if initial_states is None
                              else torch.empty_like(initial_states))}
    lo, hi = dt_limit
    _lib.check(lib.ssd_scan_bwd_ex(
        _ptr(x), _ptr(dt), _ptr(dt_bias), int(bool(dt_softplus)), float(lo), float(hi),
        _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(initial_states), _ptr(seq_idx),
        _ptr(dout), Bsz, L, H, P, N, G, int(chunk_size), _DT[xd], _ptr(g["dx"]),
        _ptr(g["ddt"]), _ptr(g["d_dt_bias"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
        _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["d_initial_states"]), _ptr(workspace), ws_bytes,
        _stream(stream)))
    return g


# --- autograd ----------------------------------------------------------------

class _SSDScan(torch.autograd.Function):
    """ssd_scan_fwd forward, ssd_scan_bwd backward."""

    @staticmethod
    def forward(ctx, x, dt, A, B, C, dt_bias, D, z, initial_states, seq_idx, chunk_size,
                dt_softplus, dt_limit):
        out = ssd_scan_fwd(x, dt, A, B, C, chunk_size=chunk_size, dt_bias=dt_bias,
                           dt_softplus=dt_softplus, dt_limit=dt_limit, D=D, z=z,
                           initial_states=initial_states, seq_idx=seq_idx)
        ctx.save_for_backward(x, dt, A, B, C, dt_bias, D, z, initial_states, seq_idx)
        ctx.opts = (chunk_size, dt_softplus, dt_limit)
        return out

    @staticmethod
    def backward(ctx, dout):
        x, dt, A, B, C, dt_bias, D, z, initial_states, seq_idx = ctx.saved_tensors
        chunk_size, dt_softplus, dt_limit = ctx.opts
        # the backward takes dense tensors (views of a projection are copied)
        x, dt, B, C = x.contiguous(), dt.contiguous(), B.contiguous(), C.contiguous()
        z = None if z is None else z.contiguous()
        g = ssd_scan_bwd(dout.contiguous(), x, dt, A, B, C, chunk_size=chunk_size,
                         dt_bias=dt_bias, dt_softplus=dt_softplus, dt_limit=dt_limit, D=D, z=z,
                         initial_states=initial_states, seq_idx=seq_idx)
        return (g["dx"], g["ddt"], g["dA"], g["dB"], g["dC"],
                g["d_dt_bias"] if dt_bias is not None else None,
                g["dD"] if D is not None else None, g["dz"], g["d_initial_states"],
                None, None, None, None)


def ssd_scan(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             C: torch.Tensor, *, chunk_size: int = 256, dt_bias: Optional[torch.Tensor] = None,
             dt_softplus: bool = True, dt_limit: Tuple[float, float] = (0.0, math.inf),
             D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
             initial_states: Optional[torch.Tensor] = None,
             seq_idx: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The scan as a differentiable torch function (x, dt, B, C, z fp32 or
    bf16): the forward is ssd_scan_fwd, the backward ssd_scan_bwd (computed
    in fp32), giving gradients for x, dt (raw), A, B, C, dt_bias, D, z and
    initial_states.  Returns out."""
    return _SSDScan.apply(x, dt, A, B, C, dt_bias, D, z, initial_states, seq_idx, chunk_size,
                          dt_softplus, tuple(dt_limit))
