"""ctypes view of ``libssd_gb300.so`` (the C ABI declared in include/ssd_scan.h).

Argument marshalling only.  Loading fails loudly when the library has not been
built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libssd_gb300.so"

SSD_DTYPE_F32 = 0
SSD_DTYPE_BF16 = 1
SSD_NOALLOC_SCRATCH_BYTES = 64 << 20   # static scratch of ssd_scan_fwd_noalloc

SSD_OK = 0
SSD_ERR_TIMEOUT = -7
ERRORS = {-1: "SSD_ERR_ARG", -2: "SSD_ERR_NULL", -3: "SSD_ERR_ALIGN",
          -4: "SSD_ERR_UNSUPPORTED", -5: "SSD_ERR_WORKSPACE", -6: "SSD_ERR_CUDA",
          -7: "SSD_ERR_TIMEOUT"}


class Stride(ctypes.Structure):
    """ssd_stride_t: element strides between batch rows and between tokens."""
    _fields_ = [("batch", ctypes.c_int64), ("token", ctypes.c_int64)]


_vp = ctypes.c_void_p
_i, _i64, _f, _sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_st = Stride

# every symbol the header declares, with (restype, argtypes); pointers are
# passed as integers (device addresses) through c_void_p
SIGNATURES = {
    "ssd_abi_version": (_i, []),
    "ssd_last_error": (ctypes.c_char_p, []),
    "ssd_scan_status": (_i, [_i, _vp]),
    "ssd_causal_conv1d": (_i, [_vp, _st, _vp, _vp, _vp, _i64, _i64, _i, _i, _i, _i, _vp, _vp]),
    "ssd_group_rmsnorm": (_i, [_vp, _vp, _f, _i64, _i, _i, _i, _vp]),
    "ssd_decode_step": (_i, [_vp, _vp, _vp, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i, _i,
                             _i, _i, _i, _vp, _vp]),
    "ssd_scan_fwd_strided": (_i, [_vp, _st, _vp, _st, _vp, _i, _f, _f, _vp, _vp, _st, _vp, _st,
                                  _vp, _vp, _st, _vp, _vp, _i64, _i64, _i, _i, _i, _i, _i, _i,
                                  _vp, _vp, _vp, _sz, _vp]),
    "ssd_scan_workspace_bytes": (_sz, [_i64, _i64, _i, _i, _i, _i, _i, _i]),
    "ssd_scan_workspace_bytes_min": (_sz, [_i64, _i64, _i, _i, _i, _i, _i, _i]),
    "ssd_scan_bwd_workspace_bytes": (_sz, [_i64, _i64, _i, _i, _i, _i, _i]),
    "ssd_scan_bwd_ex_workspace_bytes": (_sz, [_i64, _i64, _i, _i, _i, _i, _i, _i]),
    "ssd_scan_bwd_ex": (_i, [_vp, _vp, _vp, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                             _i64, _i64, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                             _vp, _vp, _vp, _vp, _sz, _vp]),
    "ssd_scan_bwd": (_i, [_vp, _vp, _vp, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                          _i64, _i64, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                          _vp, _vp, _vp, _sz, _vp]),
    "ssd_scan_fwd": (_i, [_vp, _vp, _vp, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                          _i64, _i64, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "ssd_dt_cumsum": (_i, [_vp, _vp, _i, _f, _f, _vp, _vp, _i64, _i64, _i, _i, _i,
                           _vp, _vp, _vp, _vp]),
    "ssd_chunk_state": (_i, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i, _i, _i, _i, _i,
                             _vp, _vp]),
    "ssd_state_passing": (_i, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i, _i, _i, _vp]),
    "ssd_chunk_fused": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i,
                             _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "ssd_scan_fwd_noalloc": (_i, [_vp, _vp, _vp, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _i64, _i64, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp]),
    "ssd_chunk_scan": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i,
                            _i, _i, _i, _i, _vp, _vp]),
    "ssd_scan_host_workspace_bytes": (_sz, [_i64, _i64, _i, _i, _i, _i, _i, _i, _i64]),
    "ssd_scan_fwd_host": (_i, [_vp, _vp, _vp, _i, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                               _i64, _i64, _i, _i, _i, _i, _i, _i, _vp, _vp, _i64, _vp, _sz,
                               _vp]),
}

_LIB = None


def load(path: Path = LIB_PATH) -> ctypes.CDLL:
    """Load the library once.  Raises if it is missing (build it with
    ``python -c "import __graft_entry__ as g; g.build()"``)."""
    global _LIB
    if _LIB is None:
        if not Path(path).exists():
            raise RuntimeError(f"CUDA library not built: {path} is missing")
        lib = ctypes.CDLL(str(path))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


class SSDError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def check(code: int) -> None:
    if code != SSD_OK:
        raise SSDError(code, load().ssd_last_error().decode())
