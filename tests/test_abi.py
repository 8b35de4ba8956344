"""The C-ABI library loads and exports every symbol include/*.h declares;
host-side validation answers before anything touches a GPU."""
import math
import re
from pathlib import Path

import pytest

from selective_state_space_05_gb300 import _lib

ROOT = Path(__file__).resolve().parent.parent


def declared_functions():
    names = []
    for h in sorted((ROOT / "include").glob("*.h")):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(ssd_[a-z0-9_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_05_gb300 import build
    build.build()
    return _lib.load()


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for n in ("ssd_scan_fwd", "ssd_last_error", "ssd_abi_version", "ssd_scan_workspace_bytes",
              "ssd_dt_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan",
              "ssd_chunk_fused", "ssd_scan_bwd", "ssd_scan_bwd_workspace_bytes",
              "ssd_scan_workspace_bytes_min"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_abi_version(lib):
    assert lib.ssd_abi_version() == 3


def test_workspace_bytes(lib):
    # dt + cumsum [B,H,nc,Q] f32, segments [B,nc,Q] i32, states [B,nc,H,P,N] f32
    B, L, H, P, N, G, Q = 8, 4096, 80, 64, 128, 1, 256
    nc = L // Q
    ctrl = (64 + B * H) * 4
    want = ctrl + 2 * B * H * nc * Q * 4 + B * nc * Q * 4 + B * nc * H * P * N * 4
    got = lib.ssd_scan_workspace_bytes(B, L, H, P, N, G, Q, _lib.SSD_DTYPE_BF16)
    assert want <= got <= want + 5 * 256
    # fp32 at chunk 256 runs its stages at 128 tokens (the fp32 tensor-core
    # stages' chunk), so its states are counted per 128-token chunk, plus
    # C B^T per (batch, chunk, group), computed once for all heads, and B
    # pre-split as chunk_state's tiles (dstate 128)
    nc2 = L // 128
    want32 = (ctrl + 2 * B * H * nc2 * 128 * 4 + B * nc2 * 128 * 4 + B * nc2 * H * P * N * 4
              + B * nc2 * G * 128 * 128 * 4 + B * nc2 * G * 8 * 128 * 16 * 2 * 4)
    got32 = lib.ssd_scan_workspace_bytes(B, L, H, P, N, G, Q, _lib.SSD_DTYPE_F32)
    assert want32 <= got32 <= want32 + 7 * 256
    assert lib.ssd_scan_workspace_bytes(B, L, H, P, N, G, 100, 1) == 0      # bad chunk
    assert lib.ssd_scan_workspace_bytes(B, L, H, 48, N, G, Q, 1) == 0       # bad headdim
    assert lib.ssd_scan_workspace_bytes(B, L, 80, P, N, 3, Q, 1) == 0       # H % G != 0


def test_least_workspace(lib):
    """ssd_scan_workspace_bytes_min: below the full size only for bf16 shapes
    outside the fused kernel, by the fp32 copies of x, z, out (B*L*H*P each)
    and B, C (B*L*G*N each), each piece on a 256-byte boundary; the least
    size is then the bf16 stage kernels' workspace at the caller's chunk."""
    BF, F32 = _lib.SSD_DTYPE_BF16, _lib.SSD_DTYPE_F32

    def sizes(*a):
        return lib.ssd_scan_workspace_bytes(*a), lib.ssd_scan_workspace_bytes_min(*a)

    def up(v):
        return (v + 255) // 256 * 256

    # fused shape (bf16) and fp32: nothing to leave out
    for dt in (BF, F32):
        full, least = sizes(8, 4096, 80, 64, 128, 1, 256, dt)
        assert 0 < least == full
    # bf16, headdim 128: the fp32 stages on copies
    B, L, H, P, N, G, Q = 2, 1000, 4, 128, 64, 2, 256
    full, least = sizes(B, L, H, P, N, G, Q, BF)
    xs, bs = B * L * H * P * 4, B * L * G * N * 4
    copies = 3 * up(xs) + 2 * up(bs)
    nc = -(-L // Q)   # the stage kernels' chunk: the caller's 256
    stage = ((64 + B * H) * 4 + 2 * B * H * nc * Q * 4 + B * nc * Q * 4
             + B * nc * H * P * N * 4)
    assert stage <= least <= stage + 5 * 256
    assert least < full and full >= copies
    assert lib.ssd_scan_workspace_bytes_min(B, L, H, 48, N, G, Q, BF) == 0   # bad headdim


def _fwd(lib, **kw):
    a = dict(x=16, dt=16, dt_bias=None, sp=1, lo=0.0, hi=math.inf, A=16, B=16, C=16, D=None,
             z=None, init=None, seq=None, batch=1, L=64, H=2, P=16, N=16, G=1, Q=64, dtype=0,
             out=16, fin=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.ssd_scan_fwd(a["x"], a["dt"], a["dt_bias"], a["sp"], a["lo"], a["hi"], a["A"],
                            a["B"], a["C"], a["D"], a["z"], a["init"], a["seq"], a["batch"],
                            a["L"], a["H"], a["P"], a["N"], a["G"], a["Q"], a["dtype"], a["out"],
                            a["fin"], a["ws"], a["wsb"], a["stream"])


def test_validation_errors_before_any_launch(lib):
    # fake (never dereferenced) addresses: validation fails before any CUDA call
    assert _fwd(lib, Q=100) == -4 and b"chunk_size" in lib.ssd_last_error()
    assert _fwd(lib, x=None) == -2
    assert _fwd(lib, x=24) == -3                      # not 16-byte aligned
    assert _fwd(lib, dtype=7) == -1
    assert _fwd(lib, H=3, G=2) == -1
    assert _fwd(lib, P=48) == -4
    assert _fwd(lib, N=8) == -4
    assert _fwd(lib, L=0) == -1                       # empty sequence
    assert _fwd(lib, batch=0) == -1                   # empty batch
    assert _fwd(lib, batch=-1) == -1
    assert _fwd(lib, H=0) == -1
    assert _fwd(lib, batch=65536) == -4               # above the supported batch
    assert _fwd(lib, lo=1.0, hi=0.5) == -1
    assert _fwd(lib, ws=4096, wsb=16) == -5           # caller workspace too small


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        saved = _lib._LIB
        _lib._LIB = None
        try:
            _lib.load(tmp_path / "nope.so")
        finally:
            _lib._LIB = saved


def test_host_workspace_bytes(lib):
    # two staging buffers of rows_per_slice rows (x, z, out, dt, B, C, seq_idx,
    # initial / final states and the slice's scan workspace) plus dt_bias, A, D
    B, L, H, P, N, G, Q = 8, 4096, 80, 64, 128, 1, 256
    bf16 = _lib.SSD_DTYPE_BF16
    for rows in (1, 2, 8):
        per_row = 3 * L * H * P * 2 + L * H * 2 + 2 * L * G * N * 2 + L * 4 + 2 * H * P * N * 4
        scan = lib.ssd_scan_workspace_bytes(rows, L, H, P, N, G, Q, bf16)
        want = 2 * (rows * per_row + scan)
        got = lib.ssd_scan_host_workspace_bytes(B, L, H, P, N, G, Q, bf16, rows)
        assert want <= got <= want + 2 * 11 * 256 + 3 * (H * 4 + 256)
    # default: an eighth of the batch per slice
    assert (lib.ssd_scan_host_workspace_bytes(B, L, H, P, N, G, Q, bf16, 0)
            == lib.ssd_scan_host_workspace_bytes(B, L, H, P, N, G, Q, bf16, 1))
    assert lib.ssd_scan_host_workspace_bytes(B, L, H, P, N, G, 100, bf16, 0) == 0   # bad chunk


def test_host_call_validation_before_any_cuda_call(lib):
    args = [16, 16, None, 1, 0.0, math.inf, 16, 16, 16, None, None, None, None,
            1, 64, 2, 16, 16, 1, 64, 0, 16, None, 0, None, 0, None]
    assert lib.ssd_scan_fwd_host(*args) == -2                # no workspace
    args[24], args[25] = 4096, 16
    assert lib.ssd_scan_fwd_host(*args) == -5                # workspace too small
    assert b"workspace" in lib.ssd_last_error()


def test_strided_validation_before_any_launch(lib):
    """Negative or huge strides are refused before anything is launched."""
    ok, bad, huge = _lib.Stride(1024, 64), _lib.Stride(-1, 64), _lib.Stride(1, 1 << 41)

    def call(xs=ok, dts=ok, bs=ok, cs=ok, zs=ok, z=None, x=16):
        return lib.ssd_scan_fwd_strided(x, xs, 16, dts, None, 1, 0.0, math.inf, 16, 16, bs, 16,
                                        cs, None, z, zs, None, None, 1, 64, 2, 16, 16, 1, 64, 0,
                                        16, None, None, 0, None)
    assert call(xs=bad) == -1 and b"x strides" in lib.ssd_last_error()
    assert call(dts=huge) == -1 and b"dt strides" in lib.ssd_last_error()
    assert call(cs=bad) == -1
    assert call(zs=bad, z=16) == -1 and b"z strides" in lib.ssd_last_error()
    assert call(x=None) == -2
    assert call(x=24) == -3


def test_header_declares_status_and_strided_calls():
    names = declared_functions()
    assert "ssd_scan_status" in names and "ssd_scan_fwd_strided" in names
    text = (ROOT / "include" / "ssd_scan.h").read_text()
    assert "SSD_ERR_TIMEOUT = -7" in text


def test_decode_step_validation_before_any_launch(lib):
    def call(**kw):
        a = dict(x=16, dt=16, bias=None, sp=1, lo=0.0, hi=math.inf, A=16, B=16, C=16, D=None,
                 z=None, state=16, batch=1, H=2, P=64, N=128, G=1, dtype=1, out=16)
        a.update(kw)
        return lib.ssd_decode_step(a["x"], a["dt"], a["bias"], a["sp"], a["lo"], a["hi"], a["A"],
                                   a["B"], a["C"], a["D"], a["z"], a["state"], a["batch"], a["H"],
                                   a["P"], a["N"], a["G"], a["dtype"], a["out"], None)
    assert call(N=12) == -4 and b"dstate" in lib.ssd_last_error()
    assert call(H=3, G=2) == -1
    assert call(state=None) == -2
    assert call(state=24) == -3
    assert call(lo=1.0, hi=0.5) == -1
    assert call(dtype=5) == -1


def test_backward_validation_before_any_launch(lib):
    B, L, H, P, N, G, Q = 2, 100, 4, 32, 64, 2, 64
    need = lib.ssd_scan_bwd_workspace_bytes(B, L, H, P, N, G, Q)
    assert need > 0
    assert lib.ssd_scan_bwd_workspace_bytes(B, L, H, P, 48, G, Q) == 0
    assert lib.ssd_scan_bwd_workspace_bytes(B, L, H, 256, N, G, Q) == 0

    def call(**kw):
        a = dict(x=16, dt=16, bias=None, sp=1, lo=0.0, hi=math.inf, A=16, B=16, C=16, D=None,
                 z=None, h0=None, seq=None, dout=16, batch=B, L=L, H=H, P=P, N=N, G=G, Q=Q,
                 dx=16, ddt=16, dbias=None, dA=16, dB=16, dC=16, dD=None, dz=None, dh0=None,
                 ws=16, wsb=need)
        a.update(kw)
        return lib.ssd_scan_bwd(a["x"], a["dt"], a["bias"], a["sp"], a["lo"], a["hi"], a["A"],
                                a["B"], a["C"], a["D"], a["z"], a["h0"], a["seq"], a["dout"],
                                a["batch"], a["L"], a["H"], a["P"], a["N"], a["G"], a["Q"],
                                a["dx"], a["ddt"], a["dbias"], a["dA"], a["dB"], a["dC"], a["dD"],
                                a["dz"], a["dh0"], a["ws"], a["wsb"], None)
    assert call(N=48) == -4 and b"dstate" in lib.ssd_last_error()
    assert call(Q=100) == -4
    assert call(H=3) == -4                 # ngroups must divide nheads
    assert call(lo=1.0, hi=0.5) == -1
    assert call(dout=None) == -2
    assert call(z=16) == -2                # dz is required with z
    assert call(dB=24) == -3
    assert call(wsb=need - 1) == -5


def test_backward_ex_workspace_and_validation(lib):
    B, L, H, P, N, G, Q = 2, 100, 4, 32, 64, 2, 64
    f32 = lib.ssd_scan_bwd_ex_workspace_bytes(B, L, H, P, N, G, Q, _lib.SSD_DTYPE_F32)
    assert f32 == lib.ssd_scan_bwd_workspace_bytes(B, L, H, P, N, G, Q)
    bf = lib.ssd_scan_bwd_ex_workspace_bytes(B, L, H, P, N, G, Q, _lib.SSD_DTYPE_BF16)
    assert bf > f32
    assert lib.ssd_scan_bwd_ex_workspace_bytes(B, L, H, P, N, G, Q, 7) == 0
    assert lib.ssd_scan_bwd_ex_workspace_bytes(B, L, H, P, 48, G, Q, _lib.SSD_DTYPE_BF16) == 0

    def call(**kw):
        a = dict(x=16, dt=16, B=16, C=16, z=None, dout=16, dtype=_lib.SSD_DTYPE_BF16, dx=16,
                 ddt=16, dB=16, dC=16, dz=None, wsb=bf)
        a.update(kw)
        return lib.ssd_scan_bwd_ex(a["x"], a["dt"], None, 1, 0.0, math.inf, 16, a["B"], a["C"],
                                   None, a["z"], None, None, a["dout"], B, L, H, P, N, G, Q,
                                   a["dtype"], a["dx"], a["ddt"], None, 16, a["dB"], a["dC"],
                                   None, a["dz"], None, 16, a["wsb"], None)
    assert call(dtype=7) == -1
    assert call(dout=None) == -2
    assert call(z=16) == -2
    assert call(dC=24) == -3
    assert call(wsb=bf - 1) == -5
