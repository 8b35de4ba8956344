"""GB300-native (sm_103a) Mamba-2 SSD chunked scan: forward, backward,
decode step and the block's conv1d and grouped norm.

The computation lives in ``libssd_gb300.so`` (CUDA kernels behind the C ABI
of include/ssd_scan.h); this package only marshals torch tensors into it.
"""
from .scan import (abi_version, bwd_workspace_bytes, causal_conv1d,  # noqa: F401
                   group_rmsnorm_, host_workspace_bytes, scan_status, ssd_chunk_fused,
                   ssd_chunk_scan, ssd_chunk_state, ssd_decode_step, ssd_dt_cumsum,
                   ssd_scan, ssd_scan_bwd, ssd_scan_fwd, ssd_scan_fwd_host, ssd_state_passing,
                   workspace_bytes)
