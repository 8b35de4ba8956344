"""CPU fp64 oracle of the SSD chunked-scan forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.
"""
from .ssd_oracle import (causal_conv1d, dt_process, dt_process_c, f64,  # noqa: F401
                         group_rmsnorm, scan_chunked,
                         scan_quadratic, scan_sequential, default_threads)
