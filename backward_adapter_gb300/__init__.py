"""GB300-native fused flash-attention training op (forward + backward).

The compute path is the C-ABI library libfa_train.so (hand-written sm_103a
CUDA kernels); this package holds its build script, the ctypes binding and
the seeded synthetic workloads used by tests and the benchmark.
"""
from .fa_train import (FaError, FaParams, bwd, bwd_accum, bwd_accum_rows, bwd_noalloc, bwd_q8,  # noqa: F401
                       bwd_workspace_size, device_status, fwd, fwd_q8, fwd_workspace_size, load_library,
                       make_params, set_rows_backward)
