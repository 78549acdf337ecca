"""GB300-native persistent FP16 GEMM (C[M,N] = A[M,K] @ B[K,N], FP32 accumulate).

The compute path is the C-ABI library ``libgemm_f16.so`` built from ``csrc/``
(hand-written CUDA for sm_103a). This package only marshals arguments to it;
importing the package does not load the library, and every call raises if the
library has not been built.
"""
from .binding import (  # noqa: F401
    GemmError, SCHED_GROUPED, SCHED_CROSS_TILE, SCHED_SINGLE_CTA, SCHED_NON_PERSISTENT, SCHED_DYNAMIC, SCHED_TAIL_SPLIT,
    sched_flags, gemm, gemm_raw, tile_map, get_config,
    sync_status, status_str, kernel_info, load_library, library_path, set_wait_timeout,
    gemm_from_host, selftest_wait_timeout, selftest_pair_abort, selftest_check, HostPipeline, gemm_splitk, splitk_workspace_size,
    gemm_splitk_noalloc, gemm_packed, packed_workspace_size,
)
