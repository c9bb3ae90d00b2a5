"""libbfp8 for Python: the GB300-native blocked W8A8 FP8 linear layer.

    q, s = bfp8_group_quant(x, col_major=True)      # 1x128 groups, amax/448 scales
    out  = bfp8_gemm(q, B, s, Bs)                   # 128x128 weight-scale tiles, bf16 out

Both run in libbfp8's sm_103a kernels (see include/bfp8.h); this package only
marshals tensors into the C ABI.  `workloads` draws the seeded synthetic inputs
and `metrics` holds the FLOP / byte accounting.
"""
from ._binding import (  # noqa: F401
    BFP8Error, BFP8_OK, EXPORTS, GemmOptions,
    KSPLIT_AUTO, KSPLIT_CLUSTER, KSPLIT_NONE, KSPLIT_STREAM_K, PAIRS_ALWAYS, PAIRS_AUTO, PAIRS_NEVER,
    SCALE_FP32, SCALE_UE8M0, SCHEDULE_AUTO, SCHEDULE_GEMV, SCHEDULE_SWAP_AB, SCHEDULE_WIDE,
    LIB_PATH, bfp8_device_status, bfp8_gemm, bfp8_gemm_fused, bfp8_gemm_grouped,
    bfp8_gemm_grouped_workspace_size, bfp8_gemm_plan, bfp8_linear, bfp8_linear_workspace_size, bfp8_gemm_workspace_size, bfp8_group_quant,
    bfp8_scale_ceil_ue8m0, bfp8_last_error, bfp8_plan_unit, bfp8_scale_ld,
    bfp8_selftest_bounded_wait, bfp8_version, drop_workspaces, lib, linear, workspace_for,
)
