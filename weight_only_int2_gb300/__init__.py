"""GB300 (sm_103a) weight-only quantized linear layers: WNA16 for 2..8-bit
codes, W4A8, and the quantized-embedding gather, behind the C ABI of libwq.so.

The Python functions here marshal arguments into that ABI; all arithmetic runs
in the library's CUDA kernels.
"""
from ._lib import (  # noqa: F401
    LIB_PATH,
    WQError,
    act_quant_int8,
    check_status,
    ROUTES,
    debug_decode_plan,
    debug_mma_peak,
    debug_route,
    debug_unpack,
    debug_w4a8_group_acc,
    drop_workspaces,
    load,
    packed_words_per_row,
    qembed_gather,
    version,
    w4a8_gemm,
    w4a8_scratch_bytes,
    w4a8_workspace_bytes,
    scratch,
    wna16_gemm,
    wna16_gemm_noalloc,
    wna16_gemm_zp,
    wna16_moe_gemm,
    wna16_repack,
    wna16_workspace_bytes,
    wna16_zp_workspace_bytes,
    workspace,
)
