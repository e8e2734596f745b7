"""GB300-native (sm_103a) fused QKV context-encoding projection.

The computation runs in libqkvcte.so (hand-written CUDA: a tcgen05 MXFP8 GEMM with
a fused dequant/bias/sum-of-squares epilogue, then an in-place across-heads
RMSNorm + rotate-half RoPE pass, and the producer step that quantises bf16
activations per row or unpacks packed [T, H + 4] rows). This package is the thin binding over its C ABI
(include/qkv_cte.h) plus the in-tree build script.
"""
from .qkv_cte import (  # noqa: F401
    EXPORTED, QKV_CTE_ERR_ARCH, QKV_CTE_ERR_CUDA, QKV_CTE_ERR_DEVICE_TIMEOUT, QKV_CTE_ERR_INVALID,
    QKV_CTE_ERR_UNSUPPORTED, QKV_CTE_FLAG_GEMM_CTA_PAIR, QKV_CTE_FLAG_GEMM_SINGLE_CTA, QKV_CTE_FLAG_PROFILE, QKV_CTE_FLAG_NORM_IN_GEMM, QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE, QKV_CTE_FLAG_SERIAL_PASSES, QKV_CTE_FLAG_TEST_STALL, QKV_CTE_LAYOUT_BSD, QKV_CTE_LAYOUT_NBSD,
    QKV_CTE_INPUT_BF16, QKV_CTE_INPUT_PACKED, QKV_CTE_INPUT_ROW_FP8,
    QKV_CTE_NORM_ACROSS_HEADS, QKV_CTE_NORM_HEAD_LAYER, QKV_CTE_NORM_HEAD_RMS, QKV_CTE_NORM_NONE,
    QKV_CTE_MODE_FUSED, QKV_CTE_MODE_SEPARATE, QKV_CTE_NOALLOC_SCRATCH_BYTES, QKV_CTE_OK, QkvCte, QkvCteError, library_path, load,
    make_desc, qkv_cte_desc, qkv_cte_destroy, qkv_cte_get_plan_info, qkv_cte_last_error, qkv_cte_pass_times, qkv_cte_plan, qkv_cte_run, qkv_cte_run_noalloc,
    qkv_cte_row_quantize, qkv_cte_unpack_rows, qkv_cte_interleaved_to_rotate_half,
    qkv_cte_run_host, qkv_cte_host_scratch_bytes,
    qkv_cte_status, qkv_cte_version,
)
