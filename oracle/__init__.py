"""CPU float64 oracle for the fused QKV context-encoding projection.

Test infrastructure only: the product path never imports this package.
"""
from .qkv_cte_oracle import (  # noqa: F401
    decode_bf16, decode_e4m3, decode_ue8m0, dequant_activations, dequant_weights, project,
    segments, segment_sumsq, inv_rms, rotate_half, apply_norm_rope, qkv_cte,
    qkv_cte_from_inputs, to_nbsd, encode_e4m3, row_quantise, pack_rows, unpack_rows,
    head_norm, rope_interleaved, interleaved_to_rotate_half, permute_qk_rows,
    NORM_NONE, NORM_ACROSS_HEADS, NORM_HEAD_RMS, NORM_HEAD_LAYER,
    SEG_Q, SEG_K, SEG_V,
)
