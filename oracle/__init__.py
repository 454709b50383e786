"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference arm.  The product path never imports it.
"""
from .attention_ref import (  # noqa: F401
    attn_fwd_ref,
    attn_fwd_ref_rows,
    attn_fwd_ref_end_aligned,
    attn_bwd_ref,
    attn_bwd_ref_sampled,
    attn_fwd_dropout_ref,
    attn_bwd_dropout_ref,
    philox4x32_10,
    dropout_keep,
    dropout_threshold,
    dropout_scale,
    bwd_preprocess_ref,
    online_softmax_scalar,
    online_softmax_blocks,
    merge_two_blocks,
    attn_fwd_tiled_ref,
    max_abs_err,
    rel_fro_err,
    lse_max_abs_err,
)
from . import fp8_ref  # noqa: F401,E402  (e4m3 quantisation and the FP8 forward)
