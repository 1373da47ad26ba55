"""GB300-native Kimi Delta Attention (KDA): chunked forward and decode, plus
lightning attention (fixed per-head decay) forward and decode.

The compute lives in ``libkda.so`` (CUDA for sm_103a, C ABI in
``include/kda.h``); ``gated_delta_rule_40_gb300.kda`` is its Python binding.
Build the library with ``gated_delta_rule_40_gb300.build.build()``.
"""
from .kda import (  # noqa: F401
    KdaError,
    KdaLibraryError,
    kda_bwd,
    kda_decode_step,
    kda_decode_tokens,
    kda_fwd,
    kda_fwd_bf16_state,
    kda_fwd_host,
    kda_fwd_noalloc,
    kda_fwd_scalar_gate,
    kda_fwd_workspace_size,
    kda_get_status,
    kda_la_decode,
    kda_la_fwd,
    kda_last_launch_count,
    load,
    status_string,
)
