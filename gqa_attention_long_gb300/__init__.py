"""GB300-native (sm_103a) expert attention: the per-layer attention of a flow-matching action
expert over a long VLM KV cache (16 query heads, 8 KV heads, head width 128, 64 tokens).

The compute path is the C-ABI library ``libexpert_attn.so`` (hand-written CUDA kernels); this
package holds its ctypes binding, its build script and the seeded synthetic input generator.
"""
from ._lib import (  # noqa: F401
    EA_KV_BF16, EA_KV_FP8_E4M3, EA_OK, ExpertAttnError, LayerBuffers, alloc_workspace,
    expert_attn_layer, expert_attn_layers, expert_attn_layers_profiled, expert_attn_prologue,
    expert_attn_quantize_cache, expert_attn_quantize_cache_mxfp4, expert_attn_read_status,
    expert_attn_selftest_wait_timeout, expert_attn_set_splits,
    expert_attn_status_string, expert_attn_workspace_init, expert_attn_workspace_size,
    kernels_per_call, lib, make_args, split_parts, split_units,
    alloc_decoder_layer_workspace, expert_decoder_layer, expert_decoder_layer_workspace_size,
    expert_linear64, expert_linear64_workspace_size,
    DecodeBuffers, alloc_decode_workspace, make_decode_args, text_decode_attention,
    text_decode_workspace_init, text_decode_workspace_size,
)
