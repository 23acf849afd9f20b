"""Test infrastructure: a plain, slow, float64 CPU oracle of the expert attention path.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package. The product library never links, imports or
calls it, and it shares no code, tables or constants with the CUDA path.

Modules
-------
expert_attention : the per-layer attention of the flow-matching action expert
                   (q/k RMSNorm, HF rotate_half RoPE, tail placement, masked
                   non-causal GQA softmax attention), written out in fp64.
fp8_e4m3         : the OCP E4M3 ("e4m3fn") code table, a round-to-nearest-even
                   saturating encoder, and the per-(kv head, 128-row block)
                   cache quantiser used by the FP8 cache variant.
mxfp4            : the OCP MX FP4 format: E2M1 codes, a round-to-nearest-even
                   saturating encoder, and one power-of-two scale per 32 channels
                   of a cache row (the 4-bit cache variant).
decoder_layer    : the whole decoder layer around that attention (RMSNorm, fused
                   qkv projection, head split, attention, head concat, wo, residual,
                   RMSNorm, SwiGLU MLP, residual), for synthetic weights.
decode_attention : the text model's single-token decode attention over the same caches
                   (64 query heads / 8 KV heads, norm and RoPE at pos + rope_delta, the
                   new row written at pos, attention over rows 0..pos).

Every function is pinned by ``tests/test_oracle_pins.py``, ``tests/test_oracle_fp8_pins.py``,
``tests/test_oracle_layer_pins.py``, ``tests/test_oracle_decode_pins.py`` and
``tests/test_oracle_mxfp4_pins.py`` against closed forms, invariants, brute force on tiny
inputs and independent library routines.
"""
from .expert_attention import (  # noqa: F401
    D, EPS, HQ, HKV, MASK_MIN, REP, T, THETA,
    attention_concat, attention_tail_masked, bf16_round, expert_attention_layer,
    expert_attention_layer_fp8, expert_attention_layer_mxfp4, inv_freq, prologue, rms_norm,
    rope_angles, rope_rotate_half,
)
from .mxfp4 import (  # noqa: F401
    E2M1_MAX, MX_BLOCK, block_exponent, decode_e2m1, dequantize_rows, e2m1_magnitudes,
    encode_e2m1_rne_sat, quantize_rows,
)
from .fp8_e4m3 import (  # noqa: F401
    E4M3_MAX, decode_e4m3, dequantize_cache, e4m3_magnitudes, encode_e4m3_rne_sat,
    quantize_cache_blocks, quantize_tail_rows,
)
from .decoder_layer import (  # noqa: F401
    HIDDEN, INTER, KV_DIM, Q_DIM, QKV_DIM, concat_heads, expert_layer, linear, silu,
    split_qkv_heads, swiglu_mlp,
)
from .decode_attention import (  # noqa: F401
    HKV_TEXT, HQ_TEXT, REP_TEXT, decode_attend, decode_prologue, text_decode_attention,
)
