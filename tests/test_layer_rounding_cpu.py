"""The decoder layer's GPU parity bar against a model of the device's roundings (CPU only).

The device path of ``expert_decoder_layer`` keeps the layer's activations in bf16 and fuses both
RMSNorms into the projections that read them: ``bf16(gain * x)`` enters the tensor cores and
``1 / rms`` (from the rows' sums of squares over all channels) scales the fp32 sums, whose
result is rounded to bf16 once. This test models those roundings step by step on the CPU
(fp64 arithmetic, a bf16 rounding at every point where the device stores bf16; the attention as
the oracle's, on bf16 q/k/v, its output rounded to bf16) and checks that the modelled layer
output stays within 60 % of the bar that the GPU test applies (relative L2 6e-3, max-abs
6e-2; the model gives ~2.9e-3 and ~3.3e-2, about one bf16 step of |x2| up to 5), so that the bar
keeps a margin for what the model leaves out (fp32 instead of fp64 sums, the attention kernel's
own internal roundings). It also checks that the model is
not trivially exact (its error is of the size one bf16 rounding per stored tensor gives).
"""
import numpy as np

import oracle
from gqa_attention_long_gb300.inputs import expert_layer_weights, layer_inputs, residual_stream
from oracle.expert_attention import EPS, bf16_round
from tests._gpu_util import f64

LAYER_REL_L2 = 6e-3   # the GPU test's bar (tests/test_gpu_layer.py)
LAYER_MAX_ABS = 6e-2


def _inv_rms(x: np.ndarray) -> np.ndarray:
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)


def device_model(x, w: dict, k_cache, v_cache, S: int, Smax: int, rope_delta: int) -> np.ndarray:
    """The layer with the device's bf16 storage points and fused RMSNorms (see the module)."""
    lin = oracle.decoder_layer.linear
    hq = bf16_round(w["ln1"] * x)                                   # bf16(gain * x) into wqkv
    qkv = bf16_round(_inv_rms(x) * lin(hq, w["wqkv"]))              # 1/rms on the sums, bf16 out
    q_raw, k_raw, v_raw = oracle.decoder_layer.split_qkv_heads(qkv)
    r = oracle.expert_attention_layer(q_raw, k_raw, v_raw, w["q_norm"], w["k_norm"], k_cache, v_cache,
                                      S, Smax, rope_delta)
    attn = bf16_round(r["out"])
    x1 = bf16_round(x + lin(oracle.decoder_layer.concat_heads(attn), w["wo"]))
    h2q = bf16_round(w["ln2"] * x1)
    s2 = _inv_rms(x1)
    gu = bf16_round(oracle.decoder_layer.silu(s2 * lin(h2q, w["w1"])) * (s2 * lin(h2q, w["w3"])))
    return bf16_round(x1 + lin(gu, w["w2"]))


def test_fused_norm_rounding_model_within_the_gpu_bar_with_margin():
    S, Smax, seed = 256, 512, 11   # the GPU test's first case, at the model's widths
    lay = layer_inputs(seed, S, Smax)
    w = expert_layer_weights(seed)
    x = f64(residual_stream(seed))
    wd = {k: f64(v) for k, v in w.__dict__.items()}
    kc, vc = f64(lay.k_cache), f64(lay.v_cache)
    ref = oracle.expert_layer(x, wd, kc, vc, S, Smax, 0)["x2"]
    got = device_model(x, wd, kc, vc, S, Smax, 0)
    mx = float(np.max(np.abs(got - ref)))
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= 0.6 * LAYER_REL_L2 and mx <= 0.6 * LAYER_MAX_ABS, f"max-abs {mx:.3e}, rel-L2 {rel:.3e}"
    # the model does round: one bf16 step of |x2| (up to ~5) is 0.03, so a model that rounded
    # nothing would be far below this
    assert rel > 1e-4
