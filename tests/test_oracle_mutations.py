"""Plants plausible mistakes in the oracle (CPU only) and checks that its pins catch each one.

The mistakes are patched into the oracle module for the duration of one test; nothing on the
CUDA path is involved.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.expert_attention as ea
from tests import test_oracle_pins as pins


def _rope_wrong_sign(x, pos, theta=ea.THETA):
    x = np.asarray(x, dtype=np.float64)
    a = ea.rope_angles(pos, theta, x.shape[-1])
    cos = np.concatenate([np.cos(a), np.cos(a)], -1)
    sin = np.concatenate([np.sin(a), np.sin(a)], -1)
    rot = np.concatenate([x[..., 64:], -x[..., :64]], -1)   # planted: signs swapped
    return x * cos + rot * sin


def _rms_eps_outside(x, gamma, eps=ea.EPS):
    x = np.asarray(x, dtype=np.float64)
    return np.asarray(gamma) * x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps)  # planted


def _attend_wrong_scale(q, keys, vals, bias=None):
    s = (q @ keys.T) / ea.D                                  # planted: 1/D instead of 1/sqrt(D)
    if bias is not None:
        s = s + bias
    p = np.exp(s - s.max(-1, keepdims=True))
    return (p @ vals) / p.sum(-1, keepdims=True)


def _concat_wrong_group(q, k_cache, v_cache, S, k_own, v_own):
    out = np.empty((16, 64, 128))
    for h in range(16):
        g = h % 8                                            # planted: wrong GQA map
        keys = np.concatenate([np.asarray(k_cache[g, :S], np.float64), k_own[g]], 0)
        vals = np.concatenate([np.asarray(v_cache[g, :S], np.float64), v_own[g]], 0)
        out[h] = ea._softmax_attend(q[h], keys, vals)
    return out


def _inv_freq_wrong(theta=ea.THETA, dim=ea.D):
    return theta ** (-np.arange(dim // 2, dtype=np.float64) / dim)   # planted: missing factor 2


def _prologue_wrong_pos(q_raw, k_raw, v_raw, q_gamma, k_gamma, S, rope_delta):
    pos = np.arange(64) + int(rope_delta)                    # planted: S dropped from positions
    return (ea.rope_rotate_half(ea.rms_norm(q_raw, q_gamma), pos),
            ea.rope_rotate_half(ea.rms_norm(k_raw, k_gamma), pos), np.asarray(v_raw, np.float64))


MUTATIONS = [
    ("rope_rotate_half", _rope_wrong_sign, pins.test_rope_matches_complex_rotation),
    ("rms_norm", _rms_eps_outside, pins.test_rms_norm_eps_inside_the_root),
    ("_softmax_attend", _attend_wrong_scale, pins.test_matches_torch_sdpa_fp64),
    ("attention_concat", _concat_wrong_group, pins.test_gqa_group_mapping),
    ("inv_freq", _inv_freq_wrong, pins.test_inv_freq_closed_forms),
    ("prologue", _prologue_wrong_pos, pins.test_prologue_positions_are_t_plus_delta_plus_S),
]


@pytest.mark.parametrize("name,bad,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, bad, pin):
    monkeypatch.setattr(ea, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        pin()


def test_unpatched_pins_pass():
    for _, _, pin in MUTATIONS:
        pin()
    assert math.isfinite(1.0)


# ------------------------------------------------------------------ whole-layer oracle
import oracle.decoder_layer as el  # noqa: E402
from tests import test_oracle_layer_pins as lpins  # noqa: E402


def _silu_wrong(x):
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(x))                              # planted: sigmoid(-x)


def _split_kv_swapped(qkv):
    q, k, v = _split_reference(qkv)
    return q, v, k                                            # planted: k and v swapped


def _split_reference(qkv):
    q = qkv[:, :2048].reshape(64, 16, 128).transpose(1, 0, 2)
    k = qkv[:, 2048:3072].reshape(64, 8, 128).transpose(1, 0, 2)
    v = qkv[:, 3072:].reshape(64, 8, 128).transpose(1, 0, 2)
    return q, k, v


def _concat_no_transpose(a):
    return np.asarray(a, np.float64).reshape(64, 2048)       # planted: heads not interleaved per token


def _layer_missing_residual(x, w, k_cache, v_cache, S, Smax, rope_delta):
    r = _original_layer(x, w, k_cache, v_cache, S, Smax, rope_delta)
    r["x2"] = r["x2"] - r["x1"]                               # planted: second residual dropped
    return r


_original_layer = el.expert_layer

LAYER_MUTATIONS = [
    ("silu", _silu_wrong, lpins.test_matches_torch_composition),
    ("split_qkv_heads", _split_kv_swapped, lpins.test_kv_split_order),
    ("concat_heads", _concat_no_transpose, lpins.test_matches_torch_composition),
    ("expert_layer", _layer_missing_residual, lpins.test_zero_output_projections_leave_the_residual_stream),
]


@pytest.mark.parametrize("name,bad,pin", LAYER_MUTATIONS, ids=[m[0] for m in LAYER_MUTATIONS])
def test_layer_pin_catches_planted_mistake(monkeypatch, name, bad, pin):
    monkeypatch.setattr(el, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        pin()


def test_unpatched_layer_pins_pass():
    for _, _, pin in LAYER_MUTATIONS:
        pin()


# ------------------------------------------------------------- text-model decode oracle
import oracle.decode_attention as da  # noqa: E402
from tests import test_oracle_decode_pins as dpins  # noqa: E402


def _decode_attend_wrong_group(q, k_cache, v_cache, pos):
    out = np.empty((64, 128))
    for h in range(64):
        g = h % 8                                             # planted: wrong GQA map
        s = (np.asarray(k_cache[g, :pos + 1], np.float64) @ q[h]) / math.sqrt(128)
        w = np.exp(s - s.max())
        out[h] = (w @ np.asarray(v_cache[g, :pos + 1], np.float64)) / w.sum()
    return out


def _decode_attend_exclusive(q, k_cache, v_cache, pos):
    out = np.empty((64, 128))
    n = max(pos, 1)                                           # planted: cur_pos exclusive
    for h in range(64):
        g = h // 8
        s = (np.asarray(k_cache[g, :n], np.float64) @ q[h]) / math.sqrt(128)
        w = np.exp(s - s.max())
        out[h] = (w @ np.asarray(v_cache[g, :n], np.float64)) / w.sum()
    return out


def _decode_prologue_no_delta(q_raw, k_raw, v_raw, q_gamma, k_gamma, pos, rope_delta):
    return _original_decode_prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, pos, 0)  # planted


_original_decode_prologue = da.decode_prologue

DECODE_MUTATIONS = [
    ("decode_attend", _decode_attend_wrong_group, dpins.test_decode_gqa_group_mapping),
    ("decode_attend", _decode_attend_exclusive, dpins.test_decode_attends_to_its_own_new_row),
    ("decode_prologue", _decode_prologue_no_delta, dpins.test_decode_positions_are_pos_plus_delta),
]


@pytest.mark.parametrize("name,bad,pin", DECODE_MUTATIONS,
                         ids=["gqa_map", "exclusive_cur_pos", "no_rope_delta"])
def test_decode_pin_catches_planted_mistake(monkeypatch, name, bad, pin):
    monkeypatch.setattr(da, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        pin()


def test_unpatched_decode_pins_pass():
    for _, _, pin in DECODE_MUTATIONS:
        pin()


# ------------------------------------------------------------------ MXFP4 cache format
import oracle.mxfp4 as mx  # noqa: E402
from tests import test_oracle_mxfp4_pins as mpins  # noqa: E402


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    mags = mx.e2m1_magnitudes()
    hi = np.minimum(np.searchsorted(mags, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    code = np.where(mags[hi] - a <= a - mags[lo], hi, lo)    # planted: ties away from zero
    code = np.where(a >= 6.0, 7, np.where(a == 0.0, 0, code))
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def _block_exponent_emax3(amax):
    amax = float(amax)
    if amax == 0.0:
        return 0
    return int(max(int(np.frexp(amax)[1]) - 1 - 3, -127))    # planted: emax 3 instead of 2


def _magnitudes_bias2():
    codes = np.arange(8)
    e, m = codes >> 1, codes & 1
    return np.where(e == 0, m * 0.25, (1.0 + m / 2.0) * np.exp2(e - 2.0))   # planted: bias 2


def _quantize_whole_row(x):
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)                        # planted: one scale per row
    exps = np.vectorize(mx.block_exponent, otypes=[np.int64])(amax).astype(np.int16)
    codes = mx.encode_e2m1_rne_sat(x / np.exp2(exps.astype(np.float64)).astype(np.float32)[..., None])
    return codes, np.repeat(exps[..., None], 4, axis=-1)


def _layer_mxfp4_v_with_k_scales(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_codes, k_exps, v_codes,
                                 v_exps, S, Smax, rope_delta):
    return _original_layer_mxfp4(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_codes, k_exps, v_codes,
                                 k_exps, S, Smax, rope_delta)   # planted: V read with K's scales


_original_layer_mxfp4 = ea.expert_attention_layer_mxfp4

MXFP4_MUTATIONS = [
    (mx, "encode_e2m1_rne_sat", _encode_ties_away, mpins.test_ties_go_to_the_even_code),
    (mx, "block_exponent", _block_exponent_emax3, mpins.test_block_exponent_puts_amax_in_4_to_8),
    (mx, "e2m1_magnitudes", _magnitudes_bias2, mpins.test_e2m1_values_match_the_specification),
    (mx, "quantize_rows", _quantize_whole_row, mpins.test_quantize_rows_error_bound_and_block_layout),
    (ea, "expert_attention_layer_mxfp4", _layer_mxfp4_v_with_k_scales,
     mpins.test_attention_equals_bf16_oracle_on_representable_cache),
]


@pytest.mark.parametrize("mod,name,bad,pin", MXFP4_MUTATIONS,
                         ids=["ties_away", "emax3", "bias2", "row_scale", "v_with_k_scales"])
def test_mxfp4_pin_catches_planted_mistake(monkeypatch, mod, name, bad, pin):
    monkeypatch.setattr(mod, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        pin()


def test_unpatched_mxfp4_pins_pass():
    for _, _, _, pin in MXFP4_MUTATIONS:
        pin()


# ------------------------------------------------------------ FP8 own rows (quantise on write)
import oracle.fp8_e4m3 as f8  # noqa: E402
from tests import test_oracle_fp8_pins as fpins  # noqa: E402

_original_fp8_layer = ea.expert_attention_layer_fp8


def _tail_rows_per_token_amax(x):
    x = np.asarray(x, dtype=np.float32)
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty((x.shape[0],), dtype=np.float32)
    for g in range(x.shape[0]):
        sc_t = np.maximum(np.max(np.abs(x[g]), axis=-1), np.float32(1e-30)) / np.float32(448)
        codes[g] = f8.encode_e4m3_rne_sat(x[g] / sc_t[:, None])   # planted: one amax per token
        scales[g] = sc_t.max()
    return codes, scales


def _tail_rows_amax_over_all_heads(x):
    x = np.asarray(x, dtype=np.float32)
    sc = np.float32(np.max(np.abs(x)) / np.float32(448))           # planted: amax over all 8 heads
    return f8.encode_e4m3_rne_sat(x / sc), np.full((x.shape[0],), sc, dtype=np.float32)


def _fp8_layer_k_before_rope(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_codes, k_scales, v_codes,
                             v_scales, S, Smax, rope_delta):
    r = _original_fp8_layer(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_codes, k_scales, v_codes,
                            v_scales, S, Smax, rope_delta)
    kc, ks = f8.quantize_tail_rows(ea.rms_norm(k_raw, k_gamma).astype(np.float32))  # planted: no RoPE
    r["k_tail_codes"], r["k_tail_scale"] = kc, ks
    r["k_store"] = f8.decode_e4m3(kc) * ks.astype(np.float64)[:, None, None]
    r["out"] = ea.attention_concat(r["q"], f8.dequantize_cache(k_codes, k_scales, S),
                                   f8.dequantize_cache(v_codes, v_scales, S), S, r["k_store"], r["v_store"])
    return r


_FP8_CASE = fpins.CASES[0]
FP8_MUTATIONS = [
    (f8, "quantize_tail_rows", _tail_rows_per_token_amax, fpins.test_head_amax_encodes_to_448),
    (f8, "quantize_tail_rows", _tail_rows_amax_over_all_heads, fpins.test_own_row_scale_is_head_amax_over_448),
    (ea, "expert_attention_layer_fp8", _fp8_layer_k_before_rope,
     fpins.test_own_rows_within_half_ulp_of_roped_k_and_raw_v),
]


@pytest.mark.parametrize("mod,name,bad,pin", FP8_MUTATIONS,
                         ids=["per_token_amax", "amax_over_all_heads", "k_before_rope"])
def test_fp8_own_row_pin_catches_planted_mistake(monkeypatch, mod, name, bad, pin):
    monkeypatch.setattr(mod, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        pin(*_FP8_CASE)


def test_unpatched_fp8_own_row_pins_pass():
    for _, _, _, pin in FP8_MUTATIONS:
        pin(*_FP8_CASE)
