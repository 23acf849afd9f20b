"""Pins of the oracle's FP8 own-row quantiser (CPU only).

With an e4m3 cache the 64 own rows of a layer are quantised on write (alpamayo_tt/expert.py,
``TTExpert.layer``: the new k is normed and roped, cast to the cache dtype and written by
``fill_cache``; the raw v is cast and written likewise). The FP8 variant gives every KV head's
own rows one fp32 scale ``amax / 448`` over its 64 rows, in its own scale column (the reading
of the pages' block-float cache taken for a GPU, listed in the design notes).

These tests check ``oracle.expert_attention_layer_fp8`` and ``oracle.quantize_tail_rows``
against things other than themselves:

  * the roped k is recomputed independently, with torch's ``rms_norm`` and RoPE written as a
    multiplication by unit complex numbers (not the oracle's rotate_half form);
  * each head's scale is the closed form ``fp32(amax of that head's 64 rows) / 448``, the
    amax element encodes to the largest code 0x7E (448), and no element below the midpoint
    to the next code (432 x scale) does;
  * every stored value lies within half an e4m3 ulp (times the scale) of the roped k, and of
    the raw v, which is neither normed nor roped.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_attention_long_gb300.inputs import layer_inputs


def f64(t):
    return t.to(torch.float64).numpy()


def roped_k_independent(x, S, rope_delta):
    """rms_norm (torch) then RoPE as (k[d] + i k[d+64]) * exp(i pos theta^(-d/64)), fp64."""
    k = torch.nn.functional.rms_norm(x.k_raw.double(), (128,), weight=x.k_gamma.double(), eps=1e-6)
    pos = torch.arange(64, dtype=torch.float64) + S + rope_delta
    inv = torch.tensor(5.0e6, dtype=torch.float64) ** (-torch.arange(64, dtype=torch.float64) / 64)
    rot = torch.polar(torch.ones(64, 64, dtype=torch.float64), pos[:, None] * inv[None, :])
    z = torch.complex(k[..., :64], k[..., 64:]) * rot
    return torch.cat([z.real, z.imag], -1).numpy()


def half_ulp_bound(x32, scale):
    """Half an e4m3 ulp of x / scale, times scale: ulp(y) = 2^(floor(log2 y) - 3) for normal
    codes (y >= 2^-6) and 2^-9 for subnormal ones."""
    y = np.abs(x32.astype(np.float64)) / scale
    e = np.maximum(np.floor(np.log2(np.maximum(y, 1e-30))), -6)
    return 0.5 * np.exp2(e - 3) * scale * (1 + 1e-6)


def fp8_layer(seed, S, Smax, rope_delta):
    x = layer_inputs(seed, S, Smax)
    kq, ks = oracle.quantize_cache_blocks(f64(x.k_cache), S, Smax)
    vq, vs = oracle.quantize_cache_blocks(f64(x.v_cache), S, Smax)
    r = oracle.expert_attention_layer_fp8(
        f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma), f64(x.k_gamma),
        kq, ks, vq, vs, S, Smax, rope_delta)
    return x, r


CASES = [(201, 300, 512, 0), (202, 0, 256, 17), (203, 1000, 1280, -37)]


@pytest.mark.parametrize("seed,S,Smax,rope_delta", CASES)
def test_own_row_scale_is_head_amax_over_448(seed, S, Smax, rope_delta):
    x, r = fp8_layer(seed, S, Smax, rope_delta)
    k32 = roped_k_independent(x, S, rope_delta).astype(np.float32)
    v32 = x.v_raw.float().numpy()
    for g in range(8):
        for src, got in ((k32, r["k_tail_scale"][g]), (v32, r["v_tail_scale"][g])):
            want = np.float32(np.float32(np.max(np.abs(src[g]))) / np.float32(448.0))
            # the fp64 -> fp32 rounding of the independently roped k may differ from the
            # oracle's in the last bit of a value; allow that one fp32 step of the amax
            assert abs(float(got) - float(want)) <= float(np.spacing(want)), (g, got, want)


@pytest.mark.parametrize("seed,S,Smax,rope_delta", CASES)
def test_head_amax_encodes_to_448(seed, S, Smax, rope_delta):
    # The amax element of a head is x = 448 * scale and gets the largest code 0x7E; the next
    # code down is 416, so an element gets 0x7E exactly when |x| / scale is above the midpoint
    # 432 (at 432 itself the tie goes to 0x7E, the even code).
    x, r = fp8_layer(seed, S, Smax, rope_delta)
    k32 = roped_k_independent(x, S, rope_delta).astype(np.float32)
    v32 = x.v_raw.float().numpy()
    for src, codes in ((k32, r["k_tail_codes"]), (v32, r["v_tail_codes"])):
        for g in range(8):
            a = np.abs(src[g]).astype(np.float64)
            y = a / a.max() * 448.0
            is448 = (codes[g] & 0x7F) == 0x7E
            assert np.all(is448[a == a.max()]), g
            assert not np.any(is448[y < 432.0 * (1 - 1e-6)]), g
            assert np.all(is448[y > 432.0 * (1 + 1e-6)]), g
            # sign kept
            assert np.all((codes[g][is448] & 0x80 != 0) == (src[g][is448] < 0))


@pytest.mark.parametrize("seed,S,Smax,rope_delta", CASES)
def test_own_rows_within_half_ulp_of_roped_k_and_raw_v(seed, S, Smax, rope_delta):
    x, r = fp8_layer(seed, S, Smax, rope_delta)
    k32 = roped_k_independent(x, S, rope_delta).astype(np.float32)
    v32 = x.v_raw.float().numpy()
    for src, store, sc in ((k32, r["k_store"], r["k_tail_scale"]), (v32, r["v_store"], r["v_tail_scale"])):
        scale = sc.astype(np.float64)[:, None, None]
        err = np.abs(store - src.astype(np.float64))
        # one fp32 step of slack for the independently roped k (see above)
        slack = np.abs(src.astype(np.float64)) * 2.0 ** -23
        assert np.all(err <= half_ulp_bound(src, scale) + slack)
    # the stored own rows are what the attention uses: its output equals torch's fp64 SDPA
    # over [dequantised cache rows 0..S ; stored own rows]
    kq, ks = oracle.quantize_cache_blocks(f64(x.k_cache), S, Smax)
    vq, vs = oracle.quantize_cache_blocks(f64(x.v_cache), S, Smax)
    keys = np.concatenate([oracle.dequantize_cache(kq, ks, S), r["k_store"]], 1)
    vals = np.concatenate([oracle.dequantize_cache(vq, vs, S), r["v_store"]], 1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(r["q"])[None], torch.from_numpy(keys)[None], torch.from_numpy(vals)[None],
        enable_gqa=True)[0].numpy()
    assert np.max(np.abs(ref - r["out"])) < 1e-12
