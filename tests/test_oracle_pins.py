"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a closed form, an
invariant the method must have, brute force on tiny inputs, an independent formulation
(complex-number RoPE), or a library routine (torch's fp64 scaled-dot-product attention,
torch's bf16 and e4m3 casts). A plausible mistake in the oracle (a dropped term, a wrong
sign or index, a transposed operand, a wrong GQA map or position offset) fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_long_gb300.inputs import layer_inputs, zero_inputs_like

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(t):
    return t.to(torch.float64).numpy()


def run(x, S, Smax, rope_delta=0, form="concat"):
    return oracle.expert_attention_layer(
        f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma), f64(x.k_gamma),
        f64(x.k_cache), f64(x.v_cache), S, Smax, rope_delta, form=form)


# ------------------------------------------------------------------------------ constants
def test_constants_match_pages():
    c = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    assert oracle.HQ == c["n_heads"]["value"]
    assert oracle.HKV == c["n_kv_heads"]["value"]
    assert oracle.D == c["head_dim"]["value"]
    assert oracle.T == c["n_tokens"]["value"] == c["tail_rows"]["value"]
    assert oracle.EPS == c["rms_eps"]["value"]
    assert oracle.THETA == c["rope_theta"]["value"]
    assert oracle.MASK_MIN == c["mask_min"]["value"]
    assert oracle.REP * oracle.T == c["gqa_fold_rows"]["value"]


# ---------------------------------------------------------------------------- bf16 rounding
def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e3,
                        rng.standard_normal(2000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_ties_to_even():
    # 1 + 2**-8 lies halfway between bf16 neighbours 1 and 1 + 2**-7: ties go to the even one (1).
    assert oracle.bf16_round(np.array([1 + 2 ** -8]))[0] == 1.0
    # 1 + 3 * 2**-8 lies halfway between 1 + 2**-7 (odd) and 1 + 2**-6 (even).
    assert oracle.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    # just above the tie rounds up
    assert oracle.bf16_round(np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 1 + 2 ** -7


# ---------------------------------------------------------------------------------- RMSNorm
def test_rms_norm_closed_form_example():
    x = np.zeros((1, 128))
    x[0, 0], x[0, 1] = 3.0, 4.0
    y = oracle.rms_norm(x, np.ones(128), eps=1e-6)
    expect = np.array([3.0, 4.0]) / math.sqrt(25.0 / 128 + 1e-6)
    assert np.allclose(y[0, :2], expect, rtol=0, atol=1e-14)
    assert np.all(y[0, 2:] == 0)


def test_rms_norm_eps_inside_the_root():
    # With gain 1, rms(y) = sqrt(m / (m + eps)), m = mean(x^2); tiny x makes eps visible.
    rng = np.random.default_rng(2)
    for scale in (1.0, 1e-3, 3e-4):
        x = rng.standard_normal((5, 128)) * scale
        y = oracle.rms_norm(x, np.ones(128))
        m = np.mean(x * x, -1)
        assert np.allclose(np.sqrt(np.mean(y * y, -1)), np.sqrt(m / (m + 1e-6)), rtol=1e-13)


def test_rms_norm_gain_is_multiplicative_and_scale_invariant():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 128))
    gam = 1 + 0.1 * rng.standard_normal(128)
    y1 = oracle.rms_norm(x, gam)
    assert np.allclose(y1, gam * oracle.rms_norm(x, np.ones(128)), rtol=1e-14)
    assert np.allclose(oracle.rms_norm(5.0 * x, gam), y1, rtol=1e-6)  # only eps breaks exactness


# ------------------------------------------------------------------------------------- RoPE
def test_inv_freq_closed_forms():
    f = oracle.inv_freq()
    assert f.shape == (64,) and f[0] == 1.0
    assert math.isclose(f[32], 1 / math.sqrt(5e6), rel_tol=1e-14)
    assert np.allclose(f[1:] / f[:-1], 5e6 ** (-1 / 64), rtol=1e-13)


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64, 128))
    y = oracle.rope_rotate_half(x, np.zeros(64, dtype=np.int64))
    assert np.array_equal(y, x)


def test_rope_matches_complex_rotation():
    # rotate_half RoPE == multiply z_j = x_j + i x_{j+64} by exp(i * pos * inv_freq_j).
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 64, 128))
    pos = np.arange(64) + 4700
    z = x[..., :64] + 1j * x[..., 64:]
    zr = z * np.exp(1j * np.outer(pos, 5e6 ** (-np.arange(64) / 64.0)))
    y = oracle.rope_rotate_half(x, pos)
    assert np.allclose(y[..., :64], zr.real, atol=1e-12)
    assert np.allclose(y[..., 64:], zr.imag, atol=1e-12)


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((64, 128))
    k = rng.standard_normal((64, 128))
    pa, pb = np.arange(64) + 17, np.arange(64) + 3000
    rq = oracle.rope_rotate_half(q, pa)
    pair = lambda v: v[:, :64] ** 2 + v[:, 64:] ** 2  # noqa: E731
    assert np.allclose(pair(rq), pair(q), rtol=1e-12)
    # <rope(q, a), rope(k, b)> depends on a - b only
    d1 = np.sum(oracle.rope_rotate_half(q, pa) * oracle.rope_rotate_half(k, pb), -1)
    d2 = np.sum(oracle.rope_rotate_half(q, pa + 999) * oracle.rope_rotate_half(k, pb + 999), -1)
    assert np.allclose(d1, d2, atol=1e-9)


def test_prologue_positions_are_t_plus_delta_plus_S():
    # Equal raw rows for all tokens: token t at context S equals token t-1 at context S+1,
    # and (S, delta) enter only through their sum.
    rng = np.random.default_rng(7)
    row = rng.standard_normal(128)
    q_raw = np.broadcast_to(row, (16, 64, 128)).copy()
    k_raw = np.broadcast_to(row, (8, 64, 128)).copy()
    v_raw = rng.standard_normal((8, 64, 128))
    gq, gk = np.ones(128), np.ones(128)
    qa, ka, _ = oracle.prologue(q_raw, k_raw, v_raw, gq, gk, S=10, rope_delta=5)
    qb, kb, _ = oracle.prologue(q_raw, k_raw, v_raw, gq, gk, S=11, rope_delta=5)
    qc, _, _ = oracle.prologue(q_raw, k_raw, v_raw, gq, gk, S=0, rope_delta=15)
    assert np.allclose(qa[:, 1:], qb[:, :-1], atol=1e-12)
    assert np.allclose(ka[:, 1:], kb[:, :-1], atol=1e-12)
    assert np.allclose(qa, qc, atol=0)
    q0, _, v0 = oracle.prologue(q_raw, k_raw, v_raw, gq, gk, S=0, rope_delta=0)
    assert np.allclose(q0[0, 0], oracle.rms_norm(row[None], gq)[0], atol=0)  # position 0 unrotated
    assert np.array_equal(v0, v_raw)


# ------------------------------------------------------------------------------ attention
@pytest.mark.parametrize("S", [0, 1, 5, 100, 192])
def test_tail_placement_equals_concatenation(S):
    x = layer_inputs(seed=11 + S, S=S, Smax=256)
    a = run(x, S, 256, form="concat")["out"]
    b = run(x, S, 256, form="tail")["out"]
    assert np.max(np.abs(a - b)) < 1e-12


def test_hidden_rows_do_not_matter():
    S, Smax = 70, 256
    base = run(layer_inputs(21, S, Smax, hidden_fill=7.0), S, Smax, form="tail")["out"]
    garb = run(layer_inputs(21, S, Smax, hidden_fill="garbage"), S, Smax, form="tail")["out"]
    assert np.array_equal(base, garb)
    nan = run(layer_inputs(21, S, Smax, hidden_fill="nan"), S, Smax, form="concat")["out"]
    assert np.max(np.abs(nan - base)) < 1e-12


@pytest.mark.parametrize("S", [0, 3, 130])
def test_zero_queries_give_mean_of_live_values(S):
    Smax = 256
    x = zero_inputs_like(layer_inputs(31, S, Smax), q_raw=True)
    out = run(x, S, Smax)["out"]
    vc, vr = f64(x.v_cache), f64(x.v_raw)
    for h in range(16):
        live = np.concatenate([vc[h // 2, :S], vr[h // 2]], 0)
        assert np.allclose(out[h], np.broadcast_to(live.mean(0), (64, 128)), atol=1e-13)


def test_identical_keys_give_mean_of_live_values():
    S, Smax = 77, 256
    x = layer_inputs(41, S, Smax)
    x.k_cache.zero_()
    x = zero_inputs_like(x, k_raw=True)
    out = run(x, S, Smax)["out"]
    vc, vr = f64(x.v_cache), f64(x.v_raw)
    for g in range(8):
        mean = np.concatenate([vc[g, :S], vr[g]], 0).mean(0)
        assert np.allclose(out[2 * g:2 * g + 2], np.broadcast_to(mean, (2, 64, 128)), atol=1e-13)


def test_rope_delta_irrelevant_without_cache():
    # With S = 0 every key and query is shifted by the same rope_delta, so the exact (fp64,
    # unrounded) keys give the same output; the bf16 store of the own keys is left out here
    # because its rounding depends on the rotation.
    x = layer_inputs(51, 0, 128)
    outs = []
    for delta in (0, 1234, -50):
        q, k, v = oracle.prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                                  f64(x.k_gamma), 0, delta)
        outs.append(oracle.attention_concat(q, f64(x.k_cache), f64(x.v_cache), 0, k, v))
    assert np.max(np.abs(outs[0] - outs[1])) < 1e-10
    assert np.max(np.abs(outs[0] - outs[2])) < 1e-10


def test_matches_torch_sdpa_fp64():
    # Library routine: torch's fp64 SDPA with GQA (q head h -> kv head h // 2) and its default
    # 1/sqrt(head_dim) scale, on the oracle's roped q and stored own rows.
    S, Smax = 300, 512
    x = layer_inputs(61, S, Smax)
    r = run(x, S, Smax)
    keys = np.concatenate([f64(x.k_cache)[:, :S], r["k_store"]], 1)
    vals = np.concatenate([f64(x.v_cache)[:, :S], r["v_store"]], 1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(r["q"])[None], torch.from_numpy(keys)[None], torch.from_numpy(vals)[None],
        enable_gqa=True)[0].numpy()
    assert np.max(np.abs(ref - r["out"])) < 1e-12


@pytest.mark.parametrize("S", [0, 1, 2])
def test_bruteforce_tiny(S):
    Smax = 128
    x = layer_inputs(71 + S, S, Smax)
    r = run(x, S, Smax)
    kc, vc = f64(x.k_cache), f64(x.v_cache)
    for h, t in [(0, 0), (1, 63), (6, 17), (15, 40)]:
        g = h // 2
        keys = [kc[g, j] for j in range(S)] + [r["k_store"][g, j] for j in range(64)]
        vals = [vc[g, j] for j in range(S)] + [r["v_store"][g, j] for j in range(64)]
        s = [sum(float(a) * float(b) for a, b in zip(r["q"][h, t], kk)) / math.sqrt(128) for kk in keys]
        mx = max(s)
        w = [math.exp(si - mx) for si in s]
        tot = sum(w)
        o = [sum(w[j] * float(vals[j][d]) for j in range(len(w))) / tot for d in range(128)]
        assert np.max(np.abs(np.array(o) - r["out"][h, t])) < 1e-12


def test_one_dominant_key_selects_its_value_row():
    S, Smax = 40, 128
    x = layer_inputs(81, S, Smax)
    q = run(x, S, Smax)["q"]
    h, t, j = 5, 9, 13
    qv = q[h, t]
    # a cache key along q with a score of ~400 dominates every other key by far
    x.k_cache[h // 2, j] = torch.from_numpy(400.0 * math.sqrt(128) * qv / np.dot(qv, qv)).to(torch.bfloat16)
    out = run(x, S, Smax)["out"]
    assert np.max(np.abs(out[h, t] - f64(x.v_cache)[h // 2, j])) < 1e-9


def test_gqa_group_mapping():
    # Changing KV head g must change exactly query heads 2g and 2g+1.
    S, Smax = 50, 128
    x = layer_inputs(91, S, Smax)
    a = run(x, S, Smax)["out"]
    x.v_cache[3, :S] += 1.0
    b = run(x, S, Smax)["out"]
    changed = [h for h in range(16) if np.max(np.abs(a[h] - b[h])) > 1e-6]
    assert changed == [6, 7]


# ------------------------------------------------------------------------------------ FP8
def test_e4m3_table_closed_values():
    m = oracle.e4m3_magnitudes()
    assert m.shape == (127,) and np.all(np.diff(m) > 0)
    assert m[0x00] == 0 and m[0x01] == 2.0 ** -9 and m[0x07] == 7 * 2.0 ** -9
    assert m[0x08] == 2.0 ** -6 and m[0x38] == 1.0 and m[0x3C] == 1.5 and m[0x7E] == 448.0
    v = oracle.decode_e4m3(np.array([0x7F, 0xFF, 0xB8, 0x80], dtype=np.uint8))
    assert np.isnan(v[0]) and np.isnan(v[1]) and v[2] == -1.0 and v[3] == 0 and np.signbit(v[3])


def test_e4m3_encoder_matches_torch_below_saturation():
    rng = np.random.default_rng(12)
    m = oracle.e4m3_magnitudes()
    ties = (m[1:] + m[:-1]) / 2
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(5000) * 0.01,
                        ties, -ties, [0.0, -0.0, 463.9, -463.9]]).astype(np.float32)
    ours = oracle.encode_e4m3_rne_sat(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encoder_saturates():
    codes = oracle.encode_e4m3_rne_sat(np.array([464.0, 500.0, 1e30, -1e6], dtype=np.float32))
    assert codes.tolist() == [0x7E, 0x7E, 0x7E, 0xFE]


def test_block_quantiser_error_bound_and_amax():
    x = layer_inputs(101, 300, 512)
    kc = x.k_cache.float().numpy()
    codes, scales = oracle.quantize_cache_blocks(kc, 300, 512)
    assert np.all(np.isnan(scales[:, 3:]))          # blocks 3.. hold no quantised row; col 4 = own rows
    deq = oracle.dequantize_cache(codes, scales, 300)
    err = np.abs(deq - kc[:, :300])
    # half an e4m3 ulp of the scaled value: ulp(y) = 2**(floor(log2 y) - 3), >= 2**-9
    y = np.abs(kc[:, :300]) / scales[:, np.arange(300) // 128][:, :, None]
    ulp = np.exp2(np.maximum(np.floor(np.log2(np.maximum(y, 1e-30))), -6) - 3)
    bound = 0.5 * ulp * scales[:, np.arange(300) // 128][:, :, None] * (1 + 1e-6)
    assert np.all(err <= bound)
    for g in range(8):
        for b in range(3):
            blk = np.abs(kc[g, 128 * b:min(128 * b + 128, 300)])
            assert np.max(np.abs(oracle.decode_e4m3(codes[g, 128 * b:min(128 * b + 128, 300)]))) == 448.0
            assert scales[g, b] == np.float32(np.float32(blk.max()) / np.float32(448))


def test_fp8_layer_reduces_to_bf16_layer_on_exact_values():
    # A cache whose values are exact e4m3 codes times a power-of-two block scale dequantises
    # to itself; the fp8 layer then differs from the bf16 layer only through the own rows.
    S, Smax = 200, 384
    x = layer_inputs(111, S, Smax)
    rng = np.random.default_rng(0)
    m = oracle.e4m3_magnitudes()
    for c in (x.k_cache, x.v_cache):
        codes = rng.integers(0, 127, size=c.shape)
        sign = np.where(rng.random(c.shape) < 0.5, -1.0, 1.0)
        c.copy_(torch.from_numpy(sign * m[codes] / 64.0).to(torch.bfloat16))
        c[:, :, 0] = 7.0  # fixes every block's amax at 7 = 448 / 64, so the scale is 1/64
    kq, ks = oracle.quantize_cache_blocks(f64(x.k_cache), S, Smax)
    vq, vs = oracle.quantize_cache_blocks(f64(x.v_cache), S, Smax)
    assert np.all(ks[:, :2] == np.float32(1 / 64))
    r8 = oracle.expert_attention_layer_fp8(
        f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma), f64(x.k_gamma),
        kq, ks, vq, vs, S, Smax, 0)
    assert np.array_equal(oracle.dequantize_cache(kq, ks, S), f64(x.k_cache)[:, :S])
    ref = oracle.attention_concat(r8["q"], f64(x.k_cache), f64(x.v_cache), S, r8["k_store"], r8["v_store"])
    assert np.max(np.abs(ref - r8["out"])) < 1e-13


# --------------------------------------------------------------------------- stored golden
def test_stored_oracle_samples_unchanged():
    # Written by tests/golden/make_golden.py, which calls only the oracle.
    g = json.load(open(os.path.join(GOLDEN, "oracle_samples.json")))
    for case in g["cases"]:
        x = layer_inputs(case["seed"], case["S"], case["Smax"])
        out = run(x, case["S"], case["Smax"], rope_delta=case["rope_delta"])["out"]
        idx = np.array(case["idx"])
        got = out[idx[:, 0], idx[:, 1], idx[:, 2]]
        assert np.allclose(got, np.array(case["val"]), rtol=0, atol=1e-12)
