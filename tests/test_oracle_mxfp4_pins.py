"""Pins of the oracle's MXFP4 cache format (E2M1 codes, one power-of-two scale per 32 channels of
a row) and of the expert attention layer over an MXFP4 cache (CPU only).

Each test checks ``oracle.mxfp4`` against something other than itself: the specification's
published values (``tests/golden/mxfp4_constants.json``), a brute-force nearest-value search
with the tie rule spelled out, exact round trips, the scale rule's range property, the
rounding error bound per magnitude range, and, for the attention, the independently pinned
bf16 oracle on a cache of exactly representable values.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from gqa_attention_long_gb300.inputs import layer_inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_constants.json")))


def test_e2m1_values_match_the_specification():
    assert oracle.e2m1_magnitudes().tolist() == GOLD["e2m1_values"]["value"]
    assert oracle.MX_BLOCK == GOLD["block_size"]["value"]
    assert oracle.E2M1_MAX == max(GOLD["e2m1_values"]["value"])
    # the sign bit: code c + 8 is the negative of code c
    c = np.arange(8, dtype=np.uint8)
    assert np.array_equal(oracle.decode_e2m1(c + 8), -oracle.decode_e2m1(c))


def _bruteforce_code(x: float) -> int:
    """Nearest E2M1 value by exhaustive search over the published values; on a tie the code
    with mantissa bit 0 (an even code index) wins; the sign is the input's."""
    vals = GOLD["e2m1_values"]["value"]
    a = Fraction(abs(x))  # exact distances: no rounding can fake a tie at large magnitudes
    best = None
    for i, v in enumerate(vals):
        d = abs(a - Fraction(v))
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1] | (8 if math.copysign(1.0, x) < 0 else 0)


def test_encoder_matches_bruteforce_search():
    vals = GOLD["e2m1_values"]["value"]
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    xs = set(vals + mids + [6.5, 7.0, 7.99, 8.0, 100.0, 1e30, 1e-30, 0.1, 0.26, 0.24])
    for m in mids + vals:
        xs.update([np.nextafter(np.float32(m), np.float32(0)).item(),
                   np.nextafter(np.float32(m), np.float32(10)).item()])
    rng = np.random.default_rng(3)
    xs.update(rng.uniform(0, 9, 2000).astype(np.float32).tolist())
    xs = np.array(sorted(xs), dtype=np.float32)
    xs = np.concatenate([xs, -xs])
    got = oracle.encode_e2m1_rne_sat(xs)
    want = np.array([_bruteforce_code(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_ties_go_to_the_even_code():
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, v in ties.items():
        assert oracle.decode_e2m1(oracle.encode_e2m1_rne_sat(np.float32(x))) == v, x
        assert oracle.decode_e2m1(oracle.encode_e2m1_rne_sat(np.float32(-x))) == -v, x


def test_codes_round_trip_and_saturation():
    c = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.encode_e2m1_rne_sat(oracle.decode_e2m1(c).astype(np.float32)), c)
    big = np.array([6.0, 6.1, 7.5, 1e6, -6.2, -1e9], dtype=np.float32)
    assert oracle.decode_e2m1(oracle.encode_e2m1_rne_sat(big)).tolist() == [6, 6, 6, 6, -6, -6]


@pytest.mark.parametrize("amax,e", [(4.0, 0), (7.999, 0), (8.0, 1), (6.0, 0), (3.999, -1), (1.0, -2),
                                    (0.5, -3), (2.0 ** 20, 18), (0.0, 0), (2.0 ** -130, -127)])
def test_block_exponent_rule(amax, e):
    assert oracle.block_exponent(amax) == e


def test_block_exponent_puts_amax_in_4_to_8():
    rng = np.random.default_rng(4)
    amax = np.exp2(rng.uniform(-60, 60, 5000))
    for a in amax:
        e = oracle.block_exponent(a)
        assert 4.0 <= a / 2.0 ** e < 8.0
        assert e == math.floor(math.log2(a)) - GOLD["e2m1_emax"]["value"] or abs(math.log2(a) - round(math.log2(a))) < 1e-12


def _half_spacing(r):
    """Largest rounding error, in units of the block scale, at scaled magnitude r (< 8)."""
    return np.where(r < 2, 0.25, np.where(r < 4, 0.5, np.where(r < 6, 1.0, r - 6.0)))


def test_quantize_rows_error_bound_and_block_layout():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((8, 40, 128)) * np.exp2(rng.integers(-8, 8, (8, 40, 1)))).astype(np.float32)
    codes, exps = oracle.quantize_rows(x)
    assert codes.shape == x.shape and exps.shape == (8, 40, 4) and codes.max() < 16
    deq = oracle.dequantize_rows(codes, exps)
    scale = np.repeat(np.exp2(exps.astype(np.float64)), 32, axis=-1)
    r = np.abs(x) / scale
    assert np.all(r < 8)
    assert np.all(np.abs(deq - x) <= _half_spacing(r) * scale + 1e-30)
    # each 32-channel block has its own scale: scaling one block leaves the others' codes alone
    y = x.copy()
    y[:, :, 32:64] *= 1024
    c2, e2 = oracle.quantize_rows(y)
    assert np.array_equal(c2[..., :32], codes[..., :32]) and np.array_equal(c2[..., 64:], codes[..., 64:])
    assert np.array_equal(e2[..., 1], exps[..., 1] + 10) and np.array_equal(c2[..., 32:64], codes[..., 32:64])


def test_representable_values_survive_requantisation():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 16, (8, 16, 128)).astype(np.uint8)
    exps = rng.integers(-20, 20, (8, 16, 4)).astype(np.int16)
    v = oracle.dequantize_rows(codes, exps)
    c2, e2 = oracle.quantize_rows(v.astype(np.float32))
    assert np.array_equal(oracle.dequantize_rows(c2, e2), v)


def _mxfp4_cache(rng, Smax):
    codes = rng.integers(0, 16, (8, Smax, 128)).astype(np.uint8)
    exps = rng.integers(-3, 1, (8, Smax, 4)).astype(np.int16)
    return codes, exps


def test_attention_equals_bf16_oracle_on_representable_cache():
    # Own k and v rows of zero quantise exactly (to zero), and every dequantised cache value
    # (a code value times a power of two) is a bf16 value: the MXFP4 layer must then equal the
    # bf16 oracle run on the dequantised cache.
    S, Smax = 200, 512
    x = layer_inputs(31, S, Smax)
    rng = np.random.default_rng(7)
    kc, ke = _mxfp4_cache(rng, Smax)
    vc, ve = _mxfp4_cache(rng, Smax)
    f = lambda t: t.double().numpy()  # noqa: E731
    zk, zv = np.zeros((8, 64, 128)), np.zeros((8, 64, 128))
    got = oracle.expert_attention_layer_mxfp4(f(x.q_raw), zk, zv, f(x.q_gamma), f(x.k_gamma),
                                             kc, ke, vc, ve, S, Smax, 11)
    kd, vd = oracle.dequantize_rows(kc, ke), oracle.dequantize_rows(vc, ve)
    assert np.array_equal(oracle.bf16_round(kd), kd)
    ref = oracle.expert_attention_layer(f(x.q_raw), zk, zv, f(x.q_gamma), f(x.k_gamma), kd, vd, S, Smax, 11)
    assert np.max(np.abs(got["out"] - ref["out"])) < 1e-12
    assert not np.any(got["k_store"]) and not np.any(got["v_store"])


def test_attention_own_rows_quantised_within_bound():
    S, Smax = 64, 256
    x = layer_inputs(32, S, Smax)
    rng = np.random.default_rng(8)
    kc, ke = _mxfp4_cache(rng, Smax)
    vc, ve = _mxfp4_cache(rng, Smax)
    f = lambda t: t.double().numpy()  # noqa: E731
    got = oracle.expert_attention_layer_mxfp4(f(x.q_raw), f(x.k_raw), f(x.v_raw), f(x.q_gamma),
                                             f(x.k_gamma), kc, ke, vc, ve, S, Smax, 0)
    for store, src, e in ((got["k_store"], got["k"], got["k_tail_exps"]),
                          (got["v_store"], f(x.v_raw), got["v_tail_exps"])):
        src32 = src.astype(np.float32).astype(np.float64)
        scale = np.repeat(np.exp2(e.astype(np.float64)), 32, axis=-1)
        assert np.all(np.abs(store - src32) <= _half_spacing(np.abs(src32) / scale) * scale + 1e-30)
