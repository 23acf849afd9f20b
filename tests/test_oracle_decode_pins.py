"""Pins of the fp64 decode-attention oracle (the text model's single-token step; CPU only).

Each test checks ``oracle.text_decode_attention`` against something other than itself: torch's
fp64 scaled-dot-product attention with GQA on a torch-written RMSNorm and RoPE, closed forms
(one key; zero queries), brute force with Python loops on tiny inputs, and invariants the
step must have (rows after pos unread; KV head g feeds exactly query heads 8g..8g+7; the new
row is attended to). A plausible mistake (a wrong GQA map, an exclusive cur_pos, a dropped
rope_delta) fails one of them; ``tests/test_oracle_mutations.py`` plants those mistakes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_long_gb300.inputs import decode_inputs


def f64(t):
    return t.to(torch.float64).numpy()


def run(x, rope_delta=0):
    return oracle.text_decode_attention(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                                        f64(x.k_gamma), f64(x.k_cache), f64(x.v_cache), x.pos,
                                        rope_delta)


def _torch_norm_rope(x, gamma, position):
    """RMSNorm (eps inside the root, multiplicative gain) and HF rotate_half RoPE (theta 5e6),
    written with torch ops only."""
    x = x.to(torch.float64)
    y = x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + 1e-6) * gamma.to(torch.float64)
    inv = 5e6 ** (-torch.arange(0, 128, 2, dtype=torch.float64) / 128)
    ang = float(position) * inv
    cos, sin = torch.cat([ang.cos(), ang.cos()]), torch.cat([ang.sin(), ang.sin()])
    rot = torch.cat([-y[..., 64:], y[..., :64]], -1)
    return y * cos + rot * sin


@pytest.mark.parametrize("pos,delta", [(300, 0), (77, -20), (1, 9)])
def test_decode_matches_torch_sdpa_fp64(pos, delta):
    # Library routine: torch's fp64 SDPA with enable_gqa (query head h -> kv head h // 8) and
    # its default 1/sqrt(128) scale, on keys [cache rows 0..pos-1 ; the new row stored as bf16].
    x = decode_inputs(500 + pos, pos, 512)
    r = run(x, delta)
    q = _torch_norm_rope(x.q_raw, x.q_gamma, pos + delta)
    k = _torch_norm_rope(x.k_raw, x.k_gamma, pos + delta).to(torch.bfloat16).to(torch.float64)
    keys = torch.cat([x.k_cache[:, :pos].to(torch.float64), k[:, None]], 1)
    vals = torch.cat([x.v_cache[:, :pos].to(torch.float64), x.v_raw.to(torch.float64)[:, None]], 1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None], keys[None], vals[None], enable_gqa=True)[0, :, 0].numpy()
    assert np.max(np.abs(ref - r["out"])) < 1e-12
    assert np.max(np.abs(q.numpy() - r["q"])) < 1e-12
    assert np.array_equal(k.numpy(), r["k_store"])


def test_decode_position_zero_returns_the_new_value_row():
    # At pos = 0 the only key is the new row: every query head of group g returns v_raw[g].
    x = decode_inputs(601, 0, 128)
    out = run(x)["out"]
    v = f64(x.v_raw)
    for h in range(64):
        assert np.array_equal(out[h], v[h // 8])


@pytest.mark.parametrize("pos", [1, 40, 255])
def test_decode_zero_queries_give_mean_of_keys_rows(pos):
    # q = 0 gives equal scores, so every head returns the mean of V[g, 0..pos] (row pos = v_raw).
    x = decode_inputs(610 + pos, pos, 256)
    x.q_raw.zero_()
    out = run(x)["out"]
    vals = np.concatenate([f64(x.v_cache)[:, :pos], f64(x.v_raw)[:, None]], 1)
    for h in range(64):
        assert np.max(np.abs(out[h] - vals[h // 8].mean(0))) < 1e-13


@pytest.mark.parametrize("fill", ["garbage", "nan", "inf"])
def test_decode_rows_after_pos_do_not_matter(fill):
    a = run(decode_inputs(620, 100, 256, later_fill=7.0))["out"]
    b = run(decode_inputs(620, 100, 256, later_fill=fill))["out"]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("pos", [1, 2, 5])
def test_decode_bruteforce_tiny(pos):
    # The whole step with Python loops and the math module: norm, rotation, scores, softmax.
    x = decode_inputs(630 + pos, pos, 64)
    r = run(x, rope_delta=3)
    qr, kr, vr = f64(x.q_raw), f64(x.k_raw), f64(x.v_raw)
    qg, kg = f64(x.q_gamma), f64(x.k_gamma)
    kc, vc = f64(x.k_cache), f64(x.v_cache)
    p = pos + 3

    def norm_rope(row, gamma):
        rms = math.sqrt(sum(float(a) * float(a) for a in row) / 128 + 1e-6)
        y = [float(row[d]) / rms * float(gamma[d]) for d in range(128)]
        o = [0.0] * 128
        for j in range(64):
            a = p * (5e6 ** (-(2 * j) / 128))
            o[j] = y[j] * math.cos(a) - y[j + 64] * math.sin(a)
            o[j + 64] = y[j + 64] * math.cos(a) + y[j] * math.sin(a)
        return o

    for h in (0, 7, 8, 35, 63):
        g = h // 8
        q = norm_rope(qr[h], qg)
        knew = [float(v) for v in torch.tensor(norm_rope(kr[g], kg)).to(torch.bfloat16).double()]
        keys = [list(kc[g, j]) for j in range(pos)] + [knew]
        vals = [list(vc[g, j]) for j in range(pos)] + [list(vr[g])]
        s = [sum(a * float(b) for a, b in zip(q, kk)) / math.sqrt(128) for kk in keys]
        mx = max(s)
        w = [math.exp(si - mx) for si in s]
        tot = sum(w)
        o = [sum(w[j] * float(vals[j][d]) for j in range(len(w))) / tot for d in range(128)]
        assert np.max(np.abs(np.array(o) - r["out"][h])) < 1e-12


def test_decode_gqa_group_mapping():
    # Changing KV head g must change exactly query heads 8g .. 8g+7.
    x = decode_inputs(640, 60, 128)
    a = run(x)["out"]
    x.v_cache[3, :60] += 1.0
    b = run(x)["out"]
    changed = [h for h in range(64) if np.max(np.abs(a[h] - b[h])) > 1e-6]
    assert changed == list(range(24, 32))


def test_decode_attends_to_its_own_new_row():
    # A query equal to the new key (same raw row, same gain, same position) scores |k|^2/sqrt(128)
    # ~ 11 against it and ~N(0, 1) against the cache keys, so the new value row dominates.
    x = decode_inputs(650, 10, 64)
    x.q_gamma.copy_(x.k_gamma)
    for g in range(8):
        x.q_raw[8 * g:8 * g + 8] = x.k_raw[g]
    out = run(x)["out"]
    v = f64(x.v_raw)
    for h in range(64):
        assert np.max(np.abs(out[h] - v[h // 8])) < 2e-2


def test_decode_positions_are_pos_plus_delta():
    x = decode_inputs(660, 20, 64)
    a = oracle.decode_prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                               f64(x.k_gamma), 20, 5)
    b = oracle.decode_prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                               f64(x.k_gamma), 25, 0)
    c = oracle.decode_prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                               f64(x.k_gamma), 20, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.max(np.abs(a[0] - c[0])) > 1e-3
    # position 0 is the identity rotation: the roped rows are the normed rows
    z = oracle.decode_prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                               f64(x.k_gamma), 7, -7)
    n = f64(x.k_raw) * f64(x.k_gamma) / np.sqrt((f64(x.k_raw) ** 2).mean(-1, keepdims=True) + 1e-6)
    assert np.max(np.abs(z[1] - n)) < 1e-13


def test_stored_decode_samples_unchanged():
    # Written by tests/golden/make_golden.py, which calls only the oracle.
    path = os.path.join(os.path.dirname(__file__), "golden", "decode_samples.json")
    g = json.load(open(path))
    for case in g["cases"]:
        x = decode_inputs(case["seed"], case["pos"], case["Smax"])
        out = run(x, rope_delta=case["rope_delta"])["out"]
        idx = np.array(case["idx"])
        assert np.allclose(out[idx[:, 0], idx[:, 1]], np.array(case["val"]), rtol=0, atol=1e-12)
