"""Pins of the whole-layer oracle (CPU only): each checks the oracle against something other
than itself (library routines composed independently, closed forms, brute force on tiny
widths), chosen so that a swapped projection, a missing residual, a wrong head split or a
misplaced activation fails one of them."""
import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from gqa_attention_long_gb300.inputs import expert_layer_weights, layer_inputs, residual_stream

S_SMALL, SMAX_SMALL = 40, 128


def f64(t):
    return t.detach().to(torch.float64).numpy()


def small_case(seed, hidden=48, inter=40):
    """A layer with small hidden / intermediate widths (the attention dims are the model's)."""
    x = layer_inputs(seed, S_SMALL, SMAX_SMALL)
    w = expert_layer_weights(seed, hidden=hidden, inter=inter)
    wd = {k: f64(v) for k, v in w.__dict__.items()}
    xs = f64(residual_stream(seed, hidden=hidden))
    return x, wd, xs


def run(x, wd, xs, rope_delta=0):
    return oracle.expert_layer(xs, wd, f64(x.k_cache), f64(x.v_cache), x.S, x.Smax, rope_delta)


def test_model_widths():
    # alpamayo_tt/EXPERT_NOTES.md, "Matmul program configs": wqkv 1536 x 4096, wo 2048 x 1536,
    # w1 / w3 1536 x 6144, w2 6144 x 1536
    assert (oracle.HIDDEN, oracle.QKV_DIM, oracle.Q_DIM, oracle.INTER) == (1536, 4096, 2048, 6144)
    assert oracle.Q_DIM + 2 * oracle.KV_DIM == oracle.QKV_DIM


def test_matches_torch_composition():
    """The layer written with torch's fp64 library routines (rms_norm, linear, silu, view and
    permute for the head split and concat); the attention core is the separately pinned
    attention oracle."""
    x, wd, xs = small_case(3)
    r = run(x, wd, xs, rope_delta=5)
    t = {k: torch.from_numpy(v) for k, v in wd.items()}
    X = torch.from_numpy(xs)
    hid = X.shape[-1]
    h = F.rms_norm(X, (hid,), t["ln1"], eps=1e-6)
    qkv = F.linear(h, t["wqkv"])
    q = qkv[:, :2048].view(64, 16, 128).permute(1, 0, 2)
    k = qkv[:, 2048:3072].view(64, 8, 128).permute(1, 0, 2)
    v = qkv[:, 3072:].view(64, 8, 128).permute(1, 0, 2)
    a = oracle.expert_attention_layer(q.numpy(), k.numpy(), v.numpy(), wd["q_norm"], wd["k_norm"],
                                      f64(x.k_cache), f64(x.v_cache), x.S, x.Smax, 5)["out"]
    o = torch.from_numpy(a).permute(1, 0, 2).reshape(64, 2048)
    x1 = X + F.linear(o, t["wo"])
    h2 = F.rms_norm(x1, (hid,), t["ln2"], eps=1e-6)
    x2 = x1 + F.linear(F.silu(F.linear(h2, t["w1"])) * F.linear(h2, t["w3"]), t["w2"])
    assert np.max(np.abs(r["x1"] - x1.numpy())) < 1e-12
    assert np.max(np.abs(r["x2"] - x2.numpy())) < 1e-12
    assert np.max(np.abs(r["q_raw"] - q.numpy())) < 1e-12


def test_zero_output_projections_leave_the_residual_stream():
    x, wd, xs = small_case(4)
    wd["wo"] = np.zeros_like(wd["wo"])
    wd["w2"] = np.zeros_like(wd["w2"])
    r = run(x, wd, xs)
    assert np.array_equal(r["x1"], xs) and np.array_equal(r["x2"], xs)


def test_zero_gate_gives_zero_mlp():
    # silu(0) = 0, so a zero gate projection silences the MLP whatever w3 and w2 are
    x, wd, xs = small_case(5)
    wd["w1"] = np.zeros_like(wd["w1"])
    r = run(x, wd, xs)
    assert np.array_equal(r["x2"], r["x1"])


def test_head_split_selects_rows_of_wqkv():
    """Zeroing the wqkv rows [128 h, 128 h + 128) zeroes query head h: its output is then the
    plain mean of its group's live values (closed form), and the other heads are unchanged."""
    x, wd, xs = small_case(6)
    base = run(x, wd, xs)
    h = 5
    wd["wqkv"][128 * h:128 * (h + 1)] = 0.0
    r = run(x, wd, xs)
    g = h // 2
    vals = np.concatenate([f64(x.v_cache)[g, :x.S], r["v_store"][g]], 0)
    assert np.max(np.abs(r["attn"][h] - vals.mean(0)[None, :])) < 1e-12
    others = [j for j in range(16) if j != h]
    assert np.max(np.abs(r["attn"][others] - base["attn"][others])) < 1e-12


def test_kv_split_order():
    """k comes before v in the fused projection: zeroing the v rows (features 3072..4095)
    zeroes every own v row while leaving the roped keys unchanged."""
    x, wd, xs = small_case(7)
    base = run(x, wd, xs)
    wd["wqkv"][3072:] = 0.0
    r = run(x, wd, xs)
    assert np.array_equal(r["v_store"], np.zeros_like(r["v_store"]))
    assert np.array_equal(r["k_store"], base["k_store"])


def test_mlp_bruteforce_tiny():
    """SwiGLU on tiny widths with Python loops (hidden 6, intermediate 4)."""
    x, wd, xs = small_case(8, hidden=6, inter=4)
    r = run(x, wd, xs)
    h2, w1, w3, w2 = r["h2"], wd["w1"], wd["w3"], wd["w2"]
    for t in (0, 17, 63):
        gu = []
        for j in range(4):
            g = sum(w1[j, k] * h2[t, k] for k in range(6))
            u = sum(w3[j, k] * h2[t, k] for k in range(6))
            gu.append(g / (1.0 + math.exp(-g)) * u)
        for n in range(6):
            m = sum(w2[n, j] * gu[j] for j in range(4))
            assert abs(r["x1"][t, n] + m - r["x2"][t, n]) < 1e-12
        # h2 is the ln2-normed x1 row
        ms = sum(float(v) ** 2 for v in r["x1"][t]) / 6
        for n in range(6):
            assert abs(wd["ln2"][n] * r["x1"][t, n] / math.sqrt(ms + 1e-6) - h2[t, n]) < 1e-12
