"""float64 CPU oracle of one whole action-expert decoder layer (test infrastructure only).

What it computes (alpamayo_tt/expert.py, ``TTExpert.layer``; shapes from
alpamayo_tt/EXPERT_NOTES.md, section "Matmul program configs", and ``TTExpert.__init__``,
where ``H, Q, I = tc.hidden, tc.q_dim, tc.inter``):

  * ``h = rms_norm(x, ln1)`` over the hidden channels of each of the 64 tokens;
  * ``qkv = h @ wqkv^T``: one fused projection whose output features are the q features
    (16 heads x 128), then k (8 x 128), then v (8 x 128) (``fused_qkv`` of q_proj, k_proj,
    v_proj); the features of head h are ``[128 h, 128 h + 128)`` of its block
    (``nlp_create_qkv_heads``);
  * the per-layer attention of :mod:`oracle.expert_attention` on those q, k, v (q/k norms,
    RoPE, own rows at the cache tail, masked GQA attention);
  * ``o``: the 16 heads' outputs side by side per token (``nlp_concat_heads``), then
    ``x1 = x + o @ wo^T``;
  * ``h2 = rms_norm(x1, ln2)``; ``m = (silu(h2 @ w1^T) * (h2 @ w3^T)) @ w2^T`` (SwiGLU: silu
    on the gate projection w1, times the up projection w3, then the down projection w2);
  * ``x2 = x1 + m``.

Readings where the pages leave a step open: a linear layer's weight is stored
``[out_features, in_features]`` and applied as ``y = x W^T`` (the checkpoint's convention;
the pages transpose it for their device layout); every RMSNorm of the layer uses the same
epsilon (``tc.rms_eps``, 1e-6); no intermediate bf16 rounding is modelled (the device path
keeps its activations in bf16, which the parity tolerance absorbs). The hidden and
intermediate widths are taken from the weight shapes, so that small instances can be checked
by hand; the model's are 1536 and 6144.

Everything is fp64; matrix products use numpy's matmul.
"""
from __future__ import annotations

import numpy as np

from .expert_attention import D, EPS, HKV, HQ, T, expert_attention_layer, rms_norm

HIDDEN = 1536              # tc.hidden of the expert
INTER = 6144               # tc.inter (SwiGLU width)
Q_DIM = HQ * D             # 2048
KV_DIM = HKV * D           # 1024
QKV_DIM = Q_DIM + 2 * KV_DIM  # 4096 output features of wqkv


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """``x @ w^T`` for a weight stored [out_features, in_features]."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU (swish): ``x * sigmoid(x) = x / (1 + exp(-x))``."""
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def split_qkv_heads(qkv: np.ndarray):
    """[64, 4096] fused projection -> q [16, 64, 128], k [8, 64, 128], v [8, 64, 128]:
    feature ``128 h + d`` of the q (k, v) block is channel d of head h."""
    q = qkv[:, :Q_DIM].reshape(T, HQ, D).transpose(1, 0, 2)
    k = qkv[:, Q_DIM:Q_DIM + KV_DIM].reshape(T, HKV, D).transpose(1, 0, 2)
    v = qkv[:, Q_DIM + KV_DIM:].reshape(T, HKV, D).transpose(1, 0, 2)
    return q, k, v


def concat_heads(a: np.ndarray) -> np.ndarray:
    """[16, 64, 128] per-head output -> [64, 2048]: token t's row holds head h at
    features ``[128 h, 128 h + 128)``."""
    return np.asarray(a, np.float64).transpose(1, 0, 2).reshape(T, HQ * D)


def swiglu_mlp(h2: np.ndarray, w1: np.ndarray, w3: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """``(silu(h2 @ w1^T) * (h2 @ w3^T)) @ w2^T``."""
    return linear(silu(linear(h2, w1)) * linear(h2, w3), w2)


def expert_layer(x, w: dict, k_cache, v_cache, S: int, Smax: int, rope_delta: int) -> dict:
    """One decoder layer with a bf16 cache.

    ``x`` [64, hidden]; ``w`` holds ``ln1`` [hidden], ``wqkv`` [4096, hidden], ``q_norm`` and
    ``k_norm`` [128], ``wo`` [hidden, 2048], ``ln2`` [hidden], ``w1`` and ``w3`` [inter, hidden],
    ``w2`` [hidden, inter]. Returns the fp64 intermediates ``h``, ``q_raw``, ``k_raw``, ``v_raw``,
    ``q_rope`` (the normed, roped q), ``attn`` [16, 64, 128], ``x1``, ``h2``, ``gu`` (silu(gate) *
    up) and the output ``x2``, plus the attention oracle's ``k_store``/``v_store`` (the own rows
    as written to the cache).
    """
    x = np.asarray(x, np.float64)
    assert x.shape[0] == T
    h = rms_norm(x, w["ln1"], EPS)
    q_raw, k_raw, v_raw = split_qkv_heads(linear(h, w["wqkv"]))
    r = expert_attention_layer(q_raw, k_raw, v_raw, w["q_norm"], w["k_norm"], k_cache, v_cache,
                               S, Smax, rope_delta)
    x1 = x + linear(concat_heads(r["out"]), w["wo"])
    h2 = rms_norm(x1, w["ln2"], EPS)
    gu = silu(linear(h2, w["w1"])) * linear(h2, w["w3"])
    x2 = x1 + linear(gu, w["w2"])
    return {"h": h, "q_raw": q_raw, "k_raw": k_raw, "v_raw": v_raw, "q_rope": r["q"],
            "attn": r["out"], "k_store": r["k_store"], "v_store": r["v_store"], "x1": x1, "h2": h2,
            "gu": gu, "x2": x2}
