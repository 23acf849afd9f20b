"""float64 CPU oracle of the text model's single-token decode attention (test infrastructure only).

What it computes (alpamayo_tt/text.py, ``TTText._layer_decode`` and
``TTText._decode_inputs_host``): one decode step of the Qwen3-VL text model for the token at
cache position ``pos``, per layer,

  * 64 query heads and 8 KV heads of width 128; query head h reads KV head h // 8 (HF
    ``repeat_kv`` with 8 query heads per KV head);
  * q and k of every head are RMS-normalised over the head dimension with the layer's q_norm /
    k_norm gains (eps 1e-6) and rotated with the HF rotate_half RoPE at position
    ``pos + rope_delta`` (``text_cos_sin(pos + rope_delta)``);
  * ``paged_update_cache`` writes the roped k and the raw v into row ``pos`` of the layer's K
    and V caches;
  * ``scaled_dot_product_attention_decode(..., cur_pos_tensor=pos, scale=1/sqrt(128))``: the
    token attends to cache rows ``[0, pos]``, its own new row included.

Readings taken where the pages leave a step open (each one is also listed in the design notes
of the repository):

  * ``cur_pos`` is inclusive: the keys are rows 0 .. pos (pos + 1 keys), as a causal decode
    step that has just written its own row at pos must see it.
  * The text model's cos/sin come from its multimodal RoPE with all three position ids equal
    to ``pos + rope_delta``; with equal ids the interleaved sections collapse to the plain 1-D
    rotate_half RoPE, taken here with theta 5e6 and the same HF tables as the expert's.
  * The own k row is stored in the cache's dtype: for a bf16 cache the roped k is rounded to
    bf16 (round to nearest even); v is already bf16.

Everything is fp64. Inputs are numpy arrays (bf16 values are exactly representable).
"""
from __future__ import annotations

import math

import numpy as np

from .expert_attention import D, bf16_round, rms_norm, rope_rotate_half

# Text model shapes as they appear on the pages (alpamayo_tt/text.py, ``TTText._layer_decode``:
# the head concat is [32, 8192] = 64 heads x 128; the KV cache interface is [1, 8, Smax, 128]).
HQ_TEXT = 64              # query heads of the text model
HKV_TEXT = 8              # key/value heads
REP_TEXT = HQ_TEXT // HKV_TEXT  # query heads per KV head


def decode_prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, pos: int, rope_delta: int):
    """Norm and RoPE of the decode token's heads at position ``pos + rope_delta``.

    q_raw [64, 128], k_raw/v_raw [8, 128]. Returns (q [64,128], k [8,128], v [8,128]) in fp64;
    v is neither normalised nor roped.
    """
    p = np.array([int(pos) + int(rope_delta)], dtype=np.int64)
    q = rope_rotate_half(rms_norm(np.asarray(q_raw, np.float64)[:, None, :], q_gamma), p)[:, 0]
    k = rope_rotate_half(rms_norm(np.asarray(k_raw, np.float64)[:, None, :], k_gamma), p)[:, 0]
    return q, k, np.asarray(v_raw, dtype=np.float64)


def decode_attend(q: np.ndarray, k_cache, v_cache, pos: int) -> np.ndarray:
    """softmax(q K[g, 0..pos]^T / sqrt(128)) V[g, 0..pos] for every query head h (g = h // 8).

    q [64, 128]; k_cache/v_cache [8, >pos, 128], row pos already holding the new token.
    Returns out [64, 128] fp64.
    """
    out = np.empty((HQ_TEXT, D), dtype=np.float64)
    for h in range(HQ_TEXT):
        g = h // REP_TEXT
        keys = np.asarray(k_cache[g, :pos + 1], np.float64)
        vals = np.asarray(v_cache[g, :pos + 1], np.float64)
        s = (keys @ q[h]) / math.sqrt(D)
        w = np.exp(s - np.max(s))
        out[h] = (w @ vals) / np.sum(w)
    return out


def text_decode_attention(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_cache, v_cache,
                          pos: int, rope_delta: int) -> dict:
    """One layer of the decode step with a bf16 cache [8, Smax, 128].

    Returns a dict of fp64 arrays: ``q`` [64,128] and ``k`` [8,128] normed and roped;
    ``k_store``/``v_store`` [8,128] the new rows as stored in a bf16 cache; ``out`` [64,128].
    The caller's cache arrays are not modified (the attention runs on a copy whose row pos
    holds the stored rows).
    """
    Smax = np.asarray(k_cache).shape[1]
    assert 0 <= pos < Smax
    q, k, v = decode_prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, pos, rope_delta)
    k_store = bf16_round(k)
    v_store = v
    kc = np.array(np.asarray(k_cache)[:, :pos + 1], dtype=np.float64, copy=True)
    vc = np.array(np.asarray(v_cache)[:, :pos + 1], dtype=np.float64, copy=True)
    kc[:, pos] = k_store
    vc[:, pos] = v_store
    out = decode_attend(q, kc, vc, pos)
    return {"q": q, "k": k, "k_store": k_store, "v_store": v_store, "out": out}
