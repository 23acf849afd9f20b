"""float64 CPU oracle of one action-expert attention layer (test infrastructure only).

What it computes (alpamayo_tt/expert.py, ``TTExpert.layer`` and ``TTExpert.attention_core``;
alpamayo_tt/EXPERT_NOTES.md, sections "Layouts" and "Attention over the VLM cache: masking
approach"):

  * 64 expert tokens carry 16 query heads and 8 KV heads of width 128 (the GQA group of
    query head h is KV head h // 2);
  * q and k of every head and token are RMS-normalised over the head dimension with a
    multiplicative per-channel gain (eps 1e-6), then rotated with the HF rotate_half RoPE
    (theta 5e6) at position ``t + rope_delta + S`` for token t;
  * the roped k and the raw v of the 64 tokens are written into the last 64 rows
    ``[Smax-64, Smax)`` of the layer's KV cache;
  * every token attends, non-causally, to cache rows ``[0, S)`` and to those 64 tail rows;
    rows ``[S, Smax-64)`` are hidden by an additive -1e9 mask; the score scale is 1/sqrt(128).

Readings taken where the pages leave a step open (each one is also listed in the design
notes of the repository):

  * RoPE tables are the HF default ones: inverse frequencies ``theta**(-2j/128)``, j < 64,
    duplicated over both halves; ``rotate_half(x) = cat(-x[64:], x[:64])``.
  * RMSNorm is the Qwen3 form ``gamma * x / sqrt(mean(x**2) + eps)`` with eps inside the
    root and a multiplicative gain; no intermediate bf16 roundings are modelled.
  * The own keys are stored in the cache's dtype: for a bf16 cache the roped k is rounded
    to bf16 (round to nearest even); v is already bf16.
  * Masking by an additive -1e9 is the same as leaving the hidden keys out, because
    ``exp(-1e9 + s - max)`` is exactly 0 in fp64 for any finite score. The oracle computes
    both forms: :func:`attention_concat` (hidden rows excluded) and
    :func:`attention_tail_masked` (the pages' literal form over an Smax-row copy).

Everything is fp64. Inputs are numpy arrays (bf16 values are exactly representable).
"""
from __future__ import annotations

import math

import numpy as np

# Model constants as stated on the pages (alpamayo_tt/expert.py, ``TTExpert.__init__`` reads
# them from the expert's text config; alpamayo_tt/EXPERT_NOTES.md, section "Layouts").
HQ = 16          # query heads
HKV = 8          # key/value heads
REP = HQ // HKV  # query heads per KV head (GQA group size)
D = 128          # head dimension
T = 64           # expert tokens (waypoints)
EPS = 1e-6       # RMSNorm epsilon of q_norm / k_norm
THETA = 5e6      # RoPE base
MASK_MIN = -1e9  # additive mask value for hidden cache rows (expert.py, module constant)


# ----------------------------------------------------------------------------------- helpers
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits. ``frexp`` gives x = f * 2**e with 0.5 <= |f| < 1, so
    ``rint(f * 256)`` (numpy's rint rounds half to even) is the 8-bit significand. Values are
    far from the bf16 overflow and subnormal ranges in this path, which this helper does not
    treat specially.
    """
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)
    return np.ldexp(np.rint(f * 256.0), e - 8)


# ------------------------------------------------------------------------------ a1: RMSNorm
def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float = EPS) -> np.ndarray:
    """Per-row RMSNorm over the last axis: ``gamma * x / sqrt(mean(x**2) + eps)``.

    alpamayo_tt/expert.py, ``TTExpert.layer`` (``rms_norm`` of q and of k with the layer's
    q_norm / k_norm gains); alpamayo_tt/EXPERT_NOTES.md, section "Layouts" (per-head, eps 1e-6).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return np.asarray(gamma, dtype=np.float64) * x / np.sqrt(ms + eps)


# --------------------------------------------------------------------------------- a2: RoPE
def inv_freq(theta: float = THETA, dim: int = D) -> np.ndarray:
    """HF default inverse frequencies ``theta**(-2j/dim)`` for j in [0, dim/2)."""
    j = np.arange(dim // 2, dtype=np.float64)
    return theta ** (-2.0 * j / dim)


def rope_angles(pos: np.ndarray, theta: float = THETA, dim: int = D) -> np.ndarray:
    """Angles ``pos[t] * inv_freq[j]`` in fp64, shape [len(pos), dim/2]."""
    return np.outer(np.asarray(pos, dtype=np.float64), inv_freq(theta, dim))


def rope_rotate_half(x: np.ndarray, pos: np.ndarray, theta: float = THETA) -> np.ndarray:
    """HF rotate_half RoPE of x [..., n_tok, D] at integer positions pos [n_tok].

    alpamayo_tt/expert.py, ``TTExpert.layer`` (``rotary_embedding_hf`` of q and k) and
    ``TTExpert.set_context`` (cos/sin for positions ``i + rope_delta + S``);
    alpamayo_tt/EXPERT_NOTES.md, section "Layouts" (HF rotate_half tables, theta 5e6).

    out[d]      = x[d] cos(a_d) - x[d+64] sin(a_d)        for d < 64
    out[d + 64] = x[d+64] cos(a_d) + x[d] sin(a_d)
    """
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    a = rope_angles(pos, theta, x.shape[-1])           # [n_tok, half]
    cos = np.concatenate([np.cos(a), np.cos(a)], -1)   # [n_tok, D]
    sin = np.concatenate([np.sin(a), np.sin(a)], -1)
    rot = np.concatenate([-x[..., half:], x[..., :half]], -1)
    return x * cos + rot * sin


# ---------------------------------------------------------------------- a1 + a2 + a3 inputs
def prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, S: int, rope_delta: int):
    """Per-head norm and RoPE of the 64 expert tokens.

    Returns ``(q, k, v)`` in fp64: q [16, 64, 128] and k [8, 64, 128] normalised and roped at
    positions ``t + rope_delta + S``; v [8, 64, 128] unchanged (v is neither normalised nor
    roped in ``TTExpert.layer``).
    """
    pos = np.arange(T, dtype=np.int64) + int(rope_delta) + int(S)
    q = rope_rotate_half(rms_norm(q_raw, q_gamma), pos)
    k = rope_rotate_half(rms_norm(k_raw, k_gamma), pos)
    return q, k, np.asarray(v_raw, dtype=np.float64)


# ---------------------------------------------------------------------- a4..a8: attention
def _softmax_attend(q: np.ndarray, keys: np.ndarray, vals: np.ndarray, bias=None) -> np.ndarray:
    """softmax(q keys^T / sqrt(D) + bias) vals for one KV head; q [n, D], keys/vals [m, D]."""
    s = (q @ keys.T) / math.sqrt(D)
    if bias is not None:
        s = s + bias
    s = s - np.max(s, axis=-1, keepdims=True)
    p = np.exp(s)
    return (p @ vals) / np.sum(p, axis=-1, keepdims=True)


def attention_concat(q, k_cache, v_cache, S: int, k_own, v_own) -> np.ndarray:
    """Attention over the concatenation ``[cache rows 0..S ; own 64 rows]`` (hidden rows left out).

    q [16, 64, D]; k_cache/v_cache [8, >=S, D]; k_own/v_own [8, 64, D]. Query head h uses
    KV head h // 2. Returns out [16, 64, D] fp64.
    """
    out = np.empty((HQ, T, D), dtype=np.float64)
    for h in range(HQ):
        g = h // REP
        keys = np.concatenate([np.asarray(k_cache[g, :S], np.float64), k_own[g]], 0)
        vals = np.concatenate([np.asarray(v_cache[g, :S], np.float64), v_own[g]], 0)
        out[h] = _softmax_attend(q[h], keys, vals)
    return out


def attention_tail_masked(q, k_cache, v_cache, S: int, Smax: int, k_own, v_own) -> np.ndarray:
    """The pages' literal form: own rows written into cache rows [Smax-64, Smax), one
    attention over all Smax rows with an additive mask of 0 on [0, S) and [Smax-64, Smax)
    and -1e9 elsewhere (expert.py, ``TTExpert.build_mask`` / ``TTExpert.layer``)."""
    assert 0 <= S <= Smax - T
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    kc[:, Smax - T:] = k_own
    vc[:, Smax - T:] = v_own
    bias = np.full((Smax,), MASK_MIN, dtype=np.float64)
    bias[:S] = 0.0
    bias[Smax - T:] = 0.0
    out = np.empty((HQ, T, D), dtype=np.float64)
    for h in range(HQ):
        g = h // REP
        out[h] = _softmax_attend(q[h], kc[g], vc[g], bias)
    return out


def expert_attention_layer(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_cache, v_cache,
                           S: int, Smax: int, rope_delta: int, form: str = "concat") -> dict:
    """One layer with a bf16 cache. Returns a dict of fp64 arrays:

    ``q`` roped q [16,64,128]; ``k`` roped k [8,64,128]; ``k_store``/``v_store`` the own rows as
    stored in a bf16 cache (roped k rounded to bf16; v as given); ``out`` [16,64,128].
    ``form`` selects the concatenation form ("concat") or the masked tail form ("tail").
    """
    assert 0 <= S <= Smax - T and Smax % T == 0
    q, k, v = prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, S, rope_delta)
    k_store = bf16_round(k)
    v_store = v
    if form == "concat":
        out = attention_concat(q, k_cache, v_cache, S, k_store, v_store)
    elif form == "tail":
        out = attention_tail_masked(q, k_cache, v_cache, S, Smax, k_store, v_store)
    else:
        raise ValueError(form)
    return {"q": q, "k": k, "k_store": k_store, "v_store": v_store, "out": out}


def expert_attention_layer_fp8(q_raw, k_raw, v_raw, q_gamma, k_gamma,
                               k_codes, k_scales, v_codes, v_scales,
                               S: int, Smax: int, rope_delta: int) -> dict:
    """One layer with an e4m3 cache (codes [8, Smax, 128] uint8, scales [8, Smax/128 + 1] fp32).

    The own 64 rows are quantised on write with their own scale slot (column ``Smax/128``):
    k from the roped k (taken in fp32, the precision the cache writer holds it in), v from
    the raw bf16 v. Attention then runs in fp64 on the dequantised values
    ``code_value * block_scale`` of cache rows [0, S) and of the own rows.
    Returns ``q``, ``k``, ``k_tail_codes``, ``v_tail_codes``, ``k_tail_scale``, ``v_tail_scale``,
    ``k_store``/``v_store`` (dequantised own rows) and ``out``.
    """
    from .fp8_e4m3 import decode_e4m3, dequantize_cache, quantize_tail_rows

    assert 0 <= S <= Smax - T and Smax % 128 == 0
    q, k, v = prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, S, rope_delta)
    kc, ks = quantize_tail_rows(k.astype(np.float32))
    vc, vs = quantize_tail_rows(v.astype(np.float32))
    k_store = decode_e4m3(kc) * ks.astype(np.float64)[:, None, None]
    v_store = decode_e4m3(vc) * vs.astype(np.float64)[:, None, None]
    k_deq = dequantize_cache(k_codes, k_scales, S)
    v_deq = dequantize_cache(v_codes, v_scales, S)
    out = attention_concat(q, k_deq, v_deq, S, k_store, v_store)
    return {"q": q, "k": k, "k_tail_codes": kc, "v_tail_codes": vc, "k_tail_scale": ks,
            "v_tail_scale": vs, "k_store": k_store, "v_store": v_store, "out": out}


def expert_attention_layer_mxfp4(q_raw, k_raw, v_raw, q_gamma, k_gamma,
                                 k_codes, k_exps, v_codes, v_exps,
                                 S: int, Smax: int, rope_delta: int) -> dict:
    """One layer with an MXFP4 cache (E2M1 codes [8, Smax, 128] uint8 0..15, block exponents
    [8, Smax, 4]: row r's channels [32 j, 32 j + 32) scaled by 2^exps[g, r, j]).

    The own 64 rows are quantised on write like any row (each row has its own block scales):
    k from the roped k in fp32, v from the raw bf16 v. Attention then runs in fp64 on the
    dequantised values of cache rows [0, S) and of the own rows.
    Returns ``q``, ``k``, ``k_tail_codes``, ``k_tail_exps``, ``v_tail_codes``,
    ``v_tail_exps``, ``k_store``/``v_store`` (dequantised own rows) and ``out``.
    """
    from .mxfp4 import dequantize_rows, quantize_rows

    assert 0 <= S <= Smax - T and Smax % 128 == 0
    q, k, v = prologue(q_raw, k_raw, v_raw, q_gamma, k_gamma, S, rope_delta)
    kc, ke = quantize_rows(k.astype(np.float32))
    vc, ve = quantize_rows(v.astype(np.float32))
    k_store = dequantize_rows(kc, ke)
    v_store = dequantize_rows(vc, ve)
    k_deq = dequantize_rows(np.asarray(k_codes)[:, :S], np.asarray(k_exps)[:, :S])
    v_deq = dequantize_rows(np.asarray(v_codes)[:, :S], np.asarray(v_exps)[:, :S])
    out = attention_concat(q, k_deq, v_deq, S, k_store, v_store)
    return {"q": q, "k": k, "k_tail_codes": kc, "k_tail_exps": ke, "v_tail_codes": vc,
            "v_tail_exps": ve, "k_store": k_store, "v_store": v_store, "out": out}
