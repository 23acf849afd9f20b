"""OCP E4M3 code table, encoder and block quantiser of the FP8 cache variant (test infrastructure only).

The pages store the cache either in bf16 or in Tenstorrent block-float8 (alpamayo_tt/expert.py,
``TTExpert.layer`` casts the new k/v to the cache dtype before writing them;
alpamayo_tt/EXPERT_NOTES.md, section "Timing" and "Known gaps" quote the bfp8 cache).
Block-float8 has no GPU counterpart, so the FP8 variant here uses OCP E4M3 ("e4m3fn") codes
with one fp32 scale per (kv head, 128-row block). Readings taken (listed in the design notes):

  * E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities; codes
    0x7F / 0xFF are NaN; largest finite magnitude 448; subnormals ``m * 2**-9``.
  * Encoding rounds to nearest, ties to the even code, and saturates to +-448 ("satfinite").
  * A block's scale is ``amax / 448`` in fp32 (1.0 when amax is 0), amax over the block's rows
    that are quantised; a value is encoded as ``encode(x / scale)`` with the division in fp32.
    These integer decisions are taken in fp32 on both sides so that codes can match exactly.
  * Cache rows [0, n_rows) are quantised in 128-row blocks; scale column b belongs to rows
    [128 b, 128 b + 128). The 64 own rows [Smax-64, Smax) share the last block with VLM rows,
    so they get their own scale slot, column ``Smax/128``; VLM rows are never requantised.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK_ROWS = 128


def e4m3_magnitudes() -> np.ndarray:
    """Values of the non-negative finite codes 0..126, in code order (which is ascending)."""
    codes = np.arange(127)
    e = (codes >> 3) & 0xF
    m = codes & 0x7
    sub = m.astype(np.float64) * 2.0 ** -9
    nor = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    return np.where(e == 0, sub, nor)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag_code = codes & 0x7F
    mags = np.append(e4m3_magnitudes(), np.nan)          # index 127 = NaN
    val = mags[mag_code.astype(np.int64)]
    return np.where(codes & 0x80, -val, val)


def encode_e4m3_rne_sat(x: np.ndarray) -> np.ndarray:
    """fp32 values -> uint8 E4M3 codes: round to nearest, ties to even code, saturate at 448.

    The sign bit of the input is kept (so -0.0 and negative values that round to zero give
    0x80). Inputs must be finite.
    """
    x = np.asarray(x, dtype=np.float32)
    assert np.all(np.isfinite(x)), "encoder input must be finite"
    a = np.abs(x).astype(np.float64)
    mags = e4m3_magnitudes()
    hi = np.searchsorted(mags, a, side="left")          # mags[hi-1] < a <= mags[hi]
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 126, code)            # satfinite
    code = np.where(a == 0.0, 0, code)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def _block_scale(amax: np.float32) -> np.float32:
    """``amax / 448`` in fp32, or 1 for an all-zero block."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(E4M3_MAX))


def quantize_cache_blocks(cache: np.ndarray, n_rows: int, Smax: int, fill_code: int = 0):
    """Quantise rows [0, n_rows) of a cache [8, Smax, 128] (bf16 values) in 128-row blocks.

    Returns ``codes`` uint8 [8, Smax, 128] (rows >= n_rows hold ``fill_code``) and ``scales``
    fp32 [8, Smax/128 + 1]: column b is the scale of rows [128 b, 128 b + 128) that lie
    below n_rows (NaN for blocks with no quantised row and for the own-row column).
    """
    assert Smax % BLOCK_ROWS == 0 and 0 <= n_rows <= Smax - 64
    H = cache.shape[0]
    nb = Smax // BLOCK_ROWS
    codes = np.full((H, Smax, cache.shape[2]), fill_code, dtype=np.uint8)
    scales = np.full((H, nb + 1), np.nan, dtype=np.float32)
    x32 = np.asarray(cache, dtype=np.float32)
    for g in range(H):
        for b in range(nb):
            r0, r1 = b * BLOCK_ROWS, min((b + 1) * BLOCK_ROWS, n_rows)
            if r0 >= r1:
                continue
            blk = x32[g, r0:r1]
            sc = _block_scale(np.max(np.abs(blk)))
            scales[g, b] = sc
            codes[g, r0:r1] = encode_e4m3_rne_sat(blk / sc)
    return codes, scales


def quantize_tail_rows(x: np.ndarray):
    """Quantise the 64 own rows of every kv head with one scale per head.

    x fp32 [8, 64, 128] -> (codes uint8 [8, 64, 128], scales fp32 [8]).
    """
    x = np.asarray(x, dtype=np.float32)
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty((x.shape[0],), dtype=np.float32)
    for g in range(x.shape[0]):
        sc = _block_scale(np.max(np.abs(x[g])))
        scales[g] = sc
        codes[g] = encode_e4m3_rne_sat(x[g] / sc)
    return codes, scales


def dequantize_cache(codes: np.ndarray, scales: np.ndarray, n_rows: int) -> np.ndarray:
    """Rows [0, n_rows) of an e4m3 cache as fp64 values ``code_value * scale[g, row // 128]``."""
    vals = decode_e4m3(np.asarray(codes)[:, :n_rows])
    blk = np.arange(n_rows) // BLOCK_ROWS
    sc = np.asarray(scales, dtype=np.float64)[:, blk]
    return vals * sc[:, :, None]
