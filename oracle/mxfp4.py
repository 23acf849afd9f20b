"""MXFP4 cache format: E2M1 codes with one power-of-two (E8M0) scale per 32 channels of a row
(test infrastructure only).

The pages' lowest-precision cache is Tenstorrent block-float (alpamayo_tt/EXPERT_NOTES.md,
"Known gaps" and "Timing"; the attention mask is bfp4 in decode mode), which has no GPU
counterpart. The 4-bit cache here follows the OCP Microscaling (MX) v1.0 format MXFP4, the
block-scaled 4-bit type the sm_103a tensor cores take. Readings taken (listed in the design
notes):

  * E2M1 element: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit, no infinities or
    NaN; magnitudes 0, 0.5 (the subnormal), 1, 1.5, 2, 3, 4, 6.
  * Encoding rounds to nearest, ties to the even code (mantissa bit 0), and saturates to +-6.
  * A block is 32 consecutive channels of one cache row (row r of kv head g, channels
    [32 j, 32 j + 32)), so every row, the own rows included, carries its own four scales and
    no row is ever requantised when another is written.
  * The block's scale is X = 2^e with e = floor(log2(amax)) - 2 (2 = the exponent of E2M1's
    largest normal, 6 = 1.5 * 2^2), clamped to the E8M0 range [-127, 127]; an all-zero block
    takes e = 0. An element v is encoded as encode(v / X); X is a power of two, so the
    division is exact. amax / X lies in [4, 8), so a block's largest magnitude encodes to 4 or
    6 (values in (6, 8) saturate to 6, which the format accepts).
  * Attention reads the dequantised values code_value * 2^e; the own 64 rows are quantised on
    write from the roped k (taken in fp32, as the cache writer holds it) and the raw v.
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
MX_BLOCK = 32
E8M0_MIN, E8M0_MAX = -127, 127


def e2m1_magnitudes() -> np.ndarray:
    """Values of the non-negative codes 0..7, in code order (ascending): code = (exp << 1) | man."""
    codes = np.arange(8)
    e = codes >> 1
    m = codes & 1
    sub = m * 0.5                                      # exponent field 0: m * 2^(1 - bias) / 2
    nor = (1.0 + m / 2.0) * np.exp2(e - 1.0)           # bias 1
    return np.where(e == 0, sub, nor).astype(np.float64)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """4-bit E2M1 codes (uint8 values 0..15, bit 3 = sign) -> float64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert np.all(codes < 16)
    val = e2m1_magnitudes()[(codes & 7).astype(np.int64)]
    return np.where(codes & 8, -val, val)


def encode_e2m1_rne_sat(x: np.ndarray) -> np.ndarray:
    """fp32 values -> E2M1 codes: round to nearest, ties to the even code, saturate at 6.

    The sign of the input is kept (negative values that round to zero give code 8). Inputs
    must be finite.
    """
    x = np.asarray(x, dtype=np.float32)
    assert np.all(np.isfinite(x)), "encoder input must be finite"
    a = np.abs(x).astype(np.float64)
    mags = e2m1_magnitudes()
    hi = np.minimum(np.searchsorted(mags, a, side="left"), 7)   # mags[hi-1] < a <= mags[hi]
    lo = np.maximum(hi - 1, 0)
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E2M1_MAX, 7, code)
    code = np.where(a == 0.0, 0, code)
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def block_exponent(amax: float) -> int:
    """e = floor(log2(amax)) - 2, clamped to [-127, 127]; 0 for amax = 0."""
    amax = float(amax)
    if amax == 0.0:
        return 0
    _, ex = np.frexp(amax)                             # amax = f * 2^ex with f in [0.5, 1)
    return int(min(max(int(ex) - 1 - 2, E8M0_MIN), E8M0_MAX))


def quantize_rows(x: np.ndarray):
    """Rows [..., 128] (fp32 values) -> (codes uint8 [..., 128] in 0..15, exps int16 [..., 4]).

    Block j of a row is channels [32 j, 32 j + 32), with scale 2^exps[..., j].
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] % MX_BLOCK == 0
    nb = x.shape[-1] // MX_BLOCK
    xb = x.reshape(*x.shape[:-1], nb, MX_BLOCK)
    amax = np.max(np.abs(xb), axis=-1)
    exps = np.vectorize(block_exponent, otypes=[np.int64])(amax).astype(np.int16)
    scale = np.exp2(exps.astype(np.float64)).astype(np.float32)   # exact: a power of two
    codes = encode_e2m1_rne_sat(xb / scale[..., None])
    return codes.reshape(x.shape), exps


def dequantize_rows(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """codes [..., 128] and exps [..., 4] -> float64 values code_value * 2^exp of the block."""
    codes = np.asarray(codes)
    nb = codes.shape[-1] // MX_BLOCK
    vals = decode_e2m1(codes).reshape(*codes.shape[:-1], nb, MX_BLOCK)
    return (vals * np.exp2(np.asarray(exps, dtype=np.float64))[..., None]).reshape(codes.shape)
