"""The e4m3 attention's GPU parity bar against a model of the device's roundings (CPU only).

The GPU test of the e4m3 cache path (tests/test_gpu_fp8.py) compares the kernel with the fp64
oracle run on the same dequantised cache values, within max-abs 2e-2. The kernel differs from
that oracle in four places, which this test models on the CPU, in fp64 unless stated:

  * Q enters the e4m3 tensor-core product as a high and a low set of e4m3 codes with one scale
    per row, amax / 448: hi = e4m3(q / s), lo = e4m3(q / s - hi), both from the fp32 quotient;
  * P is stored as f16 relative to the unit's largest V scale, P = f16(2^(x - m) * sv / svr),
    while the row sum counts the unrounded 2^(x - m);
  * a unit split between two CTAs is merged from f16 partials, each half row scaled by a power
    of two into [2^14, 2^15) (11 significant bits: modelled as one f16 rounding of each part's
    normalised output, the units being cut in two here);
  * the output is rounded to bf16.

The modelled output must stay within half of the GPU bar, so that the bar keeps a margin for
what the model leaves out (fp32 accumulation, the exponential's approximation, the lazy
rescaling of the running maximum). At the main shape the model's error is ~3e-4 (outputs up to
~0.12 in magnitude; the bf16 rounding of the output is most of it), far inside the bar.
"""
import numpy as np

import oracle
from gqa_attention_long_gb300.inputs import config_seed, layer_inputs
from oracle.expert_attention import D, HKV, T, bf16_round, prologue
from oracle.fp8_e4m3 import decode_e4m3, dequantize_cache, encode_e4m3_rne_sat, quantize_tail_rows
from tests._gpu_util import f64

TOL_FP8_MAX_ABS = 2e-2  # the GPU test's bar


def q_hi_lo(q: np.ndarray) -> np.ndarray:
    """Rows of q [rows, 128] as the device feeds them to the tensor cores: (hi + lo) * s."""
    q32 = q.astype(np.float32)
    am = np.max(np.abs(q32), axis=-1, keepdims=True)
    s = np.where(am > 0, am * np.float32(1.0 / 448.0), np.float32(1.0)).astype(np.float32)
    inv = np.where(am > 0, np.float32(448.0) / am, np.float32(1.0)).astype(np.float32)
    a = (q32 * inv).astype(np.float32)
    hi = decode_e4m3(encode_e4m3_rne_sat(a))
    lo = decode_e4m3(encode_e4m3_rne_sat((a - hi.astype(np.float32)).astype(np.float32)))
    return (hi + lo) * s.astype(np.float64)


def device_unit(qg, keys, vals, vscale_per_key, svr, split_at):
    """One kv head's 128 folded rows against its keys: the device's P and partial roundings."""
    s = (qg @ keys.T) / np.sqrt(D)
    out_parts, lse_parts = [], []
    for lo_k, hi_k in ((0, split_at), (split_at, keys.shape[0])):
        sp = s[:, lo_k:hi_k]
        m = sp.max(axis=1, keepdims=True)
        p = np.exp(sp - m)
        L = p.sum(axis=1, keepdims=True)
        # P relative to the reference V scale, in f16; V as its code values (exact in f16)
        P = (p * (vscale_per_key[lo_k:hi_k] / svr)[None, :]).astype(np.float16).astype(np.float64)
        vcodes = vals[lo_k:hi_k] / vscale_per_key[lo_k:hi_k, None]
        o = (P @ vcodes) * svr / L
        out_parts.append(o.astype(np.float16).astype(np.float64))  # the f16 partial
        lse_parts.append(m + np.log(L))
    M = np.maximum(lse_parts[0], lse_parts[1])
    w0, w1 = np.exp(lse_parts[0] - M), np.exp(lse_parts[1] - M)
    return (w0 * out_parts[0] + w1 * out_parts[1]) / (w0 + w1)


def test_e4m3_rounding_model_within_half_the_gpu_bar():
    S, Smax = 4700, 8192  # the GPU test's main shape
    x = layer_inputs(config_seed(3, 0), S, Smax)
    kc, ks = oracle.quantize_cache_blocks(f64(x.k_cache), S, Smax)
    vc, vs = oracle.quantize_cache_blocks(f64(x.v_cache), S, Smax)
    ref = oracle.expert_attention_layer_fp8(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                                            f64(x.k_gamma), kc, ks, vc, vs, S, Smax, 0)["out"]
    q, k, v = prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma), f64(x.k_gamma), S, 0)
    ktc, kts = quantize_tail_rows(k.astype(np.float32))
    vtc, vts = quantize_tail_rows(v.astype(np.float32))
    k_deq, v_deq = dequantize_cache(kc, ks, S), dequantize_cache(vc, vs, S)
    n_main = (S + 127) // 128
    got = np.empty_like(ref)
    for g in range(HKV):
        keys = np.concatenate([k_deq[g], decode_e4m3(ktc[g]) * float(kts[g])])
        vals = np.concatenate([v_deq[g], decode_e4m3(vtc[g]) * float(vts[g])])
        vscale = np.concatenate([np.repeat(vs[g, :n_main].astype(np.float64), 128)[:S],
                                 np.full(T, float(vts[g]))])
        svr = float(max(vs[g, :n_main].max(), vts[g]))
        qg = q_hi_lo(np.concatenate([q[2 * g], q[2 * g + 1]]))  # folded rows: head 2g, then 2g+1
        o = device_unit(qg, keys, vals, vscale, svr, split_at=keys.shape[0] // 2)
        got[2 * g], got[2 * g + 1] = o[:T], o[T:]
    got = bf16_round(got)
    err = float(np.max(np.abs(got - ref)))
    assert err <= 0.5 * TOL_FP8_MAX_ABS, f"max-abs {err:.3e}"
    assert err > 1e-4  # the modelled roundings are there
