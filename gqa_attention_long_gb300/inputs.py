"""Seeded synthetic inputs of the expert-attention workloads.

This module only draws random numbers and fills buffers; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can consume what it produces.

Shapes and distributions follow the pages' statement of the workload
(alpamayo_tt/EXPERT_NOTES.md, sections "Layouts" and "Attention over the VLM cache: masking
approach"): raw q [16, 64, 128], k and v [8, 64, 128], per-channel q_norm / k_norm gains [128],
and a per-layer VLM KV cache [8, Smax, 128] whose rows [0, S) are valid. The pages' real cache
comes from the VLM prefill of a driving prompt (about 4.6K prompt tokens plus up to 256
generated ones) and is not available, so a standard-normal bf16 cache stands in for it.
Hidden rows [S, Smax-64) are filled with a constant (the pages' tests use 7.0) or with
arbitrary garbage to check that they are never read.

Everything is drawn on the CPU from numpy's PCG64 bit generator (a platform-independent
integer stream; normals by its ziggurat in float64) and then rounded to bf16, so a given seed
yields the same bytes on x86 and on Arm. (torch's CPU ``randn`` is not bit-identical across
instruction sets: its vectorised transform differs in the last bits, which flips the bf16
rounding of a few values.)
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

HQ, HKV, D, T = 16, 8, 128, 64


def _bf16(a: np.ndarray) -> torch.Tensor:
    """float64 samples -> float32 -> bf16 tensor. Both casts are IEEE round-to-nearest-even
    conversions, so the result is the same on every platform."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


@dataclass
class LayerInputs:
    q_raw: torch.Tensor    # bf16 [16, 64, 128]
    k_raw: torch.Tensor    # bf16 [8, 64, 128]
    v_raw: torch.Tensor    # bf16 [8, 64, 128]
    q_gamma: torch.Tensor  # bf16 [128]
    k_gamma: torch.Tensor  # bf16 [128]
    k_cache: torch.Tensor  # bf16 [8, Smax, 128]
    v_cache: torch.Tensor  # bf16 [8, Smax, 128]
    S: int
    Smax: int


def layer_inputs(seed: int, S: int, Smax: int, hidden_fill: float | str = 7.0,
                 tail_fill: float | None = None) -> LayerInputs:
    """One layer's inputs, all bf16 on the CPU.

    raw q/k/v and cache K/V ~ N(0, 1); gains 1 + 0.1 N(0, 1). ``hidden_fill`` sets rows
    [S, Smax-64): a number, ``"garbage"`` (N(0, 1e4) values), ``"nan"`` or ``"inf"``.
    ``tail_fill`` optionally overwrites rows [Smax-64, Smax) before the call (they are
    rewritten by the path anyway).
    """
    assert 0 <= S <= Smax - T and Smax % T == 0
    rng = np.random.Generator(np.random.PCG64(int(seed)))
    q_raw = _bf16(rng.standard_normal((HQ, T, D)))
    k_raw = _bf16(rng.standard_normal((HKV, T, D)))
    v_raw = _bf16(rng.standard_normal((HKV, T, D)))
    q_gamma = _bf16(1.0 + 0.1 * rng.standard_normal(D))
    k_gamma = _bf16(1.0 + 0.1 * rng.standard_normal(D))
    k_cache = _bf16(rng.standard_normal((HKV, Smax, D)))
    v_cache = _bf16(rng.standard_normal((HKV, Smax, D)))
    fill_hidden(k_cache, v_cache, S, Smax, hidden_fill, seed)
    if tail_fill is not None:
        k_cache[:, Smax - T:] = tail_fill
        v_cache[:, Smax - T:] = tail_fill
    return LayerInputs(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_cache, v_cache, int(S), int(Smax))


def fill_hidden(k_cache: torch.Tensor, v_cache: torch.Tensor, S: int, Smax: int,
                hidden_fill: float | str, seed: int = 0) -> None:
    """Overwrite rows [S, Smax-64) of both caches in place."""
    lo, hi = S, Smax - T
    if hi <= lo:
        return
    if isinstance(hidden_fill, str):
        if hidden_fill == "garbage":
            rng = np.random.Generator(np.random.PCG64(int(seed) + 7919))
            for c in (k_cache, v_cache):
                c[:, lo:hi] = _bf16(1e4 * rng.standard_normal((c.shape[0], hi - lo, c.shape[2]))).to(c.device)
        elif hidden_fill == "nan":
            k_cache[:, lo:hi] = float("nan")
            v_cache[:, lo:hi] = float("nan")
        elif hidden_fill == "inf":
            k_cache[:, lo:hi] = float("inf")
            v_cache[:, lo:hi] = float("-inf")
        else:
            raise ValueError(hidden_fill)
    else:
        k_cache[:, lo:hi] = float(hidden_fill)
        v_cache[:, lo:hi] = float(hidden_fill)


def zero_inputs_like(x: LayerInputs, **zeroed: bool) -> LayerInputs:
    """A copy of x with the named tensors (e.g. ``q_raw=True``) set to zero."""
    d = dict(x.__dict__)
    for name, on in zeroed.items():
        if on:
            d[name] = torch.zeros_like(d[name])
    return LayerInputs(**d)


# Workloads of the benchmark and the parity tests. Seeds: 1000 * config + layer (config 0: 0).
CONFIGS = {
    0: dict(name="tiny single layer", layers=1, S=256, Smax=512, hidden_fill=7.0, kv="bf16"),
    1: dict(name="main shape, one layer", layers=1, S=4700, Smax=8192, hidden_fill=7.0, kv="bf16"),
    2: dict(name="tighter cache, one layer", layers=1, S=4700, Smax=5120, hidden_fill=7.0, kv="bf16"),
    3: dict(name="fp8 e4m3 cache, one layer", layers=1, S=4700, Smax=8192, hidden_fill=7.0, kv="fp8"),
    4: dict(name="64-layer Euler step", layers=64, S_sweep=(1024, 2048, 4700, 8128), Smax=8192,
            hidden_fill=7.0, kv="bf16"),
}


def config_seed(config: int, layer: int) -> int:
    return 0 if config == 0 else 1000 * config + layer


def layer_inputs_on_device(seed: int, S: int, Smax: int, device, hidden_fill: float = 7.0) -> LayerInputs:
    """Same distributions as :func:`layer_inputs`, drawn directly on ``device`` with a seeded
    generator of that device (used to fill the many layers of a full-size step quickly; the
    values differ from the CPU draw of the same seed)."""
    assert 0 <= S <= Smax - T and Smax % T == 0
    g = torch.Generator(device=device).manual_seed(int(seed))
    bf = torch.bfloat16
    r = lambda *shape: torch.randn(*shape, generator=g, device=device)  # noqa: E731
    x = LayerInputs(r(HQ, T, D).to(bf), r(HKV, T, D).to(bf), r(HKV, T, D).to(bf),
                    (1.0 + 0.1 * r(D)).to(bf), (1.0 + 0.1 * r(D)).to(bf),
                    r(HKV, Smax, D).to(bf), r(HKV, Smax, D).to(bf), int(S), int(Smax))
    fill_hidden(x.k_cache, x.v_cache, S, Smax, hidden_fill, seed)
    return x


# ------------------------------------------------------------------- whole decoder layer
# The expert's trained weights are not available, so the layer is exercised with synthetic
# ones of the model's shapes (alpamayo_tt/EXPERT_NOTES.md, "Matmul program configs": hidden
# 1536, wqkv 1536 -> 4096, wo 2048 -> 1536, w1 / w3 1536 -> 6144, w2 6144 -> 1536). Each weight
# is stored [out_features, in_features] and drawn N(0, 1 / in_features), so that activations
# stay of order one through the layer; norm gains are 1 + 0.1 N(0, 1); the residual stream
# x ~ N(0, 1).
HIDDEN, INTER, QKV_DIM, Q_DIM = 1536, 6144, 4096, 2048


@dataclass
class ExpertLayerWeights:
    ln1: torch.Tensor     # bf16 [hidden]
    wqkv: torch.Tensor    # bf16 [4096, hidden]: q (16 x 128), k (8 x 128), v (8 x 128) features
    q_norm: torch.Tensor  # bf16 [128]
    k_norm: torch.Tensor  # bf16 [128]
    wo: torch.Tensor      # bf16 [hidden, 2048]
    ln2: torch.Tensor     # bf16 [hidden]
    w1: torch.Tensor      # bf16 [inter, hidden] (gate)
    w3: torch.Tensor      # bf16 [inter, hidden] (up)
    w2: torch.Tensor      # bf16 [hidden, inter] (down)


def expert_layer_weights(seed: int, hidden: int = HIDDEN, inter: int = INTER) -> ExpertLayerWeights:
    """One layer's synthetic weights, bf16 on the CPU (numpy PCG64, as :func:`layer_inputs`)."""
    rng = np.random.Generator(np.random.PCG64(int(seed) + 104729))
    n = rng.standard_normal
    return ExpertLayerWeights(
        ln1=_bf16(1.0 + 0.1 * n(hidden)),
        wqkv=_bf16(n((QKV_DIM, hidden)) / np.sqrt(hidden)),
        q_norm=_bf16(1.0 + 0.1 * n(D)), k_norm=_bf16(1.0 + 0.1 * n(D)),
        wo=_bf16(n((hidden, Q_DIM)) / np.sqrt(Q_DIM)),
        ln2=_bf16(1.0 + 0.1 * n(hidden)),
        w1=_bf16(n((inter, hidden)) / np.sqrt(hidden)),
        w3=_bf16(n((inter, hidden)) / np.sqrt(hidden)),
        w2=_bf16(n((hidden, inter)) / np.sqrt(inter)))


def expert_layer_weights_on_device(seed: int, device, hidden: int = HIDDEN,
                                   inter: int = INTER) -> ExpertLayerWeights:
    """Same distributions drawn on ``device`` with a seeded generator of that device."""
    g = torch.Generator(device=device).manual_seed(int(seed) + 104729)
    bf = torch.bfloat16
    r = lambda *shape: torch.randn(*shape, generator=g, device=device)  # noqa: E731
    return ExpertLayerWeights(
        ln1=(1.0 + 0.1 * r(hidden)).to(bf),
        wqkv=(r(QKV_DIM, hidden) / hidden ** 0.5).to(bf),
        q_norm=(1.0 + 0.1 * r(D)).to(bf), k_norm=(1.0 + 0.1 * r(D)).to(bf),
        wo=(r(hidden, Q_DIM) / Q_DIM ** 0.5).to(bf),
        ln2=(1.0 + 0.1 * r(hidden)).to(bf),
        w1=(r(inter, hidden) / hidden ** 0.5).to(bf),
        w3=(r(inter, hidden) / hidden ** 0.5).to(bf),
        w2=(r(hidden, inter) / inter ** 0.5).to(bf))


def residual_stream(seed: int, hidden: int = HIDDEN) -> torch.Tensor:
    """The layer input x [64, hidden] ~ N(0, 1), bf16 on the CPU."""
    rng = np.random.Generator(np.random.PCG64(int(seed) + 15485863))
    return _bf16(rng.standard_normal((T, hidden)))


# ------------------------------------------------------------------- text-model decode step
# One decode step of the VLM text model over the same per-layer cache layout (alpamayo_tt/text.py,
# TTText._layer_decode): 64 query heads and 8 KV heads of width 128 for the single new token;
# the cache rows [0, pos) are valid and the step writes row pos.
HQ_TEXT = 64


@dataclass
class DecodeInputs:
    q_raw: torch.Tensor    # bf16 [64, 128]
    k_raw: torch.Tensor    # bf16 [8, 128]
    v_raw: torch.Tensor    # bf16 [8, 128]
    q_gamma: torch.Tensor  # bf16 [128]
    k_gamma: torch.Tensor  # bf16 [128]
    k_cache: torch.Tensor  # bf16 [8, Smax, 128]
    v_cache: torch.Tensor  # bf16 [8, Smax, 128]
    pos: int
    Smax: int


def decode_inputs(seed: int, pos: int, Smax: int, later_fill: float | str = 7.0) -> DecodeInputs:
    """One layer's decode-step inputs, all bf16 on the CPU (numpy PCG64, as layer_inputs).

    raw q/k/v and cache K/V ~ N(0, 1); gains 1 + 0.1 N(0, 1). Rows [pos, Smax) of both caches
    (the new token's row and the rows after it, not yet written by the text model) are set by
    ``later_fill``: a number, ``"garbage"``, ``"nan"`` or ``"inf"``.
    """
    assert 0 <= pos < Smax
    rng = np.random.Generator(np.random.PCG64(int(seed)))
    q_raw = _bf16(rng.standard_normal((HQ_TEXT, D)))
    k_raw = _bf16(rng.standard_normal((HKV, D)))
    v_raw = _bf16(rng.standard_normal((HKV, D)))
    q_gamma = _bf16(1.0 + 0.1 * rng.standard_normal(D))
    k_gamma = _bf16(1.0 + 0.1 * rng.standard_normal(D))
    k_cache = _bf16(rng.standard_normal((HKV, Smax, D)))
    v_cache = _bf16(rng.standard_normal((HKV, Smax, D)))
    _fill_rows(k_cache, v_cache, pos, Smax, later_fill, seed)
    return DecodeInputs(q_raw, k_raw, v_raw, q_gamma, k_gamma, k_cache, v_cache, int(pos), int(Smax))


def decode_inputs_on_device(seed: int, pos: int, Smax: int, device) -> DecodeInputs:
    """Same distributions as :func:`decode_inputs`, drawn on ``device`` (full-size workloads)."""
    assert 0 <= pos < Smax
    g = torch.Generator(device=device).manual_seed(int(seed))
    bf = torch.bfloat16
    r = lambda *shape: torch.randn(*shape, generator=g, device=device)  # noqa: E731
    x = DecodeInputs(r(HQ_TEXT, D).to(bf), r(HKV, D).to(bf), r(HKV, D).to(bf),
                     (1.0 + 0.1 * r(D)).to(bf), (1.0 + 0.1 * r(D)).to(bf),
                     r(HKV, Smax, D).to(bf), r(HKV, Smax, D).to(bf), int(pos), int(Smax))
    _fill_rows(x.k_cache, x.v_cache, pos, Smax, 7.0, seed)
    return x


def _fill_rows(k_cache: torch.Tensor, v_cache: torch.Tensor, lo: int, hi: int,
               fill: float | str, seed: int) -> None:
    """Overwrite rows [lo, hi) of both caches in place (a number, garbage, NaN or Inf)."""
    if hi <= lo:
        return
    if isinstance(fill, str):
        if fill == "garbage":
            rng = np.random.Generator(np.random.PCG64(int(seed) + 7919))
            for c in (k_cache, v_cache):
                c[:, lo:hi] = _bf16(1e4 * rng.standard_normal((c.shape[0], hi - lo, c.shape[2]))).to(c.device)
        elif fill == "nan":
            k_cache[:, lo:hi] = float("nan")
            v_cache[:, lo:hi] = float("nan")
        elif fill == "inf":
            k_cache[:, lo:hi] = float("inf")
            v_cache[:, lo:hi] = float("-inf")
        else:
            raise ValueError(fill)
    else:
        k_cache[:, lo:hi] = float(fill)
        v_cache[:, lo:hi] = float(fill)
