"""Shared helpers of the GPU parity tests: move seeded inputs to the device, run the library
through the C ABI, run the fp64 oracle on the same host arrays, and compare."""
from __future__ import annotations

import numpy as np
import torch

import gqa_attention_long_gb300 as ea
import oracle

# Acceptance bar for bf16 caches (max-abs and relative L2 against the fp64 oracle).
TOL_MAX_ABS = 1e-2
TOL_REL_L2 = 5e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def to_dev(x, want_q_rope=False) -> ea.LayerBuffers:
    d = torch.device("cuda")
    return ea.LayerBuffers(
        q_raw=x.q_raw.to(d), k_raw=x.k_raw.to(d), v_raw=x.v_raw.to(d), q_gamma=x.q_gamma.to(d),
        k_gamma=x.k_gamma.to(d), k_cache=x.k_cache.to(d), v_cache=x.v_cache.to(d),
        out=torch.full((16, 64, 128), float("nan"), dtype=torch.bfloat16, device=d),
        q_rope=torch.zeros(16, 64, 128, dtype=torch.bfloat16, device=d) if want_q_rope else None)


def oracle_layer(x, rope_delta=0, form="concat") -> dict:
    return oracle.expert_attention_layer(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                                         f64(x.k_gamma), f64(x.k_cache), f64(x.v_cache),
                                         x.S, x.Smax, rope_delta, form=form)


def errors(got: np.ndarray, ref: np.ndarray) -> tuple[float, float]:
    assert np.all(np.isfinite(got)), "non-finite output"
    return float(np.max(np.abs(got - ref))), float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "out") -> None:
    mx, rel = errors(got, ref)
    assert mx <= TOL_MAX_ABS and rel <= TOL_REL_L2, f"{what}: max-abs {mx:.3e}, rel-L2 {rel:.3e}"


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def check_status(ws: torch.Tensor) -> None:
    st, bits = ea.expert_attn_read_status(ws)
    assert st == ea.EA_OK, f"kernel gave up a wait, status bits {bits:#x}"
