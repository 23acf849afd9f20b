"""Randomised GPU parity: layer counts, cache lengths, valid rows, positions, rope_delta and the
split count drawn from a seeded generator, for the expert attention (bf16 and e4m3 caches) and
the text model's decode step, each layer of each call checked against the fp64 CPU oracle. The
fixed cases elsewhere pin the edges; these cover the planner's and the kernels' combinations in
between (split units with 1, 2 or many parts, several segments per CTA, clusters)."""
import random

import numpy as np
import pytest
import torch

import gqa_attention_long_gb300 as ea
import oracle
from gqa_attention_long_gb300.inputs import decode_inputs, layer_inputs
from tests._gpu_util import assert_close, check_status, f64, oracle_layer, to_dev
from tests.test_gpu_fp8 import TOL_FP8_MAX_ABS, oracle_fp8, run_fp8_layers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    ea.lib()
    yield
    ea.expert_attn_set_splits(0)


@pytest.mark.parametrize("case", range(8))
def test_random_expert_bf16(case):
    rng = random.Random(4000 + case)
    Smax = 64 * rng.randint(2, 32)
    S = rng.randint(0, Smax - 64)
    n = rng.randint(1, 9)
    delta = rng.randint(-300, 300)
    splits = rng.choice([0, 0, rng.randint(1, 152)])
    xs = [layer_inputs(5000 + 10 * case + l, S, Smax, hidden_fill=rng.choice([7.0, "garbage"]))
          for l in range(n)]
    Ls = [to_dev(x) for x in xs]
    ws = ea.alloc_workspace(n, Smax)
    ea.expert_attn_set_splits(splits)
    try:
        ea.expert_attn_layers(Ls, S, Smax, delta, ea.EA_KV_BF16, ws)
        torch.cuda.synchronize()
    finally:
        ea.expert_attn_set_splits(0)
    check_status(ws)
    for l, (x, L) in enumerate(zip(xs, Ls)):
        assert_close(f64(L.out), oracle_layer(x, rope_delta=delta)["out"],
                     f"n={n} S={S} Smax={Smax} delta={delta} splits={splits} layer {l}")


@pytest.mark.parametrize("case", range(4))
def test_random_expert_fp8(case):
    rng = random.Random(4100 + case)
    Smax = 128 * rng.randint(2, 16)
    S = rng.randint(0, Smax - 64)
    n = rng.randint(1, 6)
    delta = rng.randint(-300, 300)
    xs = [layer_inputs(5200 + 10 * case + l, S, Smax) for l in range(n)]
    Ls = run_fp8_layers(xs, rope_delta=delta)
    for l, (x, L) in enumerate(zip(xs, Ls)):
        err = np.max(np.abs(f64(L.out) - oracle_fp8(x, rope_delta=delta)["out"]))
        assert err <= TOL_FP8_MAX_ABS, f"n={n} S={S} Smax={Smax} layer {l}: max-abs {err:.3e}"


@pytest.mark.parametrize("case", range(8))
def test_random_decode(case):
    rng = random.Random(4200 + case)
    Smax = 64 * rng.randint(2, 32)
    pos = rng.randint(0, Smax - 1)
    n = rng.randint(1, 9)
    delta = rng.randint(-300, 300)
    xs = [decode_inputs(5400 + 10 * case + l, pos, Smax, later_fill=rng.choice([7.0, "garbage", "nan"]))
          for l in range(n)]
    d = torch.device("cuda")
    Ls = [ea.DecodeBuffers(q_raw=x.q_raw.to(d), k_raw=x.k_raw.to(d), v_raw=x.v_raw.to(d),
                           q_gamma=x.q_gamma.to(d), k_gamma=x.k_gamma.to(d), k_cache=x.k_cache.to(d),
                           v_cache=x.v_cache.to(d),
                           out=torch.full((64, 128), float("nan"), dtype=torch.bfloat16, device=d))
          for x in xs]
    ws = ea.alloc_decode_workspace(n)
    ea.text_decode_attention(Ls, pos, Smax, delta, ws)
    torch.cuda.synchronize()
    check_status(ws)
    for l, (x, L) in enumerate(zip(xs, Ls)):
        ref = oracle.text_decode_attention(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                                           f64(x.k_gamma), f64(x.k_cache), f64(x.v_cache), pos, delta)
        assert_close(f64(L.out), ref["out"], f"n={n} pos={pos} Smax={Smax} delta={delta} layer {l}")
