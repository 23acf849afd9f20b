"""Host-side launch planning (no GPU): the list of units that the attention kernel's partition
cuts between CTAs, which the kernel merges (in the epilogue for two-part units, across the grid
for more parts), checked against a brute-force count of the CTAs whose tile range meets each
unit."""
import random

import pytest

from gqa_attention_long_gb300 import EA_KV_BF16, EA_KV_FP8_E4M3, kernels_per_call, split_parts, split_units


def brute_force_parts(n_layers, S, n_ctas):
    T = (S + 127) // 128 + 1
    W = n_layers * 8 * T
    n = max(1, min(n_ctas, 257, W))
    ranges = [(c * W // n, (c + 1) * W // n) for c in range(n)]
    out = []
    for u in range(n_layers * 8):
        lo, hi = u * T, (u + 1) * T
        parts = sum(1 for a, b in ranges if a < hi and b > lo and b > a)
        if parts >= 2:
            out.append((u, parts))
    return out


def brute_force(n_layers, S, n_ctas):
    return [u for u, _ in brute_force_parts(n_layers, S, n_ctas)]


@pytest.mark.parametrize("n_layers,S,n_ctas", [(1, 4700, 152), (64, 4700, 152), (64, 8128, 152),
                                               (8, 1024, 152), (1, 0, 152), (2, 300, 5), (64, 4700, 1),
                                               (64, 4700, 64), (3, 129, 37)])
def test_split_units_match_brute_force(n_layers, S, n_ctas):
    assert split_units(n_layers, S, n_ctas) == brute_force(n_layers, S, n_ctas)


def test_split_units_random():
    rng = random.Random(7)
    for _ in range(200):
        n_layers, S, n_ctas = rng.randint(1, 64), rng.randint(0, 8128), rng.randint(1, 300)
        assert split_units(n_layers, S, n_ctas) == brute_force(n_layers, S, n_ctas)


def test_single_layer_splits_every_unit():
    # one layer over all 152 SMs: every (kv head) unit spans ~19 CTAs and needs the grid merge
    assert split_units(1, 4700, 152) == list(range(8))


def test_split_parts_random():
    rng = random.Random(11)
    for _ in range(200):
        n_layers, S, n_ctas = rng.randint(1, 64), rng.randint(0, 8128), rng.randint(1, 300)
        assert split_parts(n_layers, S, n_ctas) == brute_force_parts(n_layers, S, n_ctas)


def test_kernel_count():
    # the attention kernel merges every split unit itself (two-part units in the epilogue, units
    # of more parts across the grid), so a bf16 call is one kernel per 64 layers and an e4m3 call
    # two (with the prologue)
    assert all(k == 2 for _, k in split_parts(64, 4700, 152))
    assert kernels_per_call(64, 4700, 152, EA_KV_BF16) == 1
    assert kernels_per_call(64, 4700, 152, EA_KV_FP8_E4M3) == 2
    assert all(k > 2 for _, k in split_parts(1, 4700, 152))
    assert kernels_per_call(1, 4700, 152, EA_KV_BF16) == 1
    assert kernels_per_call(1, 4700, 152, EA_KV_FP8_E4M3) == 2
    assert kernels_per_call(128, 4700, 152, EA_KV_BF16) == 2
