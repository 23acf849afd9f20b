"""GPU parity of the bf16 expert-attention path (prologue, split-KV tcgen05 attention, merge)
against the fp64 CPU oracle, called through the C ABI. Bar: max-abs <= 1e-2 and relative L2
<= 5e-3 on the bf16 output; the cache tail and the roped q within one bf16 step."""
import numpy as np
import pytest
import torch

import gqa_attention_long_gb300 as ea
from gqa_attention_long_gb300.inputs import config_seed, layer_inputs, layer_inputs_on_device
from tests._gpu_util import assert_close, bf16_ulp, check_status, errors, f64, oracle_layer, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    ea.lib()
    yield
    ea.expert_attn_set_splits(0)


def run_layer(x, rope_delta=0, want_q_rope=False):
    L = to_dev(x, want_q_rope)
    ws = ea.alloc_workspace(1, x.Smax)
    ea.expert_attn_layer(L, x.S, x.Smax, rope_delta, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    check_status(ws)
    return L


def test_prologue_matches_oracle_and_touches_only_the_tail():
    S, Smax, delta = 256, 512, 3
    x = layer_inputs(5, S, Smax)
    L = to_dev(x, want_q_rope=True)
    k_before, v_before = L.k_cache.clone(), L.v_cache.clone()
    ws = ea.alloc_workspace(1, Smax)
    ea.expert_attn_prologue(L, S, Smax, delta, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    r = oracle_layer(x, rope_delta=delta)
    # fp32 evaluation of O(1) terms errs by ~1e-6 absolute; near-zero outputs (cancellation in
    # the rotation) have a bf16 step far below that, hence the absolute slack.
    q = f64(L.q_rope)
    assert np.all(np.abs(q - r["q"]) <= bf16_ulp(r["q"]) + 1e-5)
    assert np.mean(np.abs(q - r["q"]) <= 0.5 * bf16_ulp(r["q"]) + 1e-6) > 0.999
    k_tail = f64(L.k_cache[:, Smax - 64:])
    assert np.all(np.abs(k_tail - r["k"]) <= bf16_ulp(r["k"]) + 1e-5)
    assert np.mean(k_tail == r["k_store"]) > 0.99  # equal to the oracle's bf16 store but for ties
    assert torch.equal(L.v_cache[:, Smax - 64:], x.v_raw.cuda())
    assert torch.equal(L.k_cache[:, :Smax - 64], k_before[:, :Smax - 64])
    assert torch.equal(L.v_cache[:, :Smax - 64], v_before[:, :Smax - 64])


@pytest.mark.parametrize("S", [0, 1, 63, 64, 127, 128, 129, 256, 300, 448])
def test_layer_small_sizes(S):
    x = layer_inputs(100 + S, S, 512)
    L = run_layer(x)
    assert_close(f64(L.out), oracle_layer(x)["out"], f"S={S}")


def test_config0_tiny():
    x = layer_inputs(config_seed(0, 0), 256, 512)
    L = run_layer(x)
    assert_close(f64(L.out), oracle_layer(x)["out"])


@pytest.mark.parametrize("cfg,S,Smax", [(1, 4700, 8192), (2, 4700, 5120)])
def test_main_shapes(cfg, S, Smax):
    x = layer_inputs(config_seed(cfg, 0), S, Smax)
    L = run_layer(x)
    assert_close(f64(L.out), oracle_layer(x)["out"], f"config {cfg}")


def test_rope_delta_and_odd_sizes():
    x = layer_inputs(77, 1000, 1152)
    L = run_layer(x, rope_delta=-37)
    assert_close(f64(L.out), oracle_layer(x, rope_delta=-37)["out"])


def test_hidden_rows_are_never_read():
    S, Smax = 300, 1024
    outs = []
    for fill in (7.0, "nan", "inf", "garbage"):
        x = layer_inputs(9, S, Smax, hidden_fill=fill)
        L = to_dev(x)
        hidden_k = L.k_cache[:, S:Smax - 64].clone()
        hidden_v = L.v_cache[:, S:Smax - 64].clone()
        ws = ea.alloc_workspace(1, Smax)
        ea.expert_attn_layer(L, S, Smax, 0, ea.EA_KV_BF16, ws)
        torch.cuda.synchronize()
        check_status(ws)
        # hidden rows are left exactly as they were (NaN payloads compared as bytes)
        assert torch.equal(L.k_cache[:, S:Smax - 64].view(torch.int16), hidden_k.view(torch.int16))
        assert torch.equal(L.v_cache[:, S:Smax - 64].view(torch.int16), hidden_v.view(torch.int16))
        outs.append(L.out.clone())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_many_layers_one_call():
    S, Smax, n = 777, 1024, 5
    xs = [layer_inputs(300 + l, S, Smax) for l in range(n)]
    Ls = [to_dev(x) for x in xs]
    ws = ea.alloc_workspace(n, Smax)
    ea.expert_attn_layers(Ls, S, Smax, 0, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    check_status(ws)
    for x, L in zip(xs, Ls):
        assert_close(f64(L.out), oracle_layer(x)["out"])


@pytest.mark.parametrize("splits", [1, 5, 37, 0])
def test_split_count_does_not_change_the_result(splits):
    x = layer_inputs(11, 2000, 2112)
    ea.expert_attn_set_splits(splits)
    try:
        L = run_layer(x)
    finally:
        ea.expert_attn_set_splits(0)
    assert_close(f64(L.out), oracle_layer(x)["out"], f"splits={splits}")


def test_repeatable_bitwise():
    x = layer_inputs(12, 3000, 4096)
    a = run_layer(x).out
    b = run_layer(x).out
    assert torch.equal(a, b)


def test_workspace_too_small_is_refused():
    x = layer_inputs(13, 10, 128)
    L = to_dev(x)
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(ea.ExpertAttnError) as e:
        ea.expert_attn_layer(L, 10, 128, 0, ea.EA_KV_BF16, ws)
    assert e.value.rc == 4


@pytest.mark.parametrize("S", [4700, 1024, 2048, 8128])
def test_64_layer_step_full_size_sampled(S):
    """The 64-layer Euler-step workload at its full size, in the launch configuration the
    benchmark times; the oracle checks every output of a few sampled layers."""
    Smax, n = 8192, 64
    dev = torch.device("cuda")
    xs = [layer_inputs_on_device(4000 + l, S, Smax, dev) for l in range(n)]
    Ls = [ea.LayerBuffers(q_raw=x.q_raw, k_raw=x.k_raw, v_raw=x.v_raw, q_gamma=x.q_gamma,
                          k_gamma=x.k_gamma, k_cache=x.k_cache, v_cache=x.v_cache,
                          out=torch.full((16, 64, 128), float("nan"), dtype=torch.bfloat16, device=dev))
          for x in xs]
    ws = ea.alloc_workspace(n, Smax)
    ea.expert_attn_layers(Ls, S, Smax, 0, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    check_status(ws)
    for l in ([0, 31, 63] if S == 4700 else [17, 50]):
        x = xs[l]
        host = type(x)(**{k: (v.cpu() if torch.is_tensor(v) else v) for k, v in x.__dict__.items()})
        # the kernel overwrote the tail rows; the oracle recomputes them from the raw inputs
        assert_close(f64(Ls[l].out), oracle_layer(host)["out"], f"S={S} layer {l}")
    for L in Ls:
        assert torch.isfinite(L.out.float()).all()


def test_layer_writes_q_rope_and_tail_itself():
    """With a bf16 cache the attention kernel does the prologue: its roped q and cache tail are
    those of the oracle (within a bf16 step) and the same bits as the standalone prologue's."""
    S, Smax, delta = 700, 1024, -5
    x = layer_inputs(21, S, Smax)
    A = to_dev(x, want_q_rope=True)
    B = to_dev(x, want_q_rope=True)
    k_before, v_before = A.k_cache.clone(), A.v_cache.clone()
    ws = ea.alloc_workspace(1, Smax)
    ea.expert_attn_layer(A, S, Smax, delta, ea.EA_KV_BF16, ws)
    ea.expert_attn_prologue(B, S, Smax, delta, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    check_status(ws)
    r = oracle_layer(x, rope_delta=delta)
    q = f64(A.q_rope)
    assert np.all(np.abs(q - r["q"]) <= bf16_ulp(r["q"]) + 1e-5)
    k_tail = f64(A.k_cache[:, Smax - 64:])
    assert np.all(np.abs(k_tail - r["k"]) <= bf16_ulp(r["k"]) + 1e-5)
    assert torch.equal(A.v_cache[:, Smax - 64:], x.v_raw.cuda())
    assert torch.equal(A.q_rope.view(torch.int16), B.q_rope.view(torch.int16))
    assert torch.equal(A.k_cache.view(torch.int16), B.k_cache.view(torch.int16))
    assert torch.equal(A.k_cache[:, :Smax - 64], k_before[:, :Smax - 64])
    assert torch.equal(A.v_cache[:, :Smax - 64], v_before[:, :Smax - 64])
    assert_close(f64(A.out), r["out"])


def test_q_rope_of_every_layer_in_a_split_call():
    """Eight layers over few CTAs: units are cut between CTAs, and exactly one CTA per unit (the
    one holding its own-row tile) writes that unit's roped q and cache tail."""
    S, Smax, n = 900, 1024, 8
    xs = [layer_inputs(600 + l, S, Smax) for l in range(n)]
    Ls = [to_dev(x, want_q_rope=True) for x in xs]
    ws = ea.alloc_workspace(n, Smax)
    ea.expert_attn_set_splits(23)
    try:
        ea.expert_attn_layers(Ls, S, Smax, 2, ea.EA_KV_BF16, ws)
        torch.cuda.synchronize()
    finally:
        ea.expert_attn_set_splits(0)
    check_status(ws)
    for x, L in zip(xs, Ls):
        r = oracle_layer(x, rope_delta=2)
        assert np.all(np.abs(f64(L.q_rope) - r["q"]) <= bf16_ulp(r["q"]) + 1e-5)
        assert np.all(np.abs(f64(L.k_cache[:, Smax - 64:]) - r["k"]) <= bf16_ulp(r["k"]) + 1e-5)
        assert_close(f64(L.out), r["out"])


def test_repeated_calls_leave_merge_words_zero():
    """Two-part units are merged inside the attention kernel through per-unit words in the
    workspace; each call leaves them zero, so back-to-back calls on one workspace agree bit for
    bit without re-initialising it."""
    S, Smax, n = 1024, 2048, 64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    parts = ea.split_parts(n, S, sms)
    assert parts and all(k == 2 for _, k in parts)  # the in-kernel merge is taken
    dev = torch.device("cuda")
    xs = [layer_inputs_on_device(9000 + l, S, Smax, dev) for l in range(n)]
    Ls = [ea.LayerBuffers(q_raw=x.q_raw, k_raw=x.k_raw, v_raw=x.v_raw, q_gamma=x.q_gamma,
                          k_gamma=x.k_gamma, k_cache=x.k_cache, v_cache=x.v_cache,
                          out=torch.empty(16, 64, 128, dtype=torch.bfloat16, device=dev)) for x in xs]
    ws = ea.alloc_workspace(n, Smax)
    outs = []
    for _ in range(3):
        ea.expert_attn_layers(Ls, S, Smax, 0, ea.EA_KV_BF16, ws)
        torch.cuda.synchronize()
        check_status(ws)
        assert int(ws[1024:1024 + n * 8 * 2 * 4].count_nonzero()) == 0
        outs.append(torch.stack([L.out for L in Ls]).clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    host = type(xs[5])(**{k: (v.cpu() if torch.is_tensor(v) else v) for k, v in xs[5].__dict__.items()})
    assert_close(f64(Ls[5].out), oracle_layer(host)["out"])


def max_moving_inputs(seed, S=448, Smax=512):
    """Cache keys that make the running row max move by more than the softmax's lazy-rescale
    margin (8 in log2 units) inside a tile and across tiles, with moderate scores: rows
    [0, 320) are zero (every score 0: tiles 0-1 and the first half of tile 2), rows [320, S)
    are N(0, 2.8^2), whose largest score in a 64-key chunk is ~6.7 (9.7 in log2 units)."""
    x = layer_inputs(seed, S, Smax)
    j = torch.arange(Smax, dtype=torch.float32)
    sc = torch.where(j < 320, torch.zeros_like(j), torch.full_like(j, 2.8))
    x.k_cache = (x.k_cache.float() * sc[None, :, None]).to(torch.bfloat16)
    return x


def oracle_on_bf16_q(x, k_own=None, v_own=None, k_cache=None, v_cache=None):
    """The oracle's attention with the oracle's own roped q rounded to bf16 (the precision the
    tensor cores take it in): with peaked attention the rounding of q alone moves the output by
    more than the bf16 bar, which this reference leaves out, so that the check is on the rest."""
    import oracle
    q, k, v = oracle.prologue(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                              f64(x.k_gamma), x.S, 0)
    kc = f64(x.k_cache) if k_cache is None else k_cache
    vc = f64(x.v_cache) if v_cache is None else v_cache
    return oracle.attention_concat(oracle.bf16_round(q), kc, vc, x.S,
                                   oracle.bf16_round(k) if k_own is None else k_own,
                                   v if v_own is None else v_own)


@pytest.mark.parametrize("splits", [0, 3])
def test_running_max_moves_inside_and_across_tiles(splits):
    # the P already written for the first half of a tile and the accumulator of the earlier
    # tiles are rescaled, in every split of the key range
    x = max_moving_inputs(777)
    prev = ea.expert_attn_set_splits(splits)
    try:
        L = run_layer(x)
    finally:
        ea.expert_attn_set_splits(prev)
    assert_close(f64(L.out), oracle_on_bf16_q(x), f"running max moves, splits={splits}")


@pytest.mark.parametrize("scale", [3.0e5, 1.0e-6])
@pytest.mark.parametrize("splits", [0, 37])
def test_split_partials_keep_precision_at_any_magnitude(scale, splits):
    # The split partials travel as f16 with a power-of-two scale per half row. V rows (cache and
    # own) far above the f16 range (3e5) or far below its normal range (1e-6) must come out as
    # accurately as unit-size ones: one layer over every SM (units of ~19 parts, merged by the
    # grid) and 37 CTAs (two- and three-part units).
    import dataclasses
    x = layer_inputs(14, 2000, 2112)
    x = dataclasses.replace(x, v_raw=(x.v_raw.float() * scale).to(torch.bfloat16),
                            v_cache=(x.v_cache.float() * scale).to(torch.bfloat16))
    ea.expert_attn_set_splits(splits)
    try:
        L = run_layer(x)
    finally:
        ea.expert_attn_set_splits(0)
    got, ref = f64(L.out), oracle_layer(x)["out"]
    mx, rel = errors(got, ref)
    assert mx <= 1e-2 * scale and rel <= 5e-3, f"scale={scale}, splits={splits}: max-abs {mx:.3e}, rel-L2 {rel:.3e}"
