"""GPU parity of the FP8 (OCP e4m3, per-128-row block scales) cache variant against the fp64 CPU
oracle run on the same dequantised cache values. Bars: the cache quantiser is bit-exact (codes and
scales); the attention output is within max-abs 2e-2 of the oracle."""
import numpy as np
import pytest
import torch

import gqa_attention_long_gb300 as ea
import oracle
from gqa_attention_long_gb300.inputs import config_seed, layer_inputs
from tests._gpu_util import check_status, f64

pytestmark = pytest.mark.gpu
TOL_FP8_MAX_ABS = 2e-2


def ncol(Smax):
    return Smax // 128 + 1


def quantize_on_gpu(cache_bf16, n_rows, Smax, fill_code=0x7F):
    """The library's cache producer; rows >= n_rows get NaN codes (they must never be read)."""
    dst = torch.full((8, Smax, 128), fill_code, dtype=torch.uint8, device="cuda")
    sc = torch.full((8, ncol(Smax)), float("nan"), dtype=torch.float32, device="cuda")
    ea.expert_attn_quantize_cache(cache_bf16.cuda().contiguous(), n_rows, Smax, dst, sc)
    return dst, sc


def run_fp8_layers(xs, rope_delta=0):
    S, Smax = xs[0].S, xs[0].Smax
    Ls = []
    for x in xs:
        kq, ks = quantize_on_gpu(x.k_cache, S, Smax)
        vq, vs = quantize_on_gpu(x.v_cache, S, Smax)
        Ls.append(ea.LayerBuffers(
            q_raw=x.q_raw.cuda(), k_raw=x.k_raw.cuda(), v_raw=x.v_raw.cuda(), q_gamma=x.q_gamma.cuda(),
            k_gamma=x.k_gamma.cuda(), k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs,
            out=torch.full((16, 64, 128), float("nan"), dtype=torch.bfloat16, device="cuda")))
    ws = ea.alloc_workspace(len(xs), Smax, ea.EA_KV_FP8_E4M3)
    ea.expert_attn_layers(Ls, S, Smax, rope_delta, ea.EA_KV_FP8_E4M3, ws)
    torch.cuda.synchronize()
    check_status(ws)
    return Ls


def oracle_fp8(x, rope_delta=0):
    S, Smax = x.S, x.Smax
    kc, ks = oracle.quantize_cache_blocks(f64(x.k_cache), S, Smax)
    vc, vs = oracle.quantize_cache_blocks(f64(x.v_cache), S, Smax)
    return oracle.expert_attention_layer_fp8(f64(x.q_raw), f64(x.k_raw), f64(x.v_raw), f64(x.q_gamma),
                                             f64(x.k_gamma), kc, ks, vc, vs, S, Smax, rope_delta)


def check_out(L, r, what):
    got = f64(L.out)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - r["out"])
    rel = np.linalg.norm(got - r["out"]) / np.linalg.norm(r["out"])
    assert err.max() <= TOL_FP8_MAX_ABS, f"{what}: max-abs {err.max():.3e} (rel-L2 {rel:.3e})"
    return err.max(), rel


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    ea.lib()


@pytest.mark.parametrize("S,Smax", [(4700, 8192), (300, 512), (0, 256), (1, 256), (128, 384), (448, 512)])
def test_cache_quantiser_bit_exact(S, Smax):
    x = layer_inputs(config_seed(3, 0) + S, S, Smax)
    for cache in (x.k_cache, x.v_cache):
        codes, sc = quantize_on_gpu(cache, S, Smax)
        oc, os_ = oracle.quantize_cache_blocks(f64(cache), S, Smax)
        nb = (S + 127) // 128
        assert np.array_equal(codes.cpu().numpy()[:, :S], oc[:, :S])
        assert np.array_equal(sc.cpu().numpy()[:, :nb], os_[:, :nb])
        assert np.all(codes.cpu().numpy()[:, S:] == 0x7F)  # rows >= n_rows untouched


def test_config3_fp8_main_shape():
    x = layer_inputs(config_seed(3, 0), 4700, 8192)
    L = run_fp8_layers([x])[0]
    r = oracle_fp8(x)
    check_out(L, r, "config 3")
    # own rows: v codes and scale exact; k within one code step on the few values where the
    # fp32 rotation and the fp64 one fall on different sides of a rounding boundary
    Smax = 8192
    vt = L.v_cache[:, Smax - 64:].cpu().numpy()
    assert np.array_equal(vt, r["v_tail_codes"])
    assert np.array_equal(L.v_scale.cpu().numpy()[:, -1], r["v_tail_scale"])
    kt = L.k_cache[:, Smax - 64:].cpu().numpy().astype(np.int16)
    diff = np.abs(kt - r["k_tail_codes"].astype(np.int16))
    assert np.mean(diff == 0) > 0.99 and np.max(diff) <= 1
    assert np.allclose(L.k_scale.cpu().numpy()[:, -1], r["k_tail_scale"], rtol=1e-5)


@pytest.mark.parametrize("S,Smax", [(0, 256), (1, 256), (127, 384), (128, 384), (129, 384), (448, 512)])
def test_fp8_small_sizes(S, Smax):
    x = layer_inputs(500 + S, S, Smax)
    L = run_fp8_layers([x])[0]
    check_out(L, oracle_fp8(x), f"S={S}")


def test_fp8_many_layers_and_rope_delta():
    xs = [layer_inputs(600 + l, 1000, 1152) for l in range(3)]
    Ls = run_fp8_layers(xs, rope_delta=17)
    for x, L in zip(xs, Ls):
        check_out(L, oracle_fp8(x, rope_delta=17), "fp8 3 layers")


def test_fp8_sixteen_layers_split_units():
    # 16 layers at the main shape: CTAs hold several units, some split and merged
    xs = [layer_inputs(700 + l, 4700, 8192) for l in range(16)]
    Ls = run_fp8_layers(xs)
    for l in (0, 7, 15):
        check_out(Ls[l], oracle_fp8(xs[l]), f"layer {l}")
    for L in Ls:
        assert torch.isfinite(L.out.float()).all()


def test_workspace_size_by_dtype():
    """Only an e4m3 call stages the roped Q codes in the workspace (32 KB per unit); a bf16 call
    prepares Q in the attention kernel's shared memory, and a bf16-sized workspace is refused
    for an e4m3 call before anything is launched."""
    b = ea.expert_attn_workspace_size(64, 8192, ea.EA_KV_BF16)
    f = ea.expert_attn_workspace_size(64, 8192, ea.EA_KV_FP8_E4M3)
    assert f - b == 64 * 8 * 32768
    S, Smax = 256, 512
    x = layer_inputs(config_seed(3, 7), S, Smax)
    codes_k, sk = quantize_on_gpu(x.k_cache, S, Smax)
    codes_v, sv = quantize_on_gpu(x.v_cache, S, Smax)
    d = torch.device("cuda")
    L = ea.LayerBuffers(q_raw=x.q_raw.to(d), k_raw=x.k_raw.to(d), v_raw=x.v_raw.to(d),
                        q_gamma=x.q_gamma.to(d), k_gamma=x.k_gamma.to(d), k_cache=codes_k,
                        v_cache=codes_v, k_scale=sk, v_scale=sv,
                        out=torch.empty(16, 64, 128, dtype=torch.bfloat16, device=d))
    ws = ea.alloc_workspace(1, Smax, ea.EA_KV_BF16)
    with pytest.raises(ea.ExpertAttnError) as e:
        ea.expert_attn_layer(L, S, Smax, 0, ea.EA_KV_FP8_E4M3, ws)
    assert e.value.rc == 4



def test_fp8_running_max_moves_inside_and_across_tiles():
    # the bf16 test of the same name on an e4m3 cache (its P is rescaled as f16 pairs); the
    # reference is the oracle on the dequantised cache with the bf16-rounded roped q
    from tests.test_gpu_attention import max_moving_inputs, oracle_on_bf16_q
    x = max_moving_inputs(778)
    L = run_fp8_layers([x])[0]
    r = oracle_fp8(x)
    kc, ks = oracle.quantize_cache_blocks(f64(x.k_cache), x.S, x.Smax)
    vc, vs = oracle.quantize_cache_blocks(f64(x.v_cache), x.S, x.Smax)
    ref = oracle_on_bf16_q(x, r["k_store"], r["v_store"], oracle.dequantize_cache(kc, ks, x.S),
                           oracle.dequantize_cache(vc, vs, x.S))
    got = f64(L.out)
    err = np.abs(got - ref).max()
    assert np.all(np.isfinite(got)) and err <= TOL_FP8_MAX_ABS, f"max-abs {err:.3e}"
