"""The entry point without a caller workspace (expert_attn_layers_noalloc), for callers that may
not allocate device memory (a plugin inside an engine that owns the whole memory budget, or a
loop where cudaMalloc / cudaFree are banned because they can synchronise the device).

Through the C ABI: two calls in a row over the shared static scratch (the second finds the first
call's leftovers there) match the fp64 oracle within the bf16 bar, and match the workspace path;
an e4m3 call matches the oracle on the dequantised cache within the FP8 bar; the status word of
the static scratch reads back clean after each call (expert_attn_noalloc_read_status); more
layers than the scratch holds are refused before anything is launched.

Kept in a file of its own that pytest collects last."""
import ctypes

import pytest
import torch

import gqa_attention_long_gb300 as ea
from gqa_attention_long_gb300 import _lib
from gqa_attention_long_gb300.inputs import layer_inputs
from tests._gpu_util import assert_close, check_status, f64, oracle_layer, to_dev
from tests.test_gpu_fp8 import check_out, oracle_fp8, quantize_on_gpu

pytestmark = pytest.mark.gpu

MAX_LAYERS = 4  # EA_NOALLOC_MAX_LAYERS in include/expert_attn.h


def _noalloc():
    f = ea.lib().expert_attn_layers_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(_lib.EaLayerArgs), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return f


def _stream():
    return torch.cuda.current_stream().cuda_stream


def noalloc_status():
    f = ea.lib().expert_attn_noalloc_read_status
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_uint32)]
    st, bits = ctypes.c_int(-1), ctypes.c_uint32(0)
    rc = f(_stream(), ctypes.byref(st), ctypes.byref(bits))
    assert rc == 0, ea.expert_attn_status_string(rc)
    return st.value, bits.value


def _run_noalloc(Ls, S, Smax, kv_dtype):
    arr = ea.make_args(Ls, Smax, kv_dtype)
    rc = _noalloc()(arr, len(Ls), S, Smax, 0, kv_dtype, _stream())
    assert rc == 0, ea.expert_attn_status_string(rc)
    torch.cuda.synchronize()
    st, bits = noalloc_status()
    assert st == 0, f"a kernel of the no-allocation call gave up a wait, status bits {bits:#x}"


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    # call 1: four layers of the main shape; call 2: two layers of another shape over the same
    # static scratch
    for seed0, n, S, Smax in [(700, MAX_LAYERS, 4700, 8192), (800, 2, 333, 512)]:
        xs = [layer_inputs(seed0 + l, S, Smax) for l in range(n)]
        got = [to_dev(x) for x in xs]
        _run_noalloc(got, S, Smax, ea.EA_KV_BF16)
        ref = [to_dev(x) for x in xs]
        ws = ea.alloc_workspace(n, Smax)
        ea.expert_attn_layers(ref, S, Smax, 0, ea.EA_KV_BF16, ws)
        torch.cuda.synchronize()
        check_status(ws)
        for x, a, b in zip(xs, ref, got):
            assert_close(f64(b.out), oracle_layer(x)["out"], f"noalloc vs oracle, S={S}")
            assert_close(f64(b.out), f64(a.out), f"noalloc vs workspace path, S={S}")
            assert torch.equal(b.k_cache, a.k_cache) and torch.equal(b.v_cache, a.v_cache)


def test_noalloc_fp8_matches_oracle():
    S, Smax, n = 1000, 1280, 2
    xs = [layer_inputs(850 + l, S, Smax) for l in range(n)]
    Ls = []
    for x in xs:
        kq, ks = quantize_on_gpu(x.k_cache, S, Smax)
        vq, vs = quantize_on_gpu(x.v_cache, S, Smax)
        Ls.append(ea.LayerBuffers(
            q_raw=x.q_raw.cuda(), k_raw=x.k_raw.cuda(), v_raw=x.v_raw.cuda(), q_gamma=x.q_gamma.cuda(),
            k_gamma=x.k_gamma.cuda(), k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs,
            out=torch.full((16, 64, 128), float("nan"), dtype=torch.bfloat16, device="cuda")))
    _run_noalloc(Ls, S, Smax, ea.EA_KV_FP8_E4M3)
    for x, L in zip(xs, Ls):
        check_out(L, oracle_fp8(x), "noalloc e4m3 vs oracle")


def test_noalloc_refuses_more_layers_than_its_scratch_holds():
    xs = [layer_inputs(900 + l, 10, 128) for l in range(MAX_LAYERS + 1)]
    Ls = [to_dev(x) for x in xs]
    before = [L.out.clone() for L in Ls]
    arr = ea.make_args(Ls, 128, ea.EA_KV_BF16)
    rc = _noalloc()(arr, MAX_LAYERS + 1, 10, 128, 0, ea.EA_KV_BF16, _stream())
    assert rc == 4  # EA_ERR_WORKSPACE: nothing launched
    torch.cuda.synchronize()
    for L, b in zip(Ls, before):
        assert torch.equal(L.out.view(torch.int16), b.view(torch.int16))
    assert noalloc_status() == (0, 0)
