"""The entry point without a caller workspace (expert_attn_layers_noalloc), for callers that may
not allocate device memory: it must give the same result as expert_attn_layers with a normal
workspace, on two calls in a row (the second finds the first call's leftovers in the shared
static scratch), and refuse more layers than its scratch holds.

Kept in a file of its own that pytest collects last."""
import ctypes

import pytest
import torch

import gqa_attention_long_gb300 as ea
from gqa_attention_long_gb300 import _lib
from gqa_attention_long_gb300.inputs import layer_inputs
from tests._gpu_util import assert_close, check_status, f64, to_dev

pytestmark = pytest.mark.gpu

MAX_LAYERS = 4  # EA_NOALLOC_MAX_LAYERS in include/expert_attn.h


def _noalloc():
    f = ea.lib().expert_attn_layers_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(_lib.EaLayerArgs), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return f


def _run_both(seed0, n, S, Smax):
    xs = [layer_inputs(seed0 + l, S, Smax) for l in range(n)]
    ref = [to_dev(x) for x in xs]
    ws = ea.alloc_workspace(n, Smax)
    ea.expert_attn_layers(ref, S, Smax, 0, ea.EA_KV_BF16, ws)
    got = [to_dev(x) for x in xs]
    arr = ea.make_args(got, Smax, ea.EA_KV_BF16)
    rc = _noalloc()(arr, n, S, Smax, 0, ea.EA_KV_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ea.expert_attn_status_string(rc)
    torch.cuda.synchronize()
    check_status(ws)
    return ref, got


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    # call 1: four layers; call 2: two layers of another shape over the same static scratch
    for seed0, n, S, Smax in [(700, MAX_LAYERS, 4700, 8192), (800, 2, 333, 512)]:
        ref, got = _run_both(seed0, n, S, Smax)
        for a, b in zip(ref, got):
            assert torch.isfinite(b.out.float()).all()
            assert_close(f64(b.out), f64(a.out), f"noalloc vs workspace path, S={S}")
            assert torch.equal(b.k_cache, a.k_cache) and torch.equal(b.v_cache, a.v_cache)


def test_noalloc_refuses_more_layers_than_its_scratch_holds():
    xs = [layer_inputs(900 + l, 10, 128) for l in range(MAX_LAYERS + 1)]
    Ls = [to_dev(x) for x in xs]
    before = [L.out.clone() for L in Ls]
    arr = ea.make_args(Ls, 128, ea.EA_KV_BF16)
    rc = _noalloc()(arr, MAX_LAYERS + 1, 10, 128, 0, ea.EA_KV_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == 4  # EA_ERR_WORKSPACE: nothing launched
    torch.cuda.synchronize()
    for L, b in zip(Ls, before):
        assert torch.equal(L.out.view(torch.int16), b.view(torch.int16))
