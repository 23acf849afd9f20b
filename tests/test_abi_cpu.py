"""The C-ABI library loads, exports every function include/expert_attn.h declares, and rejects
bad arguments on the host before any CUDA work (runs without a GPU)."""
import ctypes
import os
import re

import pytest

import gqa_attention_long_gb300 as ea
from gqa_attention_long_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "expert_attn.h")


@pytest.fixture(scope="module")
def h():
    if not os.path.exists(_lib.LIB_PATH):
        from gqa_attention_long_gb300 import build
        build.build()
    return ea.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**((?:expert|text)_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("expert_attn_prologue", "expert_attn_layer", "expert_attn_layers",
              "expert_attn_workspace_size", "expert_attn_status_string", "expert_decoder_layer",
              "expert_decoder_layer_workspace_size", "expert_linear64", "text_decode_attention",
              "text_decode_workspace_size", "text_decode_workspace_init"):
        assert n in names


def test_every_declared_symbol_is_exported(h):
    for n in declared_functions():
        assert hasattr(h, n), n


def test_status_strings(h):
    for rc in range(7):
        assert ea.expert_attn_status_string(rc).startswith("EA_")
    assert ea.expert_attn_status_string(99) == "unknown status"


def _args(**over):
    a = (_lib.EaLayerArgs * 1)()
    for n, _ in _lib.EaLayerArgs._fields_:
        setattr(a[0], n, 0x10000)  # aligned fake device pointers: never dereferenced by validation
    a[0].k_scale = a[0].v_scale = a[0].q_rope = None
    for k, v in over.items():
        setattr(a[0], k, v)
    return a


@pytest.mark.parametrize("S,Smax,dt,rc", [
    (449, 512, 0, _lib.EA_ERR_INVALID_ARG),    # S > Smax - 64
    (-1, 512, 0, _lib.EA_ERR_INVALID_ARG),
    (10, 500, 0, _lib.EA_ERR_INVALID_ARG),     # Smax not a multiple of 64
    (10, 576, 1, _lib.EA_ERR_INVALID_ARG),     # FP8 needs Smax % 128 == 0 (and scales)
    (10, 512, 7, _lib.EA_ERR_INVALID_ARG),     # unknown dtype
])
def test_bad_sizes_rejected(h, S, Smax, dt, rc):
    assert h.expert_attn_layer(_args(), S, Smax, 0, dt, ctypes.c_void_p(0x100000), 1 << 30, None) == rc


def test_null_and_misaligned_pointers_rejected(h):
    ws = ctypes.c_void_p(0x100000)
    assert h.expert_attn_layer(_args(q_raw=None), 10, 512, 0, 0, ws, 1 << 30, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_attn_layer(_args(k_cache=0x10008), 10, 512, 0, 0, ws, 1 << 30, None) == _lib.EA_ERR_MISALIGNED
    assert h.expert_attn_layer(_args(), 10, 512, 0, 0, ctypes.c_void_p(0x100010), 1 << 30, None) == _lib.EA_ERR_MISALIGNED
    assert h.expert_attn_layer(_args(), 10, 512, 0, 0, None, 1 << 30, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_attn_layers(_args(), 0, 10, 512, 0, 0, ws, 1 << 30, None) == _lib.EA_ERR_INVALID_ARG
    # positions beyond fp32-exact integers are refused
    assert h.expert_attn_layer(_args(), 10, 512, 1 << 24, 0, ws, 1 << 30, None) == _lib.EA_ERR_INVALID_ARG


def test_binding_refuses_host_tensors(h):
    import torch
    t = torch.zeros(16, 64, 128, dtype=torch.bfloat16)
    L = ea.LayerBuffers(q_raw=t, k_raw=t[:8], v_raw=t[:8], q_gamma=t[0, 0], k_gamma=t[0, 0],
                        k_cache=t, v_cache=t, out=t)
    with pytest.raises(TypeError):
        ea.expert_attn_layer(L, 0, 128, 0, 0, torch.zeros(16, dtype=torch.uint8))


def test_set_splits_roundtrip(h):
    prev = ea.expert_attn_set_splits(7)
    assert ea.expert_attn_set_splits(prev) == 7


def test_selftest_rejects_bad_arguments_without_gpu(h):
    ws = ctypes.c_void_p(0x10000)
    assert h.expert_attn_selftest_wait_timeout(0, ws, 1 << 20, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_attn_selftest_wait_timeout(2000001, ws, 1 << 20, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_attn_selftest_wait_timeout(1000, None, 1 << 20, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_attn_selftest_wait_timeout(1000, ws, 16, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_attn_selftest_wait_timeout(1000, ctypes.c_void_p(0x10010), 1 << 20, None) == \
        _lib.EA_ERR_MISALIGNED


def _layer_args(**over):
    a = _lib.EaDecoderLayerArgs()
    for n, t in _lib.EaDecoderLayerArgs._fields_:
        if t is ctypes.c_void_p:
            setattr(a, n, 0x10000)
    a.x_out = 0x20000
    a.q_rope = None
    a.hidden, a.inter = 1536, 6144
    for k, v in over.items():
        setattr(a, k, v)
    return ctypes.byref(a)


def test_decoder_layer_rejects_bad_arguments_without_gpu(h):
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 30
    assert h.expert_decoder_layer(None, 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(), 10, 512, 0, None, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(hidden=1500), 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(inter=64), 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(hidden=16384), 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(w2=None), 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(wo=0x10008), 10, 512, 0, ws, big, None) == _lib.EA_ERR_MISALIGNED
    assert h.expert_decoder_layer(_layer_args(x_out=0x10000), 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_decoder_layer(_layer_args(), 10, 512, 0, ctypes.c_void_p(0x100080), big, None) == \
        _lib.EA_ERR_MISALIGNED
    assert h.expert_decoder_layer_workspace_size(1500, 6144) == 0


def test_linear64_rejects_bad_arguments_without_gpu(h):
    ws = ctypes.c_void_p(0x100000)
    p = ctypes.c_void_p(0x10000)
    big = 1 << 30
    assert h.expert_linear64(None, p, p, 64, 128, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert h.expert_linear64(p, p, p, 96, 128, ws, big, None) == _lib.EA_ERR_INVALID_ARG   # K % 64
    assert h.expert_linear64(p, p, p, 64, 192, ws, big, None) == _lib.EA_ERR_INVALID_ARG   # N % 128
    assert h.expert_linear64(ctypes.c_void_p(0x10004), p, p, 64, 128, ws, big, None) == _lib.EA_ERR_MISALIGNED
    assert h.expert_linear64_workspace_size(96, 128) == 0


def _decode_args(**over):
    a = _lib.EaDecodeArgs()
    for name, _ in _lib.EaDecodeArgs._fields_:
        setattr(a, name, over.get(name, 0x10000))
    return a


def test_decode_rejects_bad_arguments_without_gpu(h):
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 30
    f = h.text_decode_attention
    one = ctypes.byref(_decode_args())
    assert f(None, 1, 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert f(one, 0, 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG       # no layers
    assert f(one, 1, -1, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG       # pos < 0
    assert f(one, 1, 512, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG      # pos >= Smax
    assert f(one, 1, 10, 500, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG       # Smax % 64
    assert f(one, 1, 10, 512, 1 << 25, ws, big, None) == _lib.EA_ERR_INVALID_ARG  # position range
    assert f(one, 1, 10, 512, 0, None, big, None) == _lib.EA_ERR_INVALID_ARG
    assert f(one, 1, 10, 512, 0, ctypes.c_void_p(0x100080), big, None) == _lib.EA_ERR_MISALIGNED
    assert f(ctypes.byref(_decode_args(out=None)), 1, 10, 512, 0, ws, big, None) == _lib.EA_ERR_INVALID_ARG
    assert f(ctypes.byref(_decode_args(k_cache=0x10008)), 1, 10, 512, 0, ws, big, None) == \
        _lib.EA_ERR_MISALIGNED
    assert h.text_decode_workspace_size(0) == 0
    assert h.text_decode_workspace_init(None, 4096, None) == _lib.EA_ERR_INVALID_ARG


def test_mxfp4_quantiser_rejects_bad_arguments_without_gpu(h):
    p, c, s = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30001)
    f = h.expert_attn_quantize_cache_mxfp4
    assert f(None, 10, 512, c, s, None) == _lib.EA_ERR_INVALID_ARG
    assert f(p, 10, 512, None, s, None) == _lib.EA_ERR_INVALID_ARG
    assert f(p, 10, 512, c, None, None) == _lib.EA_ERR_INVALID_ARG
    assert f(p, -1, 512, c, s, None) == _lib.EA_ERR_INVALID_ARG
    assert f(p, 513, 512, c, s, None) == _lib.EA_ERR_INVALID_ARG
    assert f(p, 10, 0, c, s, None) == _lib.EA_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x10008), 10, 512, c, s, None) == _lib.EA_ERR_MISALIGNED
    assert f(p, 10, 512, ctypes.c_void_p(0x20004), s, None) == _lib.EA_ERR_MISALIGNED
