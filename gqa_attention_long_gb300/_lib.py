"""ctypes binding of libexpert_attn.so (argument marshalling only; every step runs in the
library's CUDA kernels). Function names match the C ABI in include/expert_attn.h.

Tensors must be CUDA tensors, contiguous, with the dtypes and shapes of the C ABI; the binding
checks this before passing raw device pointers, so a host tensor can never reach a kernel.
There is no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libexpert_attn.so")

EA_OK, EA_ERR_INVALID_ARG, EA_ERR_MISALIGNED, EA_ERR_UNSUPPORTED = 0, 1, 2, 3
EA_ERR_WORKSPACE, EA_ERR_CUDA, EA_ERR_TIMEOUT = 4, 5, 6
EA_KV_BF16, EA_KV_FP8_E4M3 = 0, 1


class EaLayerArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "q_raw", "k_raw", "v_raw", "q_gamma", "k_gamma", "k_cache", "v_cache",
        "k_scale", "v_scale", "out", "q_rope")]


class EaDecoderLayerArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_out", ctypes.c_void_p), ("hidden", ctypes.c_int),
                ("inter", ctypes.c_int)] + [(n, ctypes.c_void_p) for n in (
                    "ln1", "wqkv", "q_norm", "k_norm", "wo", "ln2", "w1", "w3", "w2",
                    "k_cache", "v_cache", "q_rope")]


class EaDecodeArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "q_raw", "k_raw", "v_raw", "q_gamma", "k_gamma", "k_cache", "v_cache", "out")]


_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m gqa_attention_long_gb300.build` (needs nvcc 13)")
        h = ctypes.CDLL(LIB_PATH)
        P, I, S, V = ctypes.POINTER(EaLayerArgs), ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        sig = {
            "expert_attn_workspace_size": (S, [I, I, I]),
            "expert_attn_workspace_init": (I, [V, S, V]),
            "expert_attn_prologue": (I, [P, I, I, I, I, V, S, V]),
            "expert_attn_layer": (I, [P, I, I, I, I, V, S, V]),
            "expert_attn_layers": (I, [P, I, I, I, I, I, V, S, V]),
            "expert_attn_layers_profiled": (I, [P, I, I, I, I, I, V, S, V, ctypes.POINTER(V)]),
            "expert_attn_quantize_cache": (I, [V, I, I, V, V, V]),
            "expert_attn_quantize_cache_mxfp4": (I, [V, I, I, V, V, V]),
            "expert_attn_set_splits": (I, [I]),
            "expert_attn_read_status": (I, [V, V, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_uint32)]),
            "expert_attn_status_string": (ctypes.c_char_p, [I]),
            "expert_attn_selftest_wait_timeout": (I, [I, V, S, V]),
            "expert_decoder_layer_workspace_size": (S, [I, I]),
            "expert_decoder_layer": (I, [ctypes.POINTER(EaDecoderLayerArgs), I, I, I, V, S, V]),
            "expert_linear64_workspace_size": (S, [I, I]),
            "expert_linear64": (I, [V, V, V, I, I, V, S, V]),
            "text_decode_workspace_size": (S, [I]),
            "text_decode_workspace_init": (I, [V, S, V]),
            "text_decode_attention": (I, [ctypes.POINTER(EaDecodeArgs), I, I, I, I, V, S, V]),
        }
        for name, (res, args) in sig.items():
            f = getattr(h, name)
            f.restype, f.argtypes = res, args
        _lib_handle = h
    return _lib_handle


class ExpertAttnError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        self.rc = rc
        super().__init__(f"{fn}: {expert_attn_status_string(rc)}")


def _check(fn: str, rc: int) -> None:
    if rc != EA_OK:
        raise ExpertAttnError(fn, rc)


def _ptr(t: torch.Tensor | None, name: str, dtype=None, numel=None) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class LayerBuffers:
    """One layer's device tensors (see include/expert_attn.h for shapes and dtypes)."""
    q_raw: torch.Tensor
    k_raw: torch.Tensor
    v_raw: torch.Tensor
    q_gamma: torch.Tensor
    k_gamma: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    out: torch.Tensor
    k_scale: torch.Tensor | None = None
    v_scale: torch.Tensor | None = None
    q_rope: torch.Tensor | None = None


def _args(layers: list[LayerBuffers], Smax: int, kv_dtype: int):
    arr = (EaLayerArgs * len(layers))()
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    cache_dt = bf if kv_dtype == EA_KV_BF16 else (u8, torch.float8_e4m3fn)
    for i, L in enumerate(layers):
        a = arr[i]
        a.q_raw = _ptr(L.q_raw, "q_raw", bf, 16 * 64 * 128)
        a.k_raw = _ptr(L.k_raw, "k_raw", bf, 8 * 64 * 128)
        a.v_raw = _ptr(L.v_raw, "v_raw", bf, 8 * 64 * 128)
        a.q_gamma = _ptr(L.q_gamma, "q_gamma", bf, 128)
        a.k_gamma = _ptr(L.k_gamma, "k_gamma", bf, 128)
        a.k_cache = _ptr(L.k_cache, "k_cache", cache_dt, 8 * Smax * 128)
        a.v_cache = _ptr(L.v_cache, "v_cache", cache_dt, 8 * Smax * 128)
        a.out = _ptr(L.out, "out", bf, 16 * 64 * 128)
        a.q_rope = _ptr(L.q_rope, "q_rope", bf, 16 * 64 * 128)
        if kv_dtype == EA_KV_FP8_E4M3:
            n_sc = 8 * (Smax // 128 + 1)
            a.k_scale = _ptr(L.k_scale, "k_scale", f32, n_sc)
            a.v_scale = _ptr(L.v_scale, "v_scale", f32, n_sc)
    return arr


def _ws(ws: torch.Tensor) -> tuple[int, int]:
    return _ptr(ws, "workspace", torch.uint8), ws.numel()


# ------------------------------------------------------------------------------ public API
def expert_attn_status_string(rc: int) -> str:
    return lib().expert_attn_status_string(int(rc)).decode()


def expert_attn_workspace_size(n_layers: int, Smax: int, kv_dtype: int = EA_KV_BF16) -> int:
    return int(lib().expert_attn_workspace_size(n_layers, Smax, kv_dtype))


def expert_attn_workspace_init(ws: torch.Tensor, stream=None) -> None:
    p, n = _ws(ws)
    _check("expert_attn_workspace_init", lib().expert_attn_workspace_init(p, n, _stream(stream)))


def alloc_workspace(n_layers: int, Smax: int, kv_dtype: int = EA_KV_BF16, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace of the size the library asks for (torch-allocated)."""
    n = expert_attn_workspace_size(n_layers, Smax, kv_dtype)
    if n == 0:
        raise RuntimeError("expert_attn_workspace_size returned 0: no sm_103 GPU available")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    expert_attn_workspace_init(ws)
    return ws


def expert_attn_prologue(layer: LayerBuffers, S: int, Smax: int, rope_delta: int, kv_dtype: int,
                         ws: torch.Tensor, stream=None) -> None:
    arr = _args([layer], Smax, kv_dtype)
    p, n = _ws(ws)
    _check("expert_attn_prologue", lib().expert_attn_prologue(arr, S, Smax, rope_delta, kv_dtype, p, n,
                                                              _stream(stream)))


def expert_attn_layer(layer: LayerBuffers, S: int, Smax: int, rope_delta: int, kv_dtype: int,
                      ws: torch.Tensor, stream=None) -> None:
    arr = _args([layer], Smax, kv_dtype)
    p, n = _ws(ws)
    _check("expert_attn_layer", lib().expert_attn_layer(arr, S, Smax, rope_delta, kv_dtype, p, n,
                                                        _stream(stream)))


def expert_attn_layers(layers: list[LayerBuffers], S: int, Smax: int, rope_delta: int, kv_dtype: int,
                       ws: torch.Tensor, stream=None, _arr=None) -> None:
    arr = _arr if _arr is not None else _args(layers, Smax, kv_dtype)
    p, n = _ws(ws)
    _check("expert_attn_layers", lib().expert_attn_layers(arr, len(arr), S, Smax, rope_delta, kv_dtype,
                                                          p, n, _stream(stream)))


def expert_attn_layers_profiled(layers: list[LayerBuffers], S: int, Smax: int, rope_delta: int,
                                kv_dtype: int, ws: torch.Tensor, events, stream=None, _arr=None) -> None:
    arr = _arr if _arr is not None else _args(layers, Smax, kv_dtype)
    p, n = _ws(ws)
    ev = (ctypes.c_void_p * 4)(*[None if e is None else e.cuda_event for e in events])
    _check("expert_attn_layers_profiled", lib().expert_attn_layers_profiled(
        arr, len(arr), S, Smax, rope_delta, kv_dtype, p, n, _stream(stream), ev))


def make_args(layers: list[LayerBuffers], Smax: int, kv_dtype: int):
    """Pre-marshalled argument array, to keep per-call Python work out of timing loops."""
    return _args(layers, Smax, kv_dtype)


def expert_attn_quantize_cache(src: torch.Tensor, n_rows: int, Smax: int, dst: torch.Tensor,
                               scales: torch.Tensor, stream=None) -> None:
    _check("expert_attn_quantize_cache", lib().expert_attn_quantize_cache(
        _ptr(src, "src", torch.bfloat16, 8 * Smax * 128), n_rows, Smax,
        _ptr(dst, "dst", (torch.uint8, torch.float8_e4m3fn), 8 * Smax * 128),
        _ptr(scales, "scales", torch.float32, 8 * (Smax // 128 + 1)), _stream(stream)))


def expert_attn_quantize_cache_mxfp4(src: torch.Tensor, n_rows: int, Smax: int, codes: torch.Tensor,
                                     scales: torch.Tensor, stream=None) -> None:
    """MXFP4 cache producer: rows [0, n_rows) of a bf16 cache [8, Smax, 128] into packed E2M1
    codes uint8 [8, Smax, 64] and block exponents uint8 [8, Smax, 4] (e + 127)."""
    _check("expert_attn_quantize_cache_mxfp4", lib().expert_attn_quantize_cache_mxfp4(
        _ptr(src, "src", torch.bfloat16, 8 * Smax * 128), n_rows, Smax,
        _ptr(codes, "codes", torch.uint8, 8 * Smax * 64),
        _ptr(scales, "scales", torch.uint8, 8 * Smax * 4), _stream(stream)))


def split_units(n_layers: int, S: int, n_ctas: int) -> list[int]:
    """Units (layer * 8 + kv head) whose key tiles the attention kernel's partition cuts between
    CTAs, i.e. the units the attention kernel merges; the same plan the library makes for a chunk
    of n_layers (<= 64) layers on n_ctas persistent CTAs (capped by the number of key tiles).
    Host-side planning only (no GPU): used to count launches and by tests."""
    T = (S + 127) // 128 + 1
    W = n_layers * 8 * T
    n = max(1, min(n_ctas, 257, W))
    units: list[int] = []
    for b in range(1, n):
        tb = b * W // n
        if tb % T and (not units or units[-1] != tb // T):
            units.append(tb // T)
    return units


def split_parts(n_layers: int, S: int, n_ctas: int) -> list[tuple[int, int]]:
    """split_units with each unit's number of parts (the CTAs whose tile range meets it)."""
    T = (S + 127) // 128 + 1
    W = n_layers * 8 * T
    n = max(1, min(n_ctas, 257, W))

    def cta_of_tile(x: int) -> int:
        c = x * n // W
        while c + 1 < n and (c + 1) * W // n <= x:
            c += 1
        while c > 0 and c * W // n > x:
            c -= 1
        return c

    return [(u, cta_of_tile(u * T + T - 1) - cta_of_tile(u * T) + 1)
            for u in split_units(n_layers, S, n_ctas)]


def kernels_per_call(n_layers: int, S: int, n_ctas: int, kv_dtype: int = EA_KV_BF16) -> int:
    """Kernels one expert_attn_layers call launches: per chunk of 64 layers the prologue kernel
    (e4m3 cache only; the bf16 attention kernel does its own prologue) and the attention kernel,
    which also merges the units that its CTA partition splits."""
    total = 0
    for l0 in range(0, n_layers, 64):
        total += (1 if kv_dtype == EA_KV_FP8_E4M3 else 0) + 1
    return total


def expert_attn_set_splits(n_ctas_or_0_for_auto: int) -> int:
    return int(lib().expert_attn_set_splits(int(n_ctas_or_0_for_auto)))


def expert_attn_selftest_wait_timeout(limit_us: int, ws: torch.Tensor, stream=None) -> None:
    """Launches the library's bounded-wait self-test: a kernel wait that nothing satisfies
    gives up after limit_us and records a timeout in the workspace's status word."""
    p, n = _ws(ws)
    _check("expert_attn_selftest_wait_timeout",
           lib().expert_attn_selftest_wait_timeout(int(limit_us), p, n, _stream(stream)))


def expert_attn_read_status(ws: torch.Tensor, stream=None) -> tuple[int, int]:
    st = ctypes.c_int(-1)
    bits = ctypes.c_uint32(0)
    _check("expert_attn_read_status", lib().expert_attn_read_status(
        _ptr(ws, "workspace", torch.uint8), _stream(stream), ctypes.byref(st), ctypes.byref(bits)))
    return st.value, bits.value


# ----------------------------------------------------------------- whole decoder layer
def expert_decoder_layer_workspace_size(hidden: int, inter: int) -> int:
    return int(lib().expert_decoder_layer_workspace_size(int(hidden), int(inter)))


def alloc_decoder_layer_workspace(hidden: int, inter: int, device="cuda") -> torch.Tensor:
    """A cleared workspace for expert_decoder_layer (torch-allocated)."""
    n = expert_decoder_layer_workspace_size(hidden, inter)
    if n == 0:
        raise RuntimeError("expert_decoder_layer_workspace_size returned 0 (bad widths or no sm_103 GPU)")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    expert_attn_workspace_init(ws)
    return ws


def expert_decoder_layer(x: torch.Tensor, x_out: torch.Tensor, w, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, S: int, Smax: int, rope_delta: int,
                         ws: torch.Tensor, q_rope: torch.Tensor | None = None, stream=None) -> None:
    """One decoder layer (include/expert_attn.h): ``w`` has the bf16 tensors ln1, wqkv, q_norm,
    k_norm, wo, ln2, w1, w3, w2 ([out_features, in_features] for the projections)."""
    bf = torch.bfloat16
    hidden, inter = x.shape[-1], w.w1.shape[0]
    a = EaDecoderLayerArgs()
    a.x = _ptr(x, "x", bf, 64 * hidden)
    a.x_out = _ptr(x_out, "x_out", bf, 64 * hidden)
    a.hidden, a.inter = int(hidden), int(inter)
    a.ln1 = _ptr(w.ln1, "ln1", bf, hidden)
    a.wqkv = _ptr(w.wqkv, "wqkv", bf, 4096 * hidden)
    a.q_norm = _ptr(w.q_norm, "q_norm", bf, 128)
    a.k_norm = _ptr(w.k_norm, "k_norm", bf, 128)
    a.wo = _ptr(w.wo, "wo", bf, hidden * 2048)
    a.ln2 = _ptr(w.ln2, "ln2", bf, hidden)
    a.w1 = _ptr(w.w1, "w1", bf, inter * hidden)
    a.w3 = _ptr(w.w3, "w3", bf, inter * hidden)
    a.w2 = _ptr(w.w2, "w2", bf, hidden * inter)
    a.k_cache = _ptr(k_cache, "k_cache", bf, 8 * Smax * 128)
    a.v_cache = _ptr(v_cache, "v_cache", bf, 8 * Smax * 128)
    a.q_rope = _ptr(q_rope, "q_rope", bf, 16 * 64 * 128)
    p, n = _ws(ws)
    _check("expert_decoder_layer", lib().expert_decoder_layer(ctypes.byref(a), S, Smax, rope_delta, p, n,
                                                              _stream(stream)))


def expert_linear64_workspace_size(K: int, N: int) -> int:
    return int(lib().expert_linear64_workspace_size(int(K), int(N)))


def expert_linear64(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """y[64][N] = x[64][K] w^T (bf16, fp32 accumulation) on the tensor cores."""
    bf = torch.bfloat16
    N, K = w.shape
    p, n = _ws(ws)
    _check("expert_linear64", lib().expert_linear64(_ptr(x, "x", bf, 64 * K), _ptr(w, "w", bf, N * K),
                                                    _ptr(y, "y", bf, 64 * N), int(K), int(N), p, n,
                                                    _stream(stream)))


# --------------------------------------------------------------- text-model decode attention
@dataclass
class DecodeBuffers:
    """One layer's device tensors for text_decode_attention (include/expert_attn.h)."""
    q_raw: torch.Tensor    # bf16 [64, 128]
    k_raw: torch.Tensor    # bf16 [8, 128]
    v_raw: torch.Tensor    # bf16 [8, 128]
    q_gamma: torch.Tensor  # bf16 [128]
    k_gamma: torch.Tensor  # bf16 [128]
    k_cache: torch.Tensor  # bf16 [8, Smax, 128]
    v_cache: torch.Tensor
    out: torch.Tensor      # bf16 [64, 128]


def make_decode_args(layers: list[DecodeBuffers], Smax: int):
    arr = (EaDecodeArgs * len(layers))()
    bf = torch.bfloat16
    for i, L in enumerate(layers):
        a = arr[i]
        a.q_raw = _ptr(L.q_raw, "q_raw", bf, 64 * 128)
        a.k_raw = _ptr(L.k_raw, "k_raw", bf, 8 * 128)
        a.v_raw = _ptr(L.v_raw, "v_raw", bf, 8 * 128)
        a.q_gamma = _ptr(L.q_gamma, "q_gamma", bf, 128)
        a.k_gamma = _ptr(L.k_gamma, "k_gamma", bf, 128)
        a.k_cache = _ptr(L.k_cache, "k_cache", bf, 8 * Smax * 128)
        a.v_cache = _ptr(L.v_cache, "v_cache", bf, 8 * Smax * 128)
        a.out = _ptr(L.out, "out", bf, 64 * 128)
    return arr


def text_decode_workspace_size(n_layers: int) -> int:
    return int(lib().text_decode_workspace_size(int(n_layers)))


def text_decode_workspace_init(ws: torch.Tensor, stream=None) -> None:
    p, n = _ws(ws)
    _check("text_decode_workspace_init", lib().text_decode_workspace_init(p, n, _stream(stream)))


def alloc_decode_workspace(n_layers: int, device="cuda") -> torch.Tensor:
    """A cleared workspace for text_decode_attention (torch-allocated)."""
    n = text_decode_workspace_size(n_layers)
    if n == 0:
        raise RuntimeError("text_decode_workspace_size returned 0: no sm_103 GPU available")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    text_decode_workspace_init(ws)
    return ws


def text_decode_attention(layers: list[DecodeBuffers], pos: int, Smax: int, rope_delta: int,
                          ws: torch.Tensor, stream=None, _arr=None) -> None:
    arr = _arr if _arr is not None else make_decode_args(layers, Smax)
    p, n = _ws(ws)
    _check("text_decode_attention", lib().text_decode_attention(arr, len(arr), int(pos), int(Smax),
                                                                int(rope_delta), p, n, _stream(stream)))
