"""The algorithmic byte counts behind bench.py's roofline fractions, recounted from the tensors
a call touches (CPU only): each count is rebuilt from the inputs' own shapes and dtypes, so a
dropped or doubled term in bench.py's closed forms fails here."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from gqa_attention_long_gb300.inputs import (  # noqa: E402
    decode_inputs, expert_layer_weights, layer_inputs, residual_stream)


def _row_bytes(cache: torch.Tensor) -> int:
    """Bytes of one cache row of one head."""
    return cache.shape[-1] * cache.element_size()


def _attention_layer_bytes(x, row_bytes: int) -> int:
    heads = x.k_cache.shape[0]
    live = 2 * heads * x.S * row_bytes                 # K and V cache rows [0, S) read
    own = 2 * 2 * heads * 64 * row_bytes               # own K and V rows written, then read back
    raw = x.q_raw.nbytes + x.k_raw.nbytes + x.v_raw.nbytes
    out = x.q_raw.nbytes                               # the output has q's shape and dtype
    return live + own + raw + out


@pytest.mark.parametrize("S,Smax", [(4700, 8192), (1024, 8192), (0, 256), (300, 512)])
def test_attention_bytes_per_layer(S, Smax):
    x = layer_inputs(1, S, Smax)
    assert bench.algo_bytes_per_layer(S) == _attention_layer_bytes(x, _row_bytes(x.k_cache))
    # e4m3 cache: one byte per K/V element, the rest unchanged (block scales left out)
    assert bench.algo_bytes_per_layer_fp8(S) == _attention_layer_bytes(x, x.k_cache.shape[-1])


def test_attention_bytes_of_the_benchmarked_step():
    # 64 layers at S = 4700: the figure the roofline line divides by the kernel's time
    assert 64 * bench.algo_bytes_per_layer(4700) == 1_315_962_880


@pytest.mark.parametrize("hidden,inter", [(1536, 6144), (256, 384)])
def test_decoder_layer_bytes(hidden, inter):
    S, Smax = 4700, 8192
    w = expert_layer_weights(2, hidden=hidden, inter=inter)
    weights = sum(t.nbytes for t in w.__dict__.values())
    x = layer_inputs(2, S, Smax)
    cache = 2 * 8 * S * _row_bytes(x.k_cache) + 2 * 2 * 8 * 64 * _row_bytes(x.k_cache)
    resid = residual_stream(2, hidden=hidden).nbytes
    assert bench.layer_bytes(S, hidden, inter) == weights + cache + 2 * resid  # read, written


@pytest.mark.parametrize("pos", [0, 1, 4700, 8190])
def test_decode_bytes_per_layer(pos):
    d = decode_inputs(3, pos, 8192)
    rb = _row_bytes(d.k_cache)
    heads = d.k_cache.shape[0]
    cache_read = 2 * heads * (pos + 1) * rb          # rows 0..pos of K and V (row pos after its write)
    new_rows = 2 * heads * rb                          # the new K and V rows written
    raw = d.q_raw.nbytes + d.k_raw.nbytes + d.v_raw.nbytes
    out = d.q_raw.nbytes
    assert bench.decode_bytes_per_layer(pos) == cache_read + new_rows + raw + out
