"""Sequential chain of dependent layers (layer i+1's raw q is layer i's output, a stand-in for
the wo/MLP between layers): one expert_attn_layer call per layer, issued directly and replayed
from a CUDA graph. Every layer's output is checked against the oracle run on that layer's own
inputs (its raw q being the previous layer's bf16 output), and the graph replay reproduces the
direct calls bit for bit."""
import numpy as np
import pytest
import torch

import gqa_attention_long_gb300 as ea
from gqa_attention_long_gb300.inputs import layer_inputs
from tests._gpu_util import assert_close, check_status, f64, oracle_layer, to_dev

pytestmark = pytest.mark.gpu


def _chain(S, Smax, n_layers, seed0):
    xs = [layer_inputs(seed0 + l, S, Smax) for l in range(n_layers)]
    Ls = [to_dev(x) for x in xs]
    for l in range(1, n_layers):  # layer l reads layer l-1's output as its raw q
        Ls[l] = ea.LayerBuffers(q_raw=Ls[l - 1].out, k_raw=Ls[l].k_raw, v_raw=Ls[l].v_raw,
                                q_gamma=Ls[l].q_gamma, k_gamma=Ls[l].k_gamma, k_cache=Ls[l].k_cache,
                                v_cache=Ls[l].v_cache, out=Ls[l].out)
    return xs, Ls


@pytest.mark.parametrize("S,Smax", [(256, 512), (4700, 8192)])
def test_chain_matches_oracle_layer_by_layer(S, Smax):
    n = 4
    xs, Ls = _chain(S, Smax, n, 7000)
    ws = ea.alloc_workspace(1, Smax)
    ea.expert_attn_workspace_init(ws)
    for L in Ls:
        ea.expert_attn_layer(L, S, Smax, 0, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    check_status(ws)
    for l in range(n):
        x = xs[l]
        if l > 0:  # the oracle sees exactly what the GPU layer read
            x.q_raw = Ls[l - 1].out.detach().cpu()
        assert_close(f64(Ls[l].out), oracle_layer(x)["out"], f"layer {l}")


def test_chain_graph_replay_is_bitwise_identical():
    S, Smax, n = 300, 512, 6
    xs, Ls = _chain(S, Smax, n, 7100)
    ws = ea.alloc_workspace(1, Smax)
    ea.expert_attn_workspace_init(ws)
    arrs = [ea.make_args([L], Smax, ea.EA_KV_BF16) for L in Ls]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for L, a in zip(Ls, arrs):
            ea.expert_attn_layers([L], S, Smax, 0, ea.EA_KV_BF16, ws, side, _arr=a)
    torch.cuda.synchronize()
    check_status(ws)
    direct = [L.out.clone() for L in Ls]
    for L in Ls:
        L.out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for L, a in zip(Ls, arrs):
            ea.expert_attn_layers([L], S, Smax, 0, ea.EA_KV_BF16, ws, side, _arr=a)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    check_status(ws)
    for l in range(n):
        assert torch.equal(Ls[l].out, direct[l]), f"layer {l}"
