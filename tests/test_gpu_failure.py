"""Failure detection on the GPU without a fault: a kernel wait that nothing satisfies gives up
after its time limit, records a timeout in the workspace's status word (which the host reads
as EA_ERR_TIMEOUT), and the CUDA context stays usable for the next call."""
import time

import pytest
import torch

import gqa_attention_long_gb300 as ea
from tests._gpu_util import assert_close, check_status, f64, oracle_layer, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    ws = ea.alloc_workspace(1, 512)
    ea.expert_attn_workspace_init(ws)
    t0 = time.perf_counter()
    ea.expert_attn_selftest_wait_timeout(50_000, ws)  # 50 ms
    st, bits = ea.expert_attn_read_status(ws)
    dt = time.perf_counter() - t0
    assert st == ea._lib.EA_ERR_TIMEOUT and bits != 0
    assert 0.04 < dt < 10.0  # it waited about the limit, then returned


def test_context_usable_after_timeout():
    from gqa_attention_long_gb300.inputs import layer_inputs
    ws = ea.alloc_workspace(1, 512)
    ea.expert_attn_workspace_init(ws)
    ea.expert_attn_selftest_wait_timeout(20_000, ws)
    assert ea.expert_attn_read_status(ws)[0] == ea._lib.EA_ERR_TIMEOUT
    # a fresh status word, then a normal layer: correct output, clean status
    ea.expert_attn_workspace_init(ws)
    x = layer_inputs(0, 256, 512)
    L = to_dev(x)
    ea.expert_attn_layer(L, 256, 512, 0, ea.EA_KV_BF16, ws)
    torch.cuda.synchronize()
    check_status(ws)
    assert_close(f64(L.out), oracle_layer(x)["out"])
