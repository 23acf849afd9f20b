"""GPU parity of the MXFP4 cache producer (expert_attn_quantize_cache_mxfp4) against the oracle's
quantiser, through the C ABI: E2M1 codes and block exponents bit-exact, rows >= n_rows
untouched."""
import numpy as np
import pytest
import torch

import gqa_attention_long_gb300 as ea
import oracle

pytestmark = pytest.mark.gpu


def _cache(seed, Smax):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((8, Smax, 128)) * np.exp2(rng.integers(-20, 20, (8, Smax, 4))).repeat(32, -1)
    x[0, 3, :32] = 0.0                                   # an all-zero block
    x[1, 5, 32:64] = rng.standard_normal(32) * 2.0 ** -130  # bf16 subnormals: exponent clamped
    x[2, 7, 64:96] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4) * 2.0 ** -3  # ties
    x[3, 9, :] = -0.0                                     # negative zeros
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("n_rows,Smax", [(1, 64), (77, 128), (512, 512), (4700, 8192)])
def test_mxfp4_quantiser_bit_exact(n_rows, Smax):
    x = _cache(n_rows, Smax)
    d = torch.device("cuda")
    codes = torch.full((8, Smax, 64), 0xAB, dtype=torch.uint8, device=d)
    scales = torch.full((8, Smax, 4), 0xCD, dtype=torch.uint8, device=d)
    ea.expert_attn_quantize_cache_mxfp4(x.to(d), n_rows, Smax, codes, scales)
    torch.cuda.synchronize()
    cg, sg = codes.cpu().numpy(), scales.cpu().numpy()
    want_c, want_e = oracle.quantize_rows(x[:, :n_rows].float().numpy())
    got_c = np.stack([cg[:, :n_rows] & 15, cg[:, :n_rows] >> 4], -1).reshape(8, n_rows, 128)
    assert np.array_equal(got_c, want_c)
    assert np.array_equal(sg[:, :n_rows].astype(np.int16) - 127, want_e)
    assert np.all(cg[:, n_rows:] == 0xAB) and np.all(sg[:, n_rows:] == 0xCD)
