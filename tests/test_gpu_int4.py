"""GPU parity of nc_int4_gemv (group-wise INT4 weights) against the
quantisation oracle (oracle/quant.py), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from helpers import guarded, rel_l2
from oracle import quant
from transformer_decode_gb300 import nc, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nc.load()
    oracle.build()


@pytest.mark.parametrize("B,K,N,group,norm", [
    (1, 896, 1152, 32, True),     # 0.5B QKV at group 32
    (1, 896, 9728, 128, True),    # 0.5B gate|up rows at group 128
    (1, 4864, 896, 32, False),    # 0.5B down
    (3, 896, 37, 64, True),       # ragged rows, small batch
    (8, 4864, 130, 128, False),   # the largest batch and K
    (5, 96, 17, 32, True),        # one chunk per lane at most: lanes past the row idle
])
def test_int4_gemv_matches_oracle(B, K, N, group, norm):
    g = torch.Generator().manual_seed(K + N + group)
    W = (torch.randn(N, K, generator=g) * 0.02).numpy().astype(np.float32)
    W[:, 5] = 0.3  # an outlier column: its groups get large scales
    q, s = quant.quantize_int4(W, group)
    p = quant.pack_int4(q)
    x = torch.randn(B, K, generator=g).float()
    gamma = synth.normal_bf16(0, 601, (K,), 0.02, 1.0) if norm else None
    y, check = guarded(B * N)
    nc.int4_gemv(x.cuda(), None if gamma is None else gamma.cuda(), 1e-6,
                 torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda(), group, y.view(B, N))
    torch.cuda.synchronize()
    check()
    got = y.view(B, N).cpu().numpy()
    for b in range(B):
        xn = oracle.rmsnorm(x[b].numpy(), gamma, 1e-6) if norm else x[b].numpy()
        ref = quant.linear_int4(p, s, group, xn)
        assert np.isfinite(got[b]).all()
        assert rel_l2(got[b], ref) < 5e-5, (b, rel_l2(got[b], ref))


def test_int4_gemv_zero_group_and_extreme_codes():
    """A zero group (scale 0) contributes nothing; all-(+7) and all-(-7) rows
    give 7 * scale * sum(x) with the sign of the code."""
    K, N, group = 256, 4, 32
    W = np.zeros((N, K), np.float32)
    W[1] = 0.5
    W[2] = -0.5
    W[3, 64:96] = 0.25  # one nonzero group
    q, s = quant.quantize_int4(W, group)
    p = quant.pack_int4(q)
    x = torch.linspace(0.1, 1.0, K).float()[None]
    y = torch.empty(1, N, device="cuda")
    nc.int4_gemv(x.cuda(), None, 0.0, torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda(),
                 group, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy()[0]
    ref = quant.linear_int4(p, s, group, x[0].numpy())
    assert got[0] == 0.0
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-6)
    assert got[1] == -got[2] and got[1] > 0
