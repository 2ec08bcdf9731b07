"""GPU parity of nc_w8a8_gemv_b32 (int8 weights per row, activations in
blocks of 32) against the quantisation oracle (oracle/quant.py), through the
C ABI: codes, block scales and per-block int32 sums bit for bit, the fp32
output within the stage tolerance."""
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


def _inputs(B, K, N, seed):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn(N, K, generator=g) * 0.02).numpy().astype(np.float32)
    wq, sw = quant.quantize_rows_i8(W)
    x = torch.randn(B, K, generator=g).float()
    x[:, 7] *= 68.0  # one outlier per row: it widens only its own block
    return wq, sw, x


@pytest.mark.parametrize("B,K,N,bias", [
    (1, 896, 1152, True),    # 0.5B QKV
    (1, 4864, 896, False),   # 0.5B down
    (4, 896, 300, True),
    (8, 4864, 64, False),    # the largest batch
    (3, 96, 17, True),       # three blocks, ragged rows
])
def test_b32_bit_exact_without_norm(B, K, N, bias):
    wq, sw, x = _inputs(B, K, N, seed=K + N)
    b16 = synth.normal_bf16(0, 611, (N,), 0.02) if bias else None
    y, check = guarded(B * N)
    nb = K // 32
    xq = torch.empty(B, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(B, nb, device="cuda")
    acc = torch.empty(B, N, nb, dtype=torch.int32, device="cuda")
    nc.w8a8_gemv_b32(x.cuda(), None, 0.0, torch.from_numpy(wq).cuda(), torch.from_numpy(sw).cuda(),
                     None if b16 is None else b16.cuda(), y.view(B, N), xq, sx, acc)
    torch.cuda.synchronize()
    check()
    bias_f = None if b16 is None else b16.float().numpy()
    for r in range(B):
        ref, q_o, s_o, acc_o = quant.linear_w8a8_blocked(wq, sw, bias_f, x[r].numpy())
        assert np.array_equal(xq[r].cpu().numpy(), q_o)
        assert np.array_equal(sx[r].cpu().numpy().view(np.uint32), s_o.view(np.uint32))
        assert np.array_equal(acc[r].cpu().numpy(), acc_o)
        assert rel_l2(y.view(B, N)[r].cpu().numpy(), ref) < 5e-5


def test_b32_with_norm_is_the_blocked_product_of_its_own_codes():
    """With the RMSNorm prologue the kernel's normed values can differ from the
    oracle's in the last bit, so a code may land on the other side of a
    rounding boundary. The product of the kernel's own codes and scales must
    still be exact, and the codes must agree with the oracle's almost
    everywhere."""
    B, K, N = 2, 4864, 300
    wq, sw, x = _inputs(B, K, N, seed=77)
    gamma = synth.normal_bf16(0, 612, (K,), 0.02, 1.0)
    y = torch.empty(B, N, device="cuda")
    xq = torch.empty(B, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(B, K // 32, device="cuda")
    acc = torch.empty(B, N, K // 32, dtype=torch.int32, device="cuda")
    nc.w8a8_gemv_b32(x.cuda(), gamma.cuda(), 1e-6, torch.from_numpy(wq).cuda(),
                     torch.from_numpy(sw).cuda(), None, y, xq, sx, acc)
    torch.cuda.synchronize()
    for r in range(B):
        q_k = xq[r].cpu().numpy()
        acc_o = quant.matvec_i8_blocked(wq, q_k)
        assert np.array_equal(acc[r].cpu().numpy(), acc_o)
        xn = oracle.rmsnorm(x[r].numpy(), gamma, 1e-6)
        q_o, _ = quant.quantize_blocks_i8(xn)
        assert (q_k != q_o).sum() <= K // 1000 + 1
        yk = [sum(float(acc_o[n, j]) * float(sw[n]) * float(sx[r, j]) for j in range(K // 32))
              for n in range(N)]
        assert rel_l2(y[r].cpu().numpy(), yk) < 5e-5
