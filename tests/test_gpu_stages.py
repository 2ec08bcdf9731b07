"""GPU parity of each stage entry point against the CPU oracle, through the
C ABI, on seeded inputs that span several tiles and ragged tails."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import REL_L2_GATE, bf16_bits, f32, guarded, rel_l2, to_device
from transformer_decode_gb300 import nc, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nc.load()
    oracle.build()


def _x(B, K, stream, std=1.0):
    g = torch.Generator().manual_seed(1000 + stream)
    return (torch.randn(B, K, generator=g) * std).float()


def _norm_ref(x, gamma, eps):
    return np.stack([oracle.rmsnorm(x[b], gamma, eps) if gamma is not None else x[b].numpy()
                     for b in range(x.shape[0])])


# ------------------------------------------------------------------ GEMV family
@pytest.mark.parametrize("B,K,N,norm,bias", [
    (1, 896, 1152, True, True),      # 0.5B QKV
    (1, 896, 151936, True, False),   # 0.5B head-sized
    (1, 4864, 896, False, False),    # 0.5B down
    (3, 896, 37, True, True),        # ragged rows, small batch
    (16, 896, 300, True, False),     # batch 16 (tensor cores)
    (9, 896, 1152, True, True),      # batch 9, QKV-shaped (tensor cores, ragged batch)
    (16, 2048, 77, True, True),      # tensor cores at the largest single k range
    (16, 4864, 40, False, False),    # batch 16, K split into tiles
    (1, 8, 5, True, True),           # minimum K
    (1, 20000, 9, True, False),      # K beyond one shared-memory tile
    (2, 4096, 600, True, False),     # 8B hidden
])
def test_rmsnorm_gemv(B, K, N, norm, bias):
    x = _x(B, K, K + N)
    W = synth.normal_bf16(0, 500 + N, (N, K), 0.02)
    gamma = synth.normal_bf16(0, 501, (K,), 0.02, 1.0) if norm else None
    b = synth.normal_bf16(0, 502, (N,), 0.02) if bias else None
    y, check = guarded(B * N)
    nc.rmsnorm_gemv(x.cuda(), None if gamma is None else gamma.cuda(), 1e-6, W.cuda(),
                    None if b is None else b.cuda(), y.view(B, N))
    torch.cuda.synchronize()
    check()
    xn = _norm_ref(x, gamma, 1e-6)
    for r in range(B):
        ref = oracle.matvec_bf16(W, xn[r])
        if b is not None:
            ref = ref + oracle.bf16_to_f32(bf16_bits(b))
        got = f32(y.view(B, N)[r])
        assert np.isfinite(got).all()
        assert rel_l2(got, ref) < REL_L2_GATE / 10, (r, rel_l2(got, ref))


@pytest.mark.parametrize("B,K,N", [(1, 896, 896), (1, 4864, 896), (5, 896, 130), (16, 4864, 64),
                                   (16, 896, 896), (12, 4864, 896)])
def test_gemv_residual(B, K, N):
    a = _x(B, K, 7 + K)
    x0 = _x(B, N, 8 + N)
    W = synth.normal_bf16(0, 510 + K, (N, K), 0.02)
    x = x0.clone().cuda()
    nc.gemv_residual(a.cuda(), W.cuda(), x)
    torch.cuda.synchronize()
    for r in range(B):
        ref = x0[r].numpy().astype(np.float64) + oracle.matvec_bf16(W, a[r].numpy())
        assert rel_l2(f32(x[r]), ref) < REL_L2_GATE / 10


@pytest.mark.parametrize("B,K,F", [(1, 896, 4864), (2, 256, 512), (16, 896, 100), (1, 4096, 333),
                                   (16, 896, 4864), (10, 896, 37)])
def test_swiglu_gemv(B, K, F):
    x = _x(B, K, 20 + F)
    W = synth.normal_bf16(0, 520 + F, (2 * F, K), 0.02)
    gamma = synth.normal_bf16(0, 521, (K,), 0.02, 1.0)
    h, check = guarded(B * F)
    nc.swiglu_gemv(x.cuda(), gamma.cuda(), 1e-6, W.cuda(), h.view(B, F))
    torch.cuda.synchronize()
    check()
    xn = _norm_ref(x, gamma, 1e-6)
    for r in range(B):
        g = oracle.matvec_bf16(W[:F], xn[r])
        u = oracle.matvec_bf16(W[F:], xn[r])
        ref = np.array([oracle.silu(gv) for gv in g]) * u
        assert rel_l2(f32(h.view(B, F)[r]), ref) < REL_L2_GATE / 10


# ------------------------------------------------------------------ W8A8
@pytest.mark.parametrize("N,K", [(1152, 896), (96, 4864), (7, 16)])
def test_quantize_weight_bit_exact(N, K):
    W = synth.normal_bf16(0, 530 + N, (N, K), 0.02)
    W[3 % N].zero_()                         # an all-zero row gets scale 0
    q = torch.empty(N, K, dtype=torch.int8, device="cuda")
    s = torch.empty(N, dtype=torch.float32, device="cuda")
    nc.quantize_weight(W.cuda(), q, s)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_weight(W)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("B,K,N", [(1, 896, 1152), (1, 4864, 896), (4, 896, 77), (16, 4864, 33)])
def test_w8a8_gemv_bit_exact_accumulators(B, K, N):
    """On identical fp32 input (no norm) the int8 activations, their scales and
    the int32 accumulators equal the oracle's bit for bit."""
    x = _x(B, K, 40 + N)
    x[0, 5] = 0.0
    W = synth.normal_bf16(0, 540 + N, (N, K), 0.02)
    qo, so = oracle.quantize_weight(W)
    bias = synth.normal_bf16(0, 541, (N,), 0.02)
    y = torch.empty(B, N, device="cuda")
    xq = torch.empty(B, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(B, device="cuda")
    acc = torch.empty(B, N, dtype=torch.int32, device="cuda")
    nc.w8a8_gemv(x.cuda(), None, 0.0, torch.from_numpy(qo).cuda(), torch.from_numpy(so).cuda(),
                 bias.cuda(), y, xq, sx, acc)
    torch.cuda.synchronize()
    for r in range(B):
        xq_o, sx_o = oracle.quantize_row(x[r].numpy())
        assert np.array_equal(xq[r].cpu().numpy(), xq_o)
        assert sx[r].item() == float(sx_o)
        assert np.array_equal(acc[r].cpu().numpy(), oracle.matvec_i8(qo, xq_o))
        ref = oracle.linear_w8a8(qo, so, bias, x[r].numpy())
        assert rel_l2(f32(y[r]), ref) < 1e-6


@pytest.mark.parametrize("B,K,N", [(1, 896, 1152), (4, 896, 77), (16, 4864, 33)])
def test_typed_stage_gemvs_w8a8_bit_exact(B, K, N):
    """The boundary's stage GEMVs with NC_INT8 weights (nc_rmsnorm_gemv with
    bias and int32 accumulators, nc_gemv_residual, nc_swiglu_gemv), on
    identical fp32 input (no norm): the accumulators equal the oracle's int64
    products of its own codes, and the bias and residual epilogues, each IEEE
    operation rounded on its own, equal the oracle's outputs bit for bit. The
    SwiGLU epilogue applies exp, whose last bit the device's and the host's
    libraries may round apart: within 4 ulp of the oracle's composition."""
    x = _x(B, K, 60 + N)
    W = synth.normal_bf16(0, 560 + N, (N, K), 0.02)
    qo, so = oracle.quantize_weight(W)
    bias = synth.normal_bf16(0, 561, (N,), 0.02)
    Wq, sw = torch.from_numpy(qo).cuda(), torch.from_numpy(so).cuda()
    y = torch.empty(B, N, device="cuda")
    acc = torch.empty(B, N, dtype=torch.int32, device="cuda")
    nc.rmsnorm_gemv(x.cuda(), None, 0.0, Wq, bias.cuda(), y, w_scale=sw, acc=acc)
    r0 = _x(B, N, 70 + N)
    res = r0.cuda()
    nc.gemv_residual(x.cuda(), Wq, res, w_scale=sw)
    Wg = synth.normal_bf16(0, 562 + N, (2 * N, K), 0.02)
    qg, sg = oracle.quantize_weight(Wg)
    h = torch.empty(B, N, device="cuda")
    nc.swiglu_gemv(x.cuda(), None, 0.0, torch.from_numpy(qg).cuda(), h,
                   s_gu=torch.from_numpy(sg).cuda())
    torch.cuda.synchronize()
    for r in range(B):
        xq_o, _ = oracle.quantize_row(x[r].numpy())
        assert np.array_equal(acc[r].cpu().numpy(), oracle.matvec_i8(qo, xq_o))
        ref = oracle.linear_w8a8(qo, so, bias, x[r].numpy())
        assert np.array_equal(f32(y[r]).view(np.uint32), ref.view(np.uint32))
        lin = oracle.linear_w8a8(qo, so, None, x[r].numpy())
        want = (r0[r].numpy() + lin).astype(np.float32)
        assert np.array_equal(f32(res[r]).view(np.uint32), want.view(np.uint32))
        gu = oracle.linear_w8a8(qg, sg, None, x[r].numpy())
        hs = np.array([np.float32(oracle.silu(float(g))) * u for g, u in zip(gu[:N], gu[N:])],
                      np.float32)
        got = f32(h[r])
        assert np.all(np.abs(got - hs) <= 4 * np.spacing(np.abs(hs).astype(np.float32))), \
            np.abs(got - hs).max()


def test_typed_stage_gemv_int8_codes_near_boundary_only():
    """With the RMSNorm in the prologue the normed input is formed on each
    side by its own fp32 sums; the activation codes then equal the oracle's
    except where the oracle's quotient lies within CODE_BOUNDARY_TOL of a .5
    boundary, where neighbouring codes are both correct."""
    B, K, N = 4, 896, 64
    x = _x(B, K, 75)
    gamma = synth.normal_bf16(0, 571, (K,), 0.02, 1.0)
    W = synth.normal_bf16(0, 572, (N, K), 0.02)
    qo, so = oracle.quantize_weight(W)
    y = torch.empty(B, N, device="cuda")
    xq = torch.empty(B, K, dtype=torch.int8, device="cuda")
    nc.w8a8_gemv(x.cuda(), gamma.cuda(), 1e-6, torch.from_numpy(qo).cuda(),
                 torch.from_numpy(so).cuda(), None, y, xq)
    torch.cuda.synchronize()
    for r in range(B):
        xn = oracle.rmsnorm(x[r].numpy(), gamma, 1e-6)
        own, s = oracle.quantize_row(xn)
        got = xq[r].cpu().numpy()
        d = np.nonzero(own != got)[0]
        if d.size:
            assert np.all(np.abs(own[d].astype(int) - got[d].astype(int)) == 1)
            q = np.abs(xn[d].astype(np.float64) / float(s))
            assert np.all(np.abs(q - np.floor(q) - 0.5) <= 2.0 ** -10)


def test_w8a8_gemv_normed_and_zero_input():
    B, K, N = 2, 896, 200
    x = _x(B, K, 55)
    x[1] = 0.0                                # amax = 0 -> all-zero codes, y = bias
    W = synth.normal_bf16(0, 550, (N, K), 0.02)
    gamma = synth.normal_bf16(0, 551, (K,), 0.02, 1.0)
    qo, so = oracle.quantize_weight(W)
    y = torch.empty(B, N, device="cuda")
    nc.w8a8_gemv(x.cuda(), gamma.cuda(), 1e-6, torch.from_numpy(qo).cuda(),
                 torch.from_numpy(so).cuda(), None, y)
    torch.cuda.synchronize()
    ref = oracle.linear_w8a8(qo, so, None, oracle.rmsnorm(x[0].numpy(), gamma, 1e-6))
    assert rel_l2(f32(y[0]), ref) < REL_L2_GATE
    assert not y[1].any()


# ------------------------------------------------------------------ RoPE + attention
def _one_layer_model(shape, max_batch, max_ctx):
    import dataclasses
    s1 = dataclasses.replace(shape.with_layers(1), vocab=512)
    w = synth.model_weights(s1, seed=0)
    return s1, w, nc.Model(s1, to_device(w), max_batch=max_batch, max_ctx=max_ctx)


def _oracle_q_kv(shape, w, qkv_row, pos):
    """Oracle of the RoPE stage for one token: rotated q heads, rotated k and
    v per kv head (fp32, before the cache stores them)."""
    D, Hq, Hkv = shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    lw = w["layers"][0]
    q = qkv_row[:Hq * D].astype(np.float32).reshape(Hq, D)
    k = qkv_row[Hq * D:(Hq + Hkv) * D].astype(np.float32).reshape(Hkv, D)
    v = qkv_row[(Hq + Hkv) * D:].astype(np.float32).reshape(Hkv, D)
    qo, ko = [], []
    for h in range(Hq):
        qh = oracle.rmsnorm(q[h], lw["g_q"], shape.rms_eps) if shape.qk_norm else q[h]
        qo.append(oracle.rope(qh, pos, shape.rope_theta))
    for g in range(Hkv):
        kh = oracle.rmsnorm(k[g], lw["g_k"], shape.rms_eps) if shape.qk_norm else k[g]
        ko.append(oracle.rope(kh, pos, shape.rope_theta))
    return np.stack(qo), np.stack(ko).astype(np.float32), v


CASES = [
    # shape, positions, paged
    (synth.QWEN2_0P5B, [0], False),                 # single key: attention returns v
    (synth.QWEN2_0P5B, [16], False),                # 16 past positions
    (synth.QWEN2_0P5B, [17, 1, 100], False),        # ragged batch
    (synth.QWEN2_0P5B, [512], False),               # nine splits of one chunk each
    (synth.QWEN2_0P5B, [15, 16, 31, 4095], True),   # paged, block boundaries, long
    (synth.QWEN3_8B, [4096], False),                # 8B shape, q/k norm, D = 128
    (synth.QWEN3_8B, [33, 700], True),
    (synth.TINY, [5, 0], True),
    # a group of 8 query heads per kv head at D = 128 (two value pairs per thread)
    (dataclasses.replace(synth.TINY_QKNORM, hidden=1024, n_q_heads=8, n_kv_heads=1), [300, 64], True),
    # one query head per kv head
    (dataclasses.replace(synth.TINY, n_kv_heads=4), [130, 2], False),
    # head size 64, scored in 8-dim slices: a full group of 8 heads, and a group
    # of 5 (three padding heads)
    (dataclasses.replace(synth.TINY, hidden=512, n_q_heads=8, n_kv_heads=1), [200, 37], True),
    (dataclasses.replace(synth.TINY, hidden=640, n_q_heads=10, n_kv_heads=2), [70, 129], False),
]


@pytest.mark.parametrize("kv_bf16", [False, True])
@pytest.mark.parametrize("shape,positions,paged", CASES)
def test_rope_append_and_attention(shape, positions, paged, kv_bf16):
    B = len(positions)
    D, Hq, Hkv = shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    max_ctx = max(positions) + 17
    s1, w, model = _one_layer_model(shape, B, max_ctx)
    kdt = torch.bfloat16 if kv_bf16 else torch.float32
    if paged:
        table, nblk = synth.block_tables(positions, 1, 16)
        kv = nc.KVCache(s1, B, paged=True, block_table=table, num_blocks=nblk, dtype=kdt)
    else:
        kv = nc.KVCache(s1, B, max_ctx=max_ctx, dtype=kdt)

    def stored(a):  # what the cache holds for fp32 values a (as the oracle stores them)
        return oracle.f32_to_bf16(a) if kv_bf16 else np.asarray(a, np.float32)

    def held(t):  # a cache tensor as the oracle reads it
        return bf16_bits(t) if kv_bf16 else f32(t)
    past = {}
    for b, p in enumerate(positions):
        for g in range(Hkv):
            kr = synth.synthetic_kv_rows(s1, 0, b, g, 0, p)
            vr = synth.synthetic_kv_rows(s1, 0, b, g, 1, p)
            past[b, g] = (kr, vr)
            if p:
                kv.write_sequence(0, b, g, kr.cuda(), vr.cuda())
    g = torch.Generator().manual_seed(sum(positions) + D)
    qkv = (torch.randn(B, (Hq + 2 * Hkv) * D, generator=g) * 0.7).float()
    pos_t = torch.tensor(positions, dtype=torch.int32)
    q_out = torch.full((B, Hq * D), float("nan"), device="cuda")
    model.rope_qkv(0, qkv.cuda(), pos_t.cuda(), pos_t, q_out, kv)
    out = torch.full((B, Hq * D), float("nan"), device="cuda")
    model.attn_decode(0, q_out, pos_t.cuda(), pos_t, kv, out)
    torch.cuda.synchronize()
    for b, p in enumerate(positions):
        qo, ko, vo = _oracle_q_kv(s1, w, qkv[b].numpy(), p)
        assert rel_l2(f32(q_out[b]).reshape(Hq, D), qo) < 1e-6
        for gk in range(Hkv):
            ks, vs = kv.slot_view(0, b, gk, p)
            want_k = oracle.bf16_to_f32(stored(ko[gk])) if kv_bf16 else ko[gk]
            assert rel_l2(f32(ks), want_k) < (1e-3 if kv_bf16 else 1e-6)
            assert np.array_equal(held(vs), stored(vo[gk]))
        for h in range(Hq):
            gk = h // (Hq // Hkv)
            kr, vr = past[b, gk]
            kk = np.concatenate([held(kr).reshape(p, D), stored(ko[gk])[None]])
            vv = np.concatenate([held(vr).reshape(p, D), stored(vo[gk])[None]])
            ref = oracle.attention_head(qo[h], kk, vv)
            got = f32(out[b, h * D:(h + 1) * D])
            assert rel_l2(got, ref) < REL_L2_GATE / 10, (b, h, rel_l2(got, ref))
            if p == 0:  # a single key: attention returns v as stored
                assert np.allclose(got, f32(kv.slot_view(0, b, gk, p)[1]), rtol=1e-6, atol=0)
    model.close()


# ------------------------------------------------------------------ LM head + argmax
@pytest.mark.parametrize("B", [4, 16])
def test_lm_head_argmax_and_ties(B):
    """LM head logits and greedy tokens; B = 16 runs on the tensor cores."""
    s = synth.TINY
    _, w, model = _one_layer_model(s, B, 32)
    V, K = 151936, 896
    W = synth.normal_bf16(0, 560, (V, K), 0.02)
    # planted exact tie: rows 1000 and 90000 identical and dominant for b = 0
    x = _x(B, K, 61)
    xn0 = oracle.rmsnorm(x[0].numpy(), synth.normal_bf16(0, 562, (K,), 0.02, 1.0), 1e-6)
    hot = torch.tensor(np.sign(xn0) * 0.1, dtype=torch.float32).to(torch.bfloat16)
    W[1000] = hot
    W[90000] = hot
    gamma = synth.normal_bf16(0, 562, (K,), 0.02, 1.0)
    logits = torch.empty(B, V, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    model.lm_head_argmax(x.cuda(), gamma.cuda(), 1e-6, W.cuda(), logits, nxt)
    torch.cuda.synchronize()
    assert nxt[0].item() == 1000
    assert logits[0, 1000].item() == logits[0, 90000].item()
    for b in range(B):
        ref = oracle.matvec_bf16(W, oracle.rmsnorm(x[b].numpy(), gamma, 1e-6))
        got = f32(logits[b])
        assert rel_l2(got, ref) < REL_L2_GATE / 10
        # the GPU's argmax is exact on its own logits
        assert nxt[b].item() == int(np.argmax(got))
    assert model.device_status() == 0
    # a NaN input gives next = -1 and a nonzero device status
    x[2, 3] = float("nan")
    model.lm_head_argmax(x.cuda(), gamma.cuda(), 1e-6, W.cuda(), logits, nxt)
    torch.cuda.synchronize()
    assert nxt[2].item() == -1 and nxt[1].item() >= 0
    assert model.device_status() != 0
    assert model.device_status() == 0      # reading clears it
    model.close()
