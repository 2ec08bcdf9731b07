"""Pins of the CPU oracle to facts outside itself: closed forms, library
routines, brute force on tiny inputs and the values the pages print.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, the wrong RoPE or GQA convention)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from transformer_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- bf16
def test_bf16_roundtrip_all_patterns(orc):
    """nanoinfer "Weights": widen then narrow is the identity on every
    non-NaN bf16 value."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = orc.bf16_to_f32(bits)
    back = orc.f32_to_bf16(f)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all(back[nan] == 0x7FC0)
    # widening appends 16 zero bits
    assert np.array_equal(f.view(np.uint32), bits.astype(np.uint32) << 16)


def test_bf16_round_half_even(orc):
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2.0 ** -8: 0x3F80,             # tie -> even (down)
        one + 3 * 2.0 ** -8: 0x3F82,         # tie -> even (up)
        one + 2.0 ** -8 + 2.0 ** -20: 0x3F81,  # above the tie
        -(one + 2.0 ** -8): 0xBF80,
        3.4e38: 0x7F80,                      # rounds up to infinity
    }
    for v, want in cases.items():
        assert int(orc.f32_to_bf16(np.array([v], np.float32))[0]) == want, v


def test_bf16_narrow_matches_torch(orc):
    """torch's fp32 -> bf16 conversion (a library routine) rounds the same way."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8)
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f32_to_bf16(x.numpy()), ref)


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_vector(orc):
    """For x = c * 1: out_i = c / sqrt(c^2 + eps) * g_i."""
    n, c, eps = 896, 0.37, 1e-6
    g = synth.normal_bf16(0, 77, (n,), 0.02, 1.0)
    gf = orc.bf16_to_f32(g.view(torch.int16).numpy()).astype(np.float64)
    out = orc.rmsnorm(np.full(n, c), g, eps, "f64")
    assert np.allclose(out, c / math.sqrt(c * c + eps) * gf, rtol=1e-13, atol=0)
    # fp32: the index-order sum of n squares is within n * 2^-24 relative
    c32 = float(np.float32(c))
    out32 = orc.rmsnorm(np.full(n, c32, np.float32), g, eps, "f32")
    assert np.allclose(out32, c32 / math.sqrt(c32 * c32 + eps) * gf, rtol=n * 2.0 ** -24, atol=0)


def test_rmsnorm_matches_torch_and_scale_invariance(orc):
    gen = torch.Generator().manual_seed(1)
    x = torch.randn(4864, generator=gen, dtype=torch.float64)
    g = synth.normal_bf16(0, 78, (4864,), 0.02, 1.0)
    ref = torch.nn.functional.rms_norm(x, (4864,), g.to(torch.float64), eps=1e-6).numpy()
    out = orc.rmsnorm(x.numpy(), g, 1e-6, "f64")
    assert _rel_l2(out, ref) < 1e-14
    # rms(ax) = rms(x) exactly without eps; with eps the shift is eps / (2 ms)
    a0 = orc.rmsnorm(x.numpy(), g, 0.0, "f64")
    assert _rel_l2(orc.rmsnorm(1024.0 * x.numpy(), g, 0.0, "f64"), a0) < 1e-15
    ms = float((x * x).mean())
    assert abs(_rel_l2(out, a0) - 1e-6 / (2 * ms)) < 1e-9


def test_rmsnorm_gain_applies_per_element(orc):
    x = np.arange(1, 9, dtype=np.float64)
    g = _bf16_bits([1, 2, 1, 1, 1, 1, 1, 0.5])
    out = orc.rmsnorm(x, g, 0.0, "f64")
    r = 1 / math.sqrt(np.mean(x * x))
    assert np.allclose(out, x * r * np.array([1, 2, 1, 1, 1, 1, 1, 0.5]), rtol=1e-15)


# ---------------------------------------------------------------- GEMV
def test_matvec_exact_small_integers(orc):
    """With entries k/8 and small-integer x the fp32 sums are exact, so the
    oracle must equal integer arithmetic: catches a transposed operand or an
    off-by-one in the row stride."""
    rng = np.random.default_rng(3)
    n, k = 37, 53
    wi = rng.integers(-8, 9, size=(n, k))
    xi = rng.integers(-5, 6, size=k)
    w = _bf16_bits(wi / 8.0).reshape(n, k)
    y = orc.matvec_bf16(w, xi.astype(np.float32), "f32")
    assert np.array_equal(y, (wi @ xi) / 8.0)


def test_matvec_matches_numpy_fp64(orc):
    n, k = 300, 896
    w = synth.normal_bf16(0, 79, (n, k), 0.02)
    x = np.random.default_rng(4).standard_normal(k)
    wf = orc.bf16_to_f32(w.view(torch.int16).numpy()).astype(np.float64)
    y = orc.matvec_bf16(w, x, "f64")
    assert _rel_l2(y, wf @ x) < 1e-14
    y32 = orc.matvec_bf16(w, x.astype(np.float32), "f32")
    # fp32 accumulation in index order: error below k * eps * sum|w x|
    bound = k * 2.0 ** -24 * (np.abs(wf) @ np.abs(x))
    assert np.all(np.abs(y32 - wf @ x) <= bound)


# ---------------------------------------------------------------- RoPE
def test_rope_inv_freq_closed_form(orc):
    f = orc.rope_inv_freq(1e6, 64)
    assert f[0] == 1.0
    assert f[16] == np.float32(1e-3)          # theta^(-1/2)
    assert np.allclose(f, 1e6 ** (-np.arange(0, 64, 2) / 64.0), rtol=1e-7)


def test_rope_half_split_closed_form(orc):
    """D = 4, theta = 10^4: inv_freq = [1, 0.01]. The half-split rotation
    pairs component 0 with 2 and 1 with 3."""
    v = np.array([1.0, 0.0, 0.0, 0.0])
    out = orc.rope(v, 1, 1e4, "f64")
    assert np.allclose(out, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    v = np.array([0.0, 1.0, 0.0, 0.0])
    out = orc.rope(v, 3, 1e4, "f64")
    a = float(np.float32(3.0) * np.float32(0.01))   # fp32 angle product
    assert np.allclose(out, [0, math.cos(a), 0, math.sin(a)], atol=1e-15)
    v = np.array([0.0, 0.0, 1.0, 0.0])
    out = orc.rope(v, 1, 1e4, "f64")
    assert np.allclose(out, [-math.sin(1), 0, math.cos(1), 0], atol=1e-15)


def test_rope_identity_norms_relative_position(orc):
    rng = np.random.default_rng(5)
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    assert np.array_equal(orc.rope(q, 0, 1e6, "f64"), q)       # pos 0 is the identity
    rq = orc.rope(q, 1234, 1e6, "f64")
    pairs = lambda v: v[:32] ** 2 + v[32:] ** 2
    assert np.allclose(pairs(rq), pairs(q), rtol=1e-12)          # each pair keeps its norm
    # <R_p q, R_p' k> depends on p - p' only (exactly representable angles:
    # D = 2 with inv_freq 1 keeps the fp32 angle product exact)
    q2, k2 = q[:2], k[:2]
    d1 = orc.rope(q2, 10, 1e6, "f64") @ orc.rope(k2, 7, 1e6, "f64")
    d2 = orc.rope(q2, 110, 1e6, "f64") @ orc.rope(k2, 107, 1e6, "f64")
    assert abs(d1 - d2) < 1e-12
    # interleaved convention differs (nanoinfer: the wrong one must differ)
    assert not np.allclose(orc.rope(q, 5, 1e6, "f64"),
                           orc.rope(q, 5, 1e6, "f64", interleaved=True))


# ---------------------------------------------------------------- SiLU, softmax
def test_silu_matches_torch(orc):
    xs = np.concatenate([np.linspace(-30, 30, 601), [0.0, -0.0, 1e-30, -1e-30, 88.0, -88.0]])
    ref = torch.nn.functional.silu(torch.tensor(xs, dtype=torch.float64)).numpy()
    out = np.array([orc.silu(x, "f64") for x in xs])
    assert np.allclose(out, ref, rtol=1e-15, atol=1e-300)
    out32 = np.array([orc.silu(x, "f32") for x in xs])
    assert np.allclose(out32, ref, rtol=1e-6, atol=1e-37)
    for x in (0.3, 2.0, 7.5):
        assert abs(orc.silu(x, "f64") - orc.silu(-x, "f64") - x) < 1e-15


def test_softmax_sums_to_one_and_shift_invariant(orc):
    s = np.random.default_rng(6).standard_normal(300) * 5
    p = orc.softmax(s, "f64")
    assert abs(p.sum() - 1) < 300 * 2.0 ** -52
    assert np.allclose(orc.softmax(s + 123.0, "f64"), p, rtol=1e-12)
    ref = torch.softmax(torch.tensor(s), 0).numpy()
    assert _rel_l2(p, ref) < 1e-14


# ---------------------------------------------------------------- attention
def test_attention_single_key_returns_v(orc):
    q = np.random.default_rng(8).standard_normal(64).astype(np.float32)
    k = synth.normal_bf16(0, 80, (1, 64), 0.5)
    v = synth.normal_bf16(0, 81, (1, 64), 0.5)
    out = orc.attention_head(q, k, v, "f32")
    assert np.array_equal(out, orc.bf16_to_f32(v.view(torch.int16).numpy())[0])


def test_attention_equal_keys_gives_mean_of_v(orc):
    q = np.random.default_rng(9).standard_normal(64)
    k = synth.normal_bf16(0, 82, (1, 64), 0.5).repeat(37, 1)
    v = synth.normal_bf16(0, 83, (37, 64), 0.5)
    vf = orc.bf16_to_f32(v.view(torch.int16).numpy()).astype(np.float64)
    out = orc.attention_head(q, k, v, "f64")
    assert np.allclose(out, vf.mean(0), rtol=1e-13, atol=1e-15)


def test_attention_matches_torch_sdpa(orc):
    """torch's scaled_dot_product_attention (a library routine) with scale
    1/sqrt(D) on the same bf16 keys and values."""
    for d, n in ((64, 1), (64, 100), (128, 513)):
        q = torch.randn(d, dtype=torch.float64, generator=torch.Generator().manual_seed(d + n))
        k = synth.normal_bf16(0, 84 + n, (n, d), 0.6)
        v = synth.normal_bf16(0, 85 + n, (n, d), 0.6)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.view(1, 1, 1, d), k.double().view(1, 1, n, d), v.double().view(1, 1, n, d)).view(d)
        out = orc.attention_head(q.numpy(), k, v, "f64")
        assert _rel_l2(out, ref.numpy()) < 1e-13
        # the same keys and values held as fp32 (the default cache type)
        out32 = orc.attention_head(q.numpy(), k.float().numpy(), v.float().numpy(), "f64")
        assert _rel_l2(out32, ref.numpy()) < 1e-13


# ---------------------------------------------------------------- int8
def test_quantize_row_half_away_from_zero(orc):
    q, s = orc.quantize_row(np.array([127.0, 0.5, -0.5, 2.5, -2.5, 1.49, 0.0], np.float32))
    assert s == 1.0
    assert q.tolist() == [127, 1, -1, 3, -3, 1, 0]       # banker's rounding would give 0, 2
    q, s = orc.quantize_row(np.array([1.0, -0.5, 0.25, 0.0], np.float32))
    assert s == np.float32(1.0) / np.float32(127.0)
    assert q.tolist() == [127, -64, 32, 0]
    q, s = orc.quantize_row(np.zeros(9, np.float32))
    assert s == 0 and not q.any()
    # symmetric: a value and its negation quantise to exact opposites
    v = np.random.default_rng(10).standard_normal(1000).astype(np.float32)
    qa, _ = orc.quantize_row(v)
    qb, _ = orc.quantize_row(-v)
    assert np.array_equal(qa, -qb) and qa.max() <= 127 and qa.min() >= -127


def test_matvec_i8_brute_force_and_range(orc):
    rng = np.random.default_rng(11)
    w = rng.integers(-127, 128, size=(23, 4864)).astype(np.int8)
    x = rng.integers(-127, 128, size=4864).astype(np.int8)
    acc = orc.matvec_i8(w, x)
    ref = [sum(int(a) * int(b) for a, b in zip(row, x)) for row in w]
    assert acc.tolist() == ref
    full = orc.matvec_i8(np.full((2, 4864), 127, np.int8), np.full(4864, -127, np.int8))
    assert full.tolist() == [-78451456, -78451456]
    with pytest.raises(OverflowError):
        orc.matvec_i8(np.full((1, 140000), 127, np.int8), np.full(140000, 127, np.int8))


def test_quantize_weight_rows(orc):
    w = _bf16_bits([[0.5, -0.25, 0.0, 0.125], [0.0, 0.0, 0.0, 0.0], [-2.0, 1.0, 0.5, 0.0]])
    q, s = orc.quantize_weight(w.reshape(3, 4))
    assert s.tolist() == [np.float32(0.5) / np.float32(127), 0.0, np.float32(2.0) / np.float32(127)]
    assert q.tolist() == [[127, -64, 0, 32], [0, 0, 0, 0], [-127, 64, 32, 0]]


def test_linear_w8a8_dequant(orc):
    rng = np.random.default_rng(12)
    w = synth.normal_bf16(0, 86, (50, 96), 0.02)
    q8, sw = orc.quantize_weight(w)
    x = rng.standard_normal(96).astype(np.float32)
    xq, sx = orc.quantize_row(x)
    acc = orc.matvec_i8(q8, xq)
    y = orc.linear_w8a8(q8, sw, None, x, "f64")
    assert np.allclose(y, acc * (sw.astype(np.float64) * float(sx)), rtol=1e-15)
    # the quantised product approximates the bf16 product
    wf = orc.bf16_to_f32(w.view(torch.int16).numpy()).astype(np.float64)
    assert _rel_l2(y, wf @ x) < 0.05


# ---------------------------------------------------------------- argmax
def test_argmax_lowest_index_and_nan(orc):
    v = np.array([1.0, 3.0, -2.0, 3.0, 3.0], np.float32)
    assert orc.argmax(v) == 1
    assert orc.argmax(np.array([-np.inf, -np.inf], np.float32)) == 0
    assert orc.argmax(np.array([0.0, np.nan, 5.0], np.float32)) == -1


# ---------------------------------------------------------------- shape
def _golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            out[k] = int(v)
    return out


def test_param_count_matches_page():
    gold = _golden("qwen2_0p5b_shape.txt")
    s = synth.QWEN2_0P5B
    pc = synth.param_count(s)
    for key in ("total", "embeddings", "mlp", "attention", "norms"):
        assert pc[key] == gold[key], key
    # the generator's own tensors have exactly these sizes
    lw = synth.layer_weights(s.with_layers(1), 0)
    per_layer = sum(t.numel() for t in lw.values() if t is not None)
    emb = s.vocab * s.hidden
    assert emb + s.n_layers * per_layer + s.hidden == gold["total"]
    # KV bytes per token at fp32 across all layers, with and without GQA
    assert s.n_layers * 2 * s.kv_dim * 4 == gold["kv_bytes_per_token_fp32"]
    assert s.n_layers * 2 * s.q_dim * 4 == gold["kv_bytes_per_token_fp32_mha"]


def test_generator_is_device_independent_and_seeded():
    a = synth.normal_bf16(0, 5, (1000,), 0.02)
    b = synth.normal_bf16(0, 5, (1000,), 0.02)
    c = synth.normal_bf16(0, 6, (1000,), 0.02)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    x = synth.normal_bf16(0, 9, (200000,), 0.02).float()
    assert abs(x.mean().item()) < 2e-4 and abs(x.std().item() / 0.02 - 1) < 0.01


def test_paged_inputs_follow_the_allocation_reading():
    """Reading R16 for the paged workloads: sequence b owns ceil((P_b + steps) / 16)
    blocks of a pool of exactly the blocks needed, each block owned once, in a
    seeded shuffled order; unused table entries are -1. Past lengths are
    seeded and inside [256, 4096]."""
    past = synth.past_lengths(16, 256, 4096).tolist()
    assert past == synth.past_lengths(16, 256, 4096).tolist()
    assert all(256 <= p <= 4096 for p in past) and len(set(past)) > 8
    table, total = synth.block_tables(past, 32, 16)
    need = [-(-(p + 32) // 16) for p in past]
    assert total == sum(need) and table.shape == (16, max(need))
    owned = []
    for b, n in enumerate(need):
        row = table[b].tolist()
        assert all(0 <= x < total for x in row[:n]) and all(x == -1 for x in row[n:])
        owned += row[:n]
    assert sorted(owned) == list(range(total))                # a permutation of the pool
    assert owned != list(range(total))                        # shuffled, not in order
    t2, _ = synth.block_tables(past, 32, 16)
    assert torch.equal(table, t2)                             # seeded
    t3, _ = synth.block_tables(past, 32, 16, seed=9)
    assert not torch.equal(table, t3)


def test_uniform_f64_is_seeded_and_in_the_open_unit_interval():
    u = synth.uniform_f64(5, 0, 100000)
    assert u.dtype == torch.float64 and torch.equal(u, synth.uniform_f64(5, 0, 100000))
    assert (u > 0).all() and (u < 1).all()
    assert abs(u.mean().item() - 0.5) < 0.005 and abs(u.var().item() - 1 / 12) < 0.002
