"""Pins of the quantisation oracle (oracle/quant.py): the footprints the
nanoinfer page prints, exact integer arithmetic, the rounding rule, and the
closed forms of symmetric quantisation. CPU only."""
import os
from decimal import ROUND_HALF_UP, Decimal

import numpy as np
import pytest

from oracle import quant
from transformer_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_footprints.txt")


def test_footprints_match_the_page():
    want = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            want[k] = float(v)
    for level, gb in want.items():
        got = quant.footprint_bytes(synth.QWEN2_0P5B, level) / 1e9
        assert round(got, 2) == gb, (level, got)
    # fp32 is four bytes per parameter of the page's total
    assert quant.footprint_bytes(synth.QWEN2_0P5B, "fp32") == 4 * 494032768
    # the page's regression test: the two group sizes store different sizes
    assert quant.footprint_bytes(synth.QWEN2_0P5B, "int4-g32") != \
        quant.footprint_bytes(synth.QWEN2_0P5B, "int4-g128")


def test_round_half_away_against_decimal():
    rng = np.random.default_rng(1)
    vals = np.concatenate([np.arange(-8, 8.5, 0.5),
                           rng.uniform(-200, 200, 2000),
                           [np.nextafter(np.float32(0.5), np.float32(0)),
                            np.nextafter(np.float32(-2.5), np.float32(0)),
                            np.nextafter(np.float32(126.5), np.float32(200))]]).astype(np.float32)
    for v in vals:
        want = int(Decimal(float(v)).quantize(Decimal(1), rounding=ROUND_HALF_UP))
        assert int(quant.round_half_away(np.float32(v))) == want, v
    # banker's rounding would differ here
    assert int(quant.round_half_away(np.float32(0.5))) == 1
    assert int(quant.round_half_away(np.float32(-0.5))) == -1
    assert int(quant.round_half_away(np.float32(2.5))) == 3


def test_group_quantiser_closed_forms():
    # a constant group is all top codes; its negation the opposite codes
    q, s = quant.quantize_group(np.full(32, 0.37, np.float32), 127)
    assert (q == 127).all() and s == np.float32(np.float32(0.37) / np.float32(127))
    qn, sn = quant.quantize_group(np.full(32, -0.37, np.float32), 127)
    assert (qn == -127).all() and sn == s
    # zero group: scale 0, codes 0
    q, s = quant.quantize_group(np.zeros(17, np.float32), 7)
    assert s == 0 and (q == 0).all()
    # symmetric: v and -v give opposite codes
    rng = np.random.default_rng(2)
    v = rng.standard_normal(64).astype(np.float32)
    q1, s1 = quant.quantize_group(v, 7)
    q2, s2 = quant.quantize_group(-v, 7)
    assert s1 == s2 and np.array_equal(q1, -q2)
    # the error bound of round-to-nearest: |v - q s| <= s / 2 (+ fp32 rounding)
    for levels in (7, 127):
        q, s = quant.quantize_group(v, levels)
        err = np.abs(v.astype(np.float64) - q.astype(np.float64) * float(s))
        assert err.max() <= float(s) * (0.5 + 1e-6)
        assert np.abs(q).max() == levels


def test_int4_fifteen_levels_and_packing():
    w = np.linspace(-1, 1, 15, dtype=np.float32)[None, :].repeat(2, 0)
    w = np.concatenate([w, np.zeros((2, 1), np.float32)], 1)  # 16 columns
    q, s = quant.quantize_int4(w, 16)
    assert sorted(set(q[0].tolist())) == list(range(-7, 8))  # fifteen levels
    # every pair of codes survives packing; the even index is the low nibble
    codes = np.array([[a, b] for a in range(-7, 8) for b in range(-7, 8)], np.int8)
    p = quant.pack_int4(codes)
    assert np.array_equal(quant.unpack_int4(p), codes)
    assert quant.pack_int4(np.array([[1, 0]], np.int8))[0, 0] == 0x01
    assert quant.pack_int4(np.array([[0, 1]], np.int8))[0, 0] == 0x10
    assert quant.pack_int4(np.array([[-1, -7]], np.int8))[0, 0] == 0x9F
    # every byte whose nibbles are codes unpacks and packs back
    for byte in range(256):
        lo, hi = byte & 0xF, byte >> 4
        if lo == 8 or hi == 8:  # -8 is not a code of the symmetric range
            continue
        b = np.array([[byte]], np.uint8)
        assert quant.pack_int4(quant.unpack_int4(b))[0, 0] == byte


def test_int4_groups_confine_outliers():
    """One large weight per row: groups of 32 keep the other groups' resolution,
    so their error is below that of groups of 128 (the page's reason for groups)."""
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    w[:, 200] = 0.5
    e = {}
    for g in (32, 128):
        q, s = quant.quantize_int4(w, g)
        assert s.shape == (8, 256 // g)
        wd = quant.dequant_int4(q, s, g)
        e[g] = np.linalg.norm(wd - w) / np.linalg.norm(w)
    assert e[32] < e[128]


def test_int4_linear_matches_fp64_brute_force():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((40, 200)) * 0.02).astype(np.float32)  # ragged last group at 32
    x = rng.standard_normal(200).astype(np.float32)
    for g in (32, 128):
        q, s = quant.quantize_int4(w, g)
        p = quant.pack_int4(q)
        y = quant.linear_int4(p, s, g, x)
        y64 = quant.linear_int4(p, s, g, x, prec="f64")
        wd = quant.dequant_int4(q, s, g).astype(np.float64)
        bound = 200 * 2.0 ** -24 * (np.abs(wd) @ np.abs(x.astype(np.float64)))
        assert (np.abs(y - y64) <= bound).all()
        # brute force from the definition, element by element
        yb = [sum(float(q[j, k]) * float(s[j, k // g]) * float(x[k]) for k in range(200))
              for j in range(3)]
        assert np.allclose(y64[:3], yb, rtol=1e-6, atol=1e-9)


def test_blocked_int8_is_exact_integer_arithmetic():
    rng = np.random.default_rng(5)
    n, k = 24, 4864 + 16  # ragged last block
    wq = rng.integers(-127, 128, (n, k)).astype(np.int8)
    x = (rng.standard_normal(k) * np.where(rng.random(k) < 0.01, 60, 1)).astype(np.float32)
    y, xq, sx, acc = quant.linear_w8a8_blocked(wq, np.full(n, 0.01, np.float32), None, x)
    assert sx.size == -(-k // 32) and acc.shape == (n, sx.size)
    for j in range(3):
        for b in (0, 7, acc.shape[1] - 1):
            lo, hi = 32 * b, min(k, 32 * b + 32)
            assert acc[j, b] == sum(int(wq[j, i]) * int(xq[i]) for i in range(lo, hi))
    # the blocks add up to the unblocked accumulator
    full = wq.astype(np.int64) @ xq.astype(np.int64)
    assert np.array_equal(acc.astype(np.int64).sum(1), full)
    # the extreme accumulator of a 4864-wide row still fits int32
    big = quant.matvec_i8_blocked(np.full((1, 4864), 127, np.int8), np.full(4864, 127, np.int8))
    assert int(big.astype(np.int64).sum()) == 4864 * 127 * 127


def test_one_block_equals_the_per_row_w8a8(orc):
    """With one block as wide as the row, the blocked path is the per-row W8A8
    path of the C oracle, bit for bit (same quantiser, same epilogue)."""
    rng = np.random.default_rng(6)
    K, N = 896, 64
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w16 = orc.f32_to_bf16(w)
    w8, sw = orc.quantize_weight(w16)
    x = rng.standard_normal(K).astype(np.float32)
    y_row = orc.linear_w8a8(w8, sw, None, x)
    y_blk, xq, sx, _ = quant.linear_w8a8_blocked(w8, sw, None, x, block=K)
    q_row, s_row = orc.quantize_row(x)
    assert np.array_equal(xq, q_row) and sx[0] == np.float32(s_row)
    assert np.array_equal(y_blk, np.asarray(y_row, np.float32))


def test_blocks_confine_an_activation_outlier():
    """A 4864-wide vector with one element 68x the median (the ratio the page
    measured): per-32 blocks quantise it with a smaller error than one scale."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal(4864).astype(np.float32)
    x[1234] = 68 * np.median(np.abs(x))
    q1, s1 = quant.quantize_blocks_i8(x, 4864)
    q32, s32 = quant.quantize_blocks_i8(x, 32)
    e1 = np.linalg.norm(q1 * np.repeat(s1, 4864)[:4864] - x) / np.linalg.norm(x)
    e32 = np.linalg.norm(q32 * np.repeat(s32, 32)[:4864] - x) / np.linalg.norm(x)
    assert e32 < e1 / 3


def test_int8_embedding_rows():
    rng = np.random.default_rng(8)
    e = (rng.standard_normal((50, 96)) * 0.02).astype(np.float32)
    eq, es = quant.quantize_rows_i8(e)
    for t in (0, 17, 49):
        row = quant.embed_i8(eq, es, t)
        assert np.array_equal(row, eq[t].astype(np.float32) * es[t])
        assert np.abs(row - e[t]).max() <= es[t] * (0.5 + 1e-6)


@pytest.mark.parametrize("K", [96, 100, 896, 4864])
def test_c_blocked_linear_equals_the_numpy_quantiser(orc, K):
    """The C oracle's blocked W8A8 product and oracle/quant.py, written
    separately, agree bit for bit in fp32 (same quantiser, same block-order
    epilogue), including a ragged last block (K = 100)."""
    rng = np.random.default_rng(K)
    N = 40
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    wq, sw = quant.quantize_rows_i8(w)
    x = rng.standard_normal(K).astype(np.float32)
    x[3] *= 68.0
    bias16 = orc.f32_to_bf16((rng.standard_normal(N) * 0.02).astype(np.float32))
    y_c = orc.linear_w8a8_blocked(wq, sw, bias16, x, 32)
    y_n, _, _, _ = quant.linear_w8a8_blocked(wq, sw, orc.bf16_to_f32(bias16), x, 32)
    assert np.array_equal(np.asarray(y_c, np.float32).view(np.uint32), y_n.view(np.uint32))
    # one block as wide as the row is the per-token path
    y_row = orc.linear_w8a8(wq, sw, bias16, x)
    y_one = orc.linear_w8a8_blocked(wq, sw, bias16, x, K)
    assert np.array_equal(np.asarray(y_row, np.float32), np.asarray(y_one, np.float32))


@pytest.mark.parametrize("N,K,group", [(40, 64, 32), (17, 896, 128), (9, 4864, 32), (5, 192, 64)])
def test_c_int4_linear_equals_the_numpy_product(orc, N, K, group):
    """The C oracle's INT4 product and oracle/quant.py, written separately,
    agree bit for bit in fp32: the same fp32 dequantised weights, the same
    index-order sum."""
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[:, 3] = 0.4
    q, s = quant.quantize_int4(w, group)
    p = quant.pack_int4(q)
    x = rng.standard_normal(K).astype(np.float32)
    y_c = np.asarray(orc.linear_int4(p, s, group, None, x), np.float32)
    y_n = quant.linear_int4(p, s, group, x)
    assert np.array_equal(y_c.view(np.uint32), y_n.view(np.uint32))
    y64 = orc.linear_int4(p, s, group, None, x.astype(np.float64), "f64")
    assert np.allclose(y64, quant.linear_int4(p, s, group, x, "f64"), rtol=1e-12, atol=1e-15)
