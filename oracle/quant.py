"""Quantised storage and arithmetic beyond the per-row W8A8 path: int8
activations in blocks of 32, int8 embedding / LM-head rows, INT4 group-wise
weights and their packing, and the byte footprint of each level.

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline use this module. Plain numpy: every step is an elementwise IEEE
operation in the precision stated, and sums run in the order the definition
gives (across rows at once, never reassociated).

Definitions (nanoinfer, "Quantization" and the INT8 activation section):

* Symmetric, no zero point: a stored value is q * scale. int8 uses the range
  [-127, 127] so a value and its negation quantise to opposite codes; INT4
  has fifteen levels, [-7, 7]. Rounding is half away from zero (not banker's
  rounding). A group whose largest magnitude is 0 gets scale 0 and codes 0.
* Weights: int8 one scale per output row; INT4 one scale per group of
  `group` consecutive weights of a row (32 or 128).
* Activations: one scale per block of 32 consecutive values of a token's
  vector ("one per 32"), so an outlier only widens its own block.
* Norms and biases are never quantised.

Readings where the page is silent: scales are fp32 (the footprint table
fixes this for INT4: fp16 group scales would put group 32 at 0.75 GB, not
0.77); scale = fp32(amax / levels) by IEEE division and code =
round_half_away(fp32(v / scale)); a ragged last block or group is shorter;
two INT4 codes share a byte, the even index in the low nibble, each nibble
two's complement; the blocked int8 product sums the per-block int32
accumulators as float(acc_b) * (s_w * s_x[b]) in block order in fp32, then
adds the bias; the INT4 product is the fp32 dot product of the dequantised
row (q * s rounded to fp32) with x, in index order, as in the page's
quantise-dequantise evaluation.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
I8_LEVELS = 127
I4_LEVELS = 7
ACT_BLOCK = 32


def round_half_away(x: np.ndarray) -> np.ndarray:
    """Nearest integer, halves away from zero, exact for any float input:
    the fractional part x - trunc(x) is computed exactly."""
    x = np.asarray(x)
    t = np.trunc(x)
    f = x - t
    return t + np.where(np.abs(f) >= 0.5, np.sign(x), 0.0).astype(x.dtype)


def quantize_group(v: np.ndarray, levels: int):
    """One symmetric scale for the values v: (codes int8, fp32 scale)."""
    v = np.asarray(v, np.float32)
    amax = F32(np.max(np.abs(v))) if v.size else F32(0)
    if amax == 0:
        return np.zeros(v.size, np.int8), F32(0)
    s = F32(amax / F32(levels))
    # elementwise: each quotient an IEEE fp32 division, then the rounding rule
    r = round_half_away((v / s).astype(np.float32))
    return np.clip(r, -levels, levels).astype(np.int8), s


# ------------------------------------------------------------------ int8
def quantize_rows_i8(w: np.ndarray):
    """Per-row int8 (weights, or embedding rows): codes [N, K], scales [N]."""
    w = np.asarray(w, np.float32)
    q = np.empty(w.shape, np.int8)
    s = np.empty(w.shape[0], np.float32)
    for n in range(w.shape[0]):
        q[n], s[n] = quantize_group(w[n], I8_LEVELS)
    return q, s


def quantize_blocks_i8(v: np.ndarray, block: int = ACT_BLOCK):
    """A token's activations in blocks of `block`: codes [n], scales [ceil(n/block)]."""
    v = np.asarray(v, np.float32)
    nb = -(-v.size // block)
    q = np.empty(v.size, np.int8)
    s = np.empty(nb, np.float32)
    for b in range(nb):
        q[b * block:(b + 1) * block], s[b] = quantize_group(v[b * block:(b + 1) * block], I8_LEVELS)
    return q, s


def matvec_i8_blocked(wq: np.ndarray, xq: np.ndarray, block: int = ACT_BLOCK) -> np.ndarray:
    """int32 accumulators [N, nblocks]: acc[n, b] = sum over block b of wq[n, k] * xq[k]
    (int64 arithmetic, checked to fit int32)."""
    wq = np.asarray(wq, np.int64)
    xq = np.asarray(xq, np.int64)
    n, k = wq.shape
    nb = -(-k // block)
    acc = np.empty((n, nb), np.int64)
    for b in range(nb):
        acc[:, b] = wq[:, b * block:(b + 1) * block] @ xq[b * block:(b + 1) * block]
    assert np.abs(acc).max(initial=0) < 2 ** 31
    return acc.astype(np.int32)


def linear_w8a8_blocked(wq, sw, bias, x, block: int = ACT_BLOCK):
    """y = dequantised int8 product of the rows wq (scales sw) with x quantised
    in blocks; bias (fp32 or None) added last. Returns (y, xq, sx, acc)."""
    xq, sx = quantize_blocks_i8(x, block)
    acc = matvec_i8_blocked(wq, xq, block)
    sw = np.asarray(sw, np.float32)
    # every row at once, the blocks in order: each step an fp32 product and an fp32 sum
    t = np.zeros(acc.shape[0], np.float32)
    for b in range(acc.shape[1]):
        t = (t + (acc[:, b].astype(np.float32) * (sw * sx[b]).astype(np.float32))
             .astype(np.float32)).astype(np.float32)
    y = t if bias is None else (t + np.asarray(bias, np.float32)).astype(np.float32)
    return y, xq, sx, acc


def embed_i8(eq: np.ndarray, es: np.ndarray, token: int) -> np.ndarray:
    """The fp32 residual row of an int8 embedding: q * s per element."""
    return (eq[token].astype(np.float32) * np.float32(es[token])).astype(np.float32)


# ------------------------------------------------------------------ INT4
def quantize_int4(w: np.ndarray, group: int):
    """Group-wise INT4: codes [N, K] in [-7, 7] (int8 holders), fp32 scales [N, ceil(K/group)]."""
    w = np.asarray(w, np.float32)
    n, k = w.shape
    ng = -(-k // group)
    q = np.empty((n, k), np.int8)
    s = np.empty((n, ng), np.float32)
    for r in range(n):
        for g in range(ng):
            q[r, g * group:(g + 1) * group], s[r, g] = quantize_group(
                w[r, g * group:(g + 1) * group], I4_LEVELS)
    return q, s


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Two codes a byte along the last axis (even length): the even index in
    the low nibble, two's complement nibbles."""
    q = np.asarray(q, np.int8)
    assert q.shape[-1] % 2 == 0 and np.abs(q).max(initial=0) <= I4_LEVELS
    lo = q[..., 0::2].astype(np.uint8) & 0xF
    hi = q[..., 1::2].astype(np.uint8) & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(p: np.ndarray) -> np.ndarray:
    p = np.asarray(p, np.uint8)
    lo = (p & 0xF).astype(np.int8)
    hi = (p >> 4).astype(np.int8)
    lo = np.where(lo >= 8, lo - 16, lo).astype(np.int8)
    hi = np.where(hi >= 8, hi - 16, hi).astype(np.int8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequant_int4(q: np.ndarray, s: np.ndarray, group: int) -> np.ndarray:
    """q * s rounded to fp32, each weight with its group's scale."""
    k = q.shape[1]
    sg = np.repeat(s, group, axis=1)[:, :k]
    return (q.astype(np.float32) * sg).astype(np.float32)


def linear_int4(packed: np.ndarray, s: np.ndarray, group: int, x: np.ndarray, prec="f32"):
    """y = W_deq x: each row's dequantised weights times x, summed in index
    order in fp32 (prec="f64": the same in fp64, the rounding reference)."""
    wd = dequant_int4(unpack_int4(packed), s, group)
    x = np.asarray(x, np.float32)
    if prec == "f64":
        return wd.astype(np.float64) @ x.astype(np.float64)
    # every row at once, k in index order: each step an fp32 product and an fp32 sum
    t = np.zeros(wd.shape[0], np.float32)
    for kk in range(wd.shape[1]):
        t = (t + (wd[:, kk] * x[kk]).astype(np.float32)).astype(np.float32)
    return t


# ------------------------------------------------------------------ footprints
def footprint_bytes(shape, level: str) -> int:
    """Bytes of a model's parameters stored at `level` (the levels of the
    nanoinfer page's perplexity table): "fp32"; "int8" (the seven per-layer
    projections int8 with one fp32 scale per row, the rest fp32);
    "int8+emb" (the embedding too, per row); "int4-g32" / "int4-g128" (the
    projections INT4 in groups, one fp32 scale per group, embedding fp32).
    Norm gains and biases stay fp32; the head is tied."""
    H, F, L, V = shape.hidden, shape.ffn, shape.n_layers, shape.vocab
    qd, kvd = shape.n_q_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim
    mats = [(qd + 2 * kvd, H), (H, qd), (2 * F, H), (H, F)]  # [rows, cols] per layer
    proj = L * sum(r * c for r, c in mats)
    rows = L * sum(r for r, _ in mats)
    emb = V * H
    small = L * 2 * H + H + (L * (qd + 2 * kvd) if shape.qkv_bias else 0)
    if level == "fp32":
        return 4 * (proj + emb + small)
    if level == "int8":
        return proj + 4 * rows + 4 * emb + 4 * small
    if level == "int8+emb":
        return proj + 4 * rows + emb + 4 * V + 4 * small
    if level.startswith("int4-g"):
        g = int(level[len("int4-g"):])
        groups = L * sum(r * -(-c // g) for r, c in mats)
        return proj // 2 + 4 * groups + 4 * emb + 4 * small
    raise ValueError(level)
