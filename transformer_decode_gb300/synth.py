"""Seeded synthetic inputs for the decode step: model shapes, weights, tokens,
past lengths, paged block tables and pre-filled KV content.

This module is the one piece both sides of every comparison share. It holds
none of the decode step's arithmetic: it only draws numbers. Every draw is a
pure function of (seed, stream, element index), computed with integer tensor
operations, so the same tensor comes out bit for bit on the CPU and on a GPU.

Generator: each element's 32-bit key is mixed with the MurmurHash3 32-bit
finalizer ("fmix32", Austin Appleby, MurmurHash3, public domain), twice with
different salts, giving eight independent bytes. Their sum is an Irwin-Hall
variate with 8 terms, which is standardised and scaled to the requested
standard deviation in fp32 and converted to bf16 by torch (round to nearest
even). The result is a bounded (|z| <= 4.88) stand-in for N(mean, std^2).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

_M32 = 0xFFFFFFFF
# Irwin-Hall over 8 uniform bytes: mean 8 * 127.5, variance 8 * (256^2 - 1) / 12.
_IH_MEAN = 1020
_IH_STD = math.sqrt(8 * (256 * 256 - 1) / 12.0)
_CHUNK = 1 << 24


# --------------------------------------------------------------------------
# Model shapes and named workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Hyperparameters of a Qwen2-style decoder."""

    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    n_layers: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    qkv_bias: bool = True
    qk_norm: bool = False
    tie_embeddings: bool = True

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_layers(self, n_layers: int) -> "ModelShape":
        return dataclasses.replace(self, n_layers=n_layers)


# Qwen2.5-0.5B shape (nanoinfer, "Model architecture" and parameter table).
QWEN2_0P5B = ModelShape(hidden=896, n_q_heads=14, n_kv_heads=2, head_dim=64,
                        ffn=4864, n_layers=24, vocab=151936)
# 8B shape: Qwen3-8B-like, per-head q/k RMSNorm, no QKV bias, untied head.
QWEN3_8B = ModelShape(hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                      ffn=12288, n_layers=36, vocab=151936, qkv_bias=False,
                      qk_norm=True, tie_embeddings=False)
# A tiny model that keeps brute force cheap: every size still spans ragged
# tails of the kernels' tiles.
TINY = ModelShape(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512,
                  n_layers=2, vocab=512)
TINY_QKNORM = ModelShape(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=384,
                         n_layers=2, vocab=328, qkv_bias=False, qk_norm=True,
                         tie_embeddings=False)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: a model plus batch, cache and step counts."""

    name: str
    shape: ModelShape
    batch: int
    prompt: int          # tokens run through the step before timing (C1)
    past: tuple          # (lo, hi) synthetic past length range, or None
    steps: int           # greedy decode steps
    paged: bool = False
    block_size: int = 16
    w8a8: bool = False


WORKLOADS = {
    # one block, 16 past positions
    "block_0p5b_past16": Workload("block_0p5b_past16", QWEN2_0P5B.with_layers(1),
                                  batch=1, prompt=0, past=(16, 16), steps=1),
    # full 24-layer model, 32-token prompt then 64 greedy tokens, contiguous KV
    "qwen2_0p5b_b1_greedy64": Workload("qwen2_0p5b_b1_greedy64", QWEN2_0P5B,
                                       batch=1, prompt=32, past=None, steps=64),
    # batch 16, paged KV (block 16, shuffled tables), past U[256, 4096], 32 steps
    "qwen2_0p5b_b16_paged": Workload("qwen2_0p5b_b16_paged", QWEN2_0P5B, batch=16,
                                     prompt=0, past=(256, 4096), steps=32,
                                     paged=True),
    # W8A8 projections, 512 past positions, 64 greedy tokens
    "qwen2_0p5b_w8a8_past512": Workload("qwen2_0p5b_w8a8_past512", QWEN2_0P5B,
                                        batch=1, prompt=0, past=(512, 512),
                                        steps=64, w8a8=True),
    # 8B shape at 4096 past positions, 64 greedy tokens
    "qwen3_8b_past4096": Workload("qwen3_8b_past4096", QWEN3_8B, batch=1,
                                  prompt=0, past=(4096, 4096), steps=64),
}

# Seeds of the input streams.
SEED_WEIGHTS, SEED_TOKENS, SEED_PAST, SEED_BLOCKS, SEED_KV = 0, 1, 2, 3, 4


# --------------------------------------------------------------------------
# Counter-based generator (integer tensor ops; identical on CPU and GPU)
# --------------------------------------------------------------------------
def _mul32(h: torch.Tensor, c: int) -> torch.Tensor:
    """(h * c) mod 2^32 for int64 tensors holding uint32 values, with every
    intermediate product below 2^49 so nothing overflows int64."""
    lo = h & 0xFFFF
    hi = h >> 16
    return (lo * c + ((hi * (c & 0xFFFF)) << 16)) & _M32


def fmix32(h: torch.Tensor) -> torch.Tensor:
    """MurmurHash3's 32-bit finalizer on int64 tensors holding uint32 values."""
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def _stream_key(seed: int, stream: int) -> int:
    k = torch.tensor([(seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x27D4EB2F) & _M32],
                     dtype=torch.int64)
    return int(fmix32(fmix32(k))[0])


def uint32_stream(seed: int, stream: int, n: int, device="cpu",
                  salt: int = 0) -> torch.Tensor:
    """n pseudo-random uint32 values (held in int64) for (seed, stream)."""
    key = _stream_key(seed, stream) ^ salt
    idx = torch.arange(n, dtype=torch.int64, device=device)
    return fmix32(fmix32((idx * 0x9E3779B1 + key) & _M32) ^ key)


def uniform_f64(seed: int, stream: int, n: int, device="cpu") -> torch.Tensor:
    """n uniform numbers in (0, 1) as fp64: (uint32 + 0.5) / 2^32."""
    return (uint32_stream(seed, stream, n, device).double() + 0.5) / 4294967296.0


def normal_bf16(seed: int, stream: int, shape, std: float, mean: float = 0.0,
                device="cpu") -> torch.Tensor:
    """A bf16 tensor of the given shape with values ~ mean + std * z, where z
    is the standardised 8-term Irwin-Hall variate described above."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    scale = torch.tensor(std / _IH_STD, dtype=torch.float32, device=device)
    key_a = _stream_key(seed, stream)
    key_b = key_a ^ 0x68E31DA4
    for start in range(0, n, _CHUNK):
        m = min(_CHUNK, n - start)
        idx = torch.arange(start, start + m, dtype=torch.int64, device=device)
        x = (idx * 0x9E3779B1) & _M32
        ha = fmix32(fmix32(x ^ key_a) ^ key_a)
        hb = fmix32(fmix32(x ^ key_b) ^ key_b)
        s = ((ha & 255) + ((ha >> 8) & 255) + ((ha >> 16) & 255) + (ha >> 24)
             + (hb & 255) + ((hb >> 8) & 255) + ((hb >> 16) & 255) + (hb >> 24))
        v = (s - _IH_MEAN).to(torch.float32) * scale
        if mean != 0.0:
            v = v + mean
        out[start:start + m] = v.to(torch.bfloat16)
    return out.view(*shape)


def uniform_ints(seed: int, stream: int, n: int, lo: int, hi: int,
                 device="cpu") -> torch.Tensor:
    """n integers in [lo, hi] (inclusive), int32."""
    span = hi - lo + 1
    return (uint32_stream(seed, stream, n, device) % span + lo).to(torch.int32)


def permutation(seed: int, stream: int, n: int, device="cpu") -> torch.Tensor:
    """A seeded permutation of range(n), int32 (stable sort of hash keys)."""
    keys = uint32_stream(seed, stream, n, device)
    return torch.sort(keys, stable=True).indices.to(torch.int32)


# --------------------------------------------------------------------------
# Model weights, natural (checkpoint) layout
# --------------------------------------------------------------------------
W_STD = 0.02


def layer_weights(shape: ModelShape, layer: int, seed: int = SEED_WEIGHTS,
                  device="cpu") -> dict:
    """One block's weights in checkpoint layout: projection matrices are
    [out_features, in_features] row-major; norm gains are 1 + N(0, 0.02^2)."""
    H, D, F = shape.hidden, shape.head_dim, shape.ffn
    base = 1000 + 64 * layer

    def g(i, shp, std=W_STD, mean=0.0):
        return normal_bf16(seed, base + i, shp, std, mean, device)

    w = {
        "wq": g(0, (shape.q_dim, H)),
        "wk": g(1, (shape.kv_dim, H)),
        "wv": g(2, (shape.kv_dim, H)),
        "wo": g(3, (H, shape.q_dim)),
        "wg": g(4, (F, H)),
        "wu": g(5, (F, H)),
        "wd": g(6, (H, F)),
        "g_attn": g(7, (H,), mean=1.0),
        "g_mlp": g(8, (H,), mean=1.0),
        "bq": None, "bk": None, "bv": None, "g_q": None, "g_k": None,
    }
    if shape.qkv_bias:
        w["bq"] = g(9, (shape.q_dim,))
        w["bk"] = g(10, (shape.kv_dim,))
        w["bv"] = g(11, (shape.kv_dim,))
    if shape.qk_norm:
        w["g_q"] = g(12, (D,), mean=1.0)
        w["g_k"] = g(13, (D,), mean=1.0)
    return w


def model_weights(shape: ModelShape, seed: int = SEED_WEIGHTS, device="cpu") -> dict:
    """All weights of the model: embed [V,H], lm_head [V,H] (None when tied),
    g_final [H] and the per-layer dicts."""
    return {
        "embed": normal_bf16(seed, 1, (shape.vocab, shape.hidden), W_STD, 0.0, device),
        "lm_head": None if shape.tie_embeddings else
        normal_bf16(seed, 2, (shape.vocab, shape.hidden), W_STD, 0.0, device),
        "g_final": normal_bf16(seed, 3, (shape.hidden,), W_STD, 1.0, device),
        "layers": [layer_weights(shape, l, seed, device) for l in range(shape.n_layers)],
    }


def param_count(shape: ModelShape) -> dict:
    """Parameter count of the shape, split the way nanoinfer's table splits it."""
    H, D, F, L, V = shape.hidden, shape.head_dim, shape.ffn, shape.n_layers, shape.vocab
    attn = H * shape.q_dim + 2 * H * shape.kv_dim + shape.q_dim * H
    if shape.qkv_bias:
        attn += shape.q_dim + 2 * shape.kv_dim
    mlp = 3 * H * F
    norms = 2 * H
    if shape.qk_norm:
        norms += 2 * D
    emb = V * H * (1 if shape.tie_embeddings else 2)
    total = emb + L * (attn + mlp + norms) + H
    return {"embeddings": emb, "mlp": L * mlp, "attention": L * attn,
            "norms": L * norms + H, "total": total}


# --------------------------------------------------------------------------
# Decode-time inputs
# --------------------------------------------------------------------------
def token_ids(n: int, vocab: int, seed: int = SEED_TOKENS, stream: int = 0,
              device="cpu") -> torch.Tensor:
    return uniform_ints(seed, stream, n, 0, vocab - 1, device)


def past_lengths(batch: int, lo: int, hi: int, seed: int = SEED_PAST,
                 device="cpu") -> torch.Tensor:
    return uniform_ints(seed, 0, batch, lo, hi, device)


def kv_std(shape: ModelShape) -> float:
    """Scale of a synthetic past K/V entry: the model's own K/V scale at init,
    0.02 * sqrt(H)."""
    return W_STD * math.sqrt(shape.hidden)


def synthetic_kv_rows(shape: ModelShape, layer: int, seq: int, kv_head: int,
                      which: int, n_pos: int, seed: int = SEED_KV,
                      device="cpu") -> torch.Tensor:
    """Past K (which=0) or V (which=1) of one (layer, sequence, kv head):
    bf16 [n_pos, D]. K is taken as already rotated."""
    stream = (((layer * 4096 + seq) * 64 + kv_head) * 2 + which)
    return normal_bf16(seed, stream, (n_pos, shape.head_dim), kv_std(shape),
                       0.0, device)


def block_tables(past: list, steps: int, block_size: int, seed: int = SEED_BLOCKS,
                 device="cpu"):
    """Paged-KV block tables. Sequence b needs ceil((past_b + steps) / bs)
    blocks; the physical pool is exactly that many blocks, handed out in a
    seeded shuffled order. Returns (table int32 [B, max_blocks] padded with -1,
    num_blocks)."""
    need = [-(-(p + steps) // block_size) for p in past]
    total = sum(need)
    perm = permutation(seed, 0, total, "cpu")
    maxb = max(need)
    table = torch.full((len(past), maxb), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table.to(device), total
