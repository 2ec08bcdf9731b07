"""nc_attn_decode_static: the decode attention for callers that cannot
allocate device memory (for example code that runs while a stream is in
global-mode graph capture, or whose device memory belongs to a framework
allocator). It keeps its scratch in a static device array instead of a
model's cudaMalloc'd workspace; its results must equal nc_attn_decode's.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import REL_L2_GATE, bf16_bits, f32, rel_l2, to_device
from transformer_decode_gb300 import nc, synth

pytestmark = pytest.mark.gpu


def _setup(shape, positions, paged, kv_dtype):
    B = len(positions)
    model = nc.Model(shape, to_device(synth.model_weights(shape)), max_batch=B,
                     max_ctx=max(positions) + 17)
    if paged:
        table, nblk = synth.block_tables(positions, 1, 16)
        kv = nc.KVCache(shape, B, paged=True, block_table=table, num_blocks=nblk, dtype=kv_dtype)
    else:
        kv = nc.KVCache(shape, B, max_ctx=max(positions) + 17, dtype=kv_dtype)
    rows = {}
    for b, p in enumerate(positions):
        for g in range(shape.n_kv_heads):
            kr = synth.synthetic_kv_rows(shape, 0, b, g, 0, p + 1, device="cuda")
            vr = synth.synthetic_kv_rows(shape, 0, b, g, 1, p + 1, device="cuda")
            kv.write_sequence(0, b, g, kr, vr)
            rows[b, g] = (kr, vr)
    gen = torch.Generator().manual_seed(sum(positions) + shape.head_dim)
    q = (torch.randn(B, shape.q_dim, generator=gen) * 0.7).cuda()
    return model, kv, q, rows


def _oracle_attention(shape, positions, q, rows, kv_dtype):
    """The CPU oracle's attention of every (sequence, query head) over slots
    0..position, on the K/V rows as the cache holds them."""
    D, G = shape.head_dim, shape.group
    held = bf16_bits if kv_dtype == torch.bfloat16 else f32
    out = np.zeros((len(positions), shape.q_dim), np.float32)
    for b, p in enumerate(positions):
        for h in range(shape.n_q_heads):
            kr, vr = rows[b, h // G]
            out[b, h * D:(h + 1) * D] = oracle.attention_head(
                f32(q[b, h * D:(h + 1) * D]), held(kr).reshape(p + 1, D),
                held(vr).reshape(p + 1, D))
    return out


def test_static_scratch_matches_model_workspace_two_calls():
    """Two calls in a row with different batch, positions and layouts: the
    second runs on scratch the first left behind. Each result equals
    nc_attn_decode's and the CPU oracle's, and the static status word reads
    0 (no device-side error)."""
    cases = [
        (dataclasses.replace(synth.QWEN2_0P5B.with_layers(1), vocab=512), [17, 1, 300], False,
         torch.float32),
        (dataclasses.replace(synth.QWEN3_8B.with_layers(1), vocab=512), [4096], True,
         torch.bfloat16),
    ]
    for shape, positions, paged, kv_dtype in cases:
        model, kv, q, rows = _setup(shape, positions, paged, kv_dtype)
        B = len(positions)
        pos_h = torch.tensor(positions, dtype=torch.int32)
        pos_d = pos_h.cuda()
        want = torch.full((B, shape.q_dim), float("nan"), device="cuda")
        got = torch.full((B, shape.q_dim), float("nan"), device="cuda")
        model.attn_decode(0, q, pos_d, pos_h, kv, want)
        nc.attn_decode_static(shape, 0, q, pos_d, pos_h, kv, got)
        torch.cuda.synchronize()
        assert nc.attn_decode_static_status() == 0
        g, w = got.cpu().numpy(), want.cpu().numpy()
        assert np.isfinite(g).all()
        assert rel_l2(g, w) < REL_L2_GATE / 10
        ref = _oracle_attention(shape, positions, q, rows, kv_dtype)
        for b in range(B):
            assert rel_l2(g[b], ref[b]) < REL_L2_GATE / 10, (b, rel_l2(g[b], ref[b]))
        model.close()


def test_static_scratch_rejects_oversized_requests():
    """A request whose partials exceed the static array is refused before any
    launch, with NC_ERR_CAPACITY."""
    # 512 query heads x at least 16 splits (one per sequence) x 130 partial
    # floats = 1,064,960 floats, beyond the 2^20 of the array
    shape = dataclasses.replace(synth.QWEN2_0P5B.with_layers(1), n_q_heads=512, n_kv_heads=64,
                                head_dim=128, vocab=512)
    B = 16
    table = torch.zeros(B, 4, dtype=torch.int32)
    kv = nc.KVCache(shape, B, paged=True, block_table=table, num_blocks=1)
    q = torch.zeros(B, shape.q_dim, device="cuda")
    out = torch.zeros(B, shape.q_dim, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32)
    with pytest.raises(nc.NCError) as e:
        nc.attn_decode_static(shape, 0, q, pos.cuda(), pos, kv, out)
    assert e.value.code == nc.STATUS.index("NC_ERR_CAPACITY")
    assert b"scratch" in nc.load().nc_last_error_message()


def test_static_tickets_reject_oversized_requests():
    """More (sequence, kv head) pairs than static merge counters: refused
    before any launch, with NC_ERR_CAPACITY."""
    shape = dataclasses.replace(synth.QWEN2_0P5B.with_layers(1), n_q_heads=128, n_kv_heads=128,
                                head_dim=64, vocab=512)
    B = 16
    table = torch.zeros(B, 4, dtype=torch.int32)
    kv = nc.KVCache(shape, B, paged=True, block_table=table, num_blocks=1)
    q = torch.zeros(B, shape.q_dim, device="cuda")
    out = torch.zeros(B, shape.q_dim, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32)
    with pytest.raises(nc.NCError) as e:
        nc.attn_decode_static(shape, 0, q, pos.cuda(), pos, kv, out)
    assert e.value.code == nc.STATUS.index("NC_ERR_CAPACITY")
    assert b"tickets" in nc.load().nc_last_error_message()
