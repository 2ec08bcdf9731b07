"""GPU parity of nc_prefill (a prompt chunk as one causal forward pass: the
projections on the tensor cores, flash-style attention) against the CPU
oracle's chunked forward (oracle forward_chunk, which runs the chunk layer by
layer with every token's K/V cached before that layer's attention), through
the C ABI: the last token's logits and arg-max, every K/V slot the chunk
wrote, and greedy decode steps that continue from the prefilled cache."""
import numpy as np
import pytest
import torch

import oracle
from helpers import REL_L2_GATE, f32, rel_l2, token_agrees, weights_both
from transformer_decode_gb300 import nc, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nc.load()
    oracle.build()


def _fill(kv, okv, shape, seq, n, layers):
    """Synthetic past K/V (seed 4) in slots 0..n-1 of sequence seq, both caches."""
    for l in range(layers):
        for g in range(shape.n_kv_heads):
            if n == 0:
                continue
            kr = synth.synthetic_kv_rows(shape, l, seq, g, 0, n, device="cuda")
            vr = synth.synthetic_kv_rows(shape, l, seq, g, 1, n, device="cuda")
            kv.write_sequence(l, seq, g, kr, vr)
            okv.k[l, seq, g, :n] = f32(kr).reshape(n, -1)
            okv.v[l, seq, g, :n] = f32(vr).reshape(n, -1)


def _run(shape, T, start, paged, decode_steps=4, seq=1):
    if not paged and seq != 0:
        decode_steps = 0
    wd, wc = weights_both(shape)
    om = oracle.OracleModel(shape, wc)
    B = 2
    cap = start + T + decode_steps + 1
    model = nc.Model(shape, wd, max_batch=B, max_ctx=cap + 16)
    if paged:
        table, nblk = synth.block_tables([cap, cap], 1, 16)
        kv = nc.KVCache(shape, B, paged=True, block_table=table, num_blocks=nblk)
    else:
        kv = nc.KVCache(shape, B, max_ctx=cap)
    okv = om.new_kv(B, cap + 1)
    _fill(kv, okv, shape, seq, start, shape.n_layers)
    tokens = synth.token_ids(T, shape.vocab, stream=5).to(torch.int32)
    logits = torch.full((shape.vocab,), float("nan"), device="cuda")
    nxt = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    model.prefill(seq, tokens.cuda(), start, kv, logits, nxt)
    ol = om.forward_chunk(okv, seq, tokens.numpy(), start)
    torch.cuda.synchronize()
    assert model.device_status() == 0
    worst = rel_l2(f32(logits), ol[-1])
    assert worst < REL_L2_GATE, worst
    assert int(nxt[0]) == int(np.argmax(f32(logits)))
    assert token_agrees(int(nxt[0]), ol[-1], worst)
    # every slot the chunk wrote, every layer and kv head
    for l in range(shape.n_layers):
        for g in range(shape.n_kv_heads):
            for p in range(start, start + T):
                ks, vs = kv.slot_view(l, seq, g, p)
                assert rel_l2(f32(ks), okv.k[l, seq, g, p]) < 1e-4, (l, g, p)
                assert rel_l2(f32(vs), okv.v[l, seq, g, p]) < 1e-4, (l, g, p)
    # the other sequence's slots stay untouched (contiguous rows are separate)
    if not paged:
        assert not kv.k[:, 1 - seq].any() and not kv.v[:, 1 - seq].any()
    # decode continues from the prefilled cache (teacher-forced on the oracle's tokens)
    tok = np.array([int(np.argmax(ol[-1]))], np.int32)
    pos = start + T
    lg = torch.empty(1, shape.vocab, device="cuda")
    nx = torch.empty(1, dtype=torch.int32, device="cuda")
    okv1 = om.new_kv(1, cap + 1)
    okv1.k[:, 0] = okv.k[:, seq]
    okv1.v[:, 0] = okv.v[:, seq]
    for i in range(decode_steps):
        # the decode step addresses batch row 0: run it on a one-sequence view
        model.decode_step(torch.from_numpy(tok).cuda(), torch.tensor([pos], dtype=torch.int32).cuda(),
                          [pos], _row_view(kv, seq), lg, nx)
        ol2, on2 = om.decode_step(okv1, tok, np.array([pos], np.int32))
        torch.cuda.synchronize()
        e = rel_l2(f32(lg[0]), ol2[0])
        worst = max(worst, e)
        assert e < REL_L2_GATE, (i, e)
        assert token_agrees(int(nx[0]), ol2[0], e)
        tok = on2.astype(np.int32)
        pos += 1
    model.close()
    return worst


class _RowView:
    """Row `seq` of a paged cache as a one-sequence cache: the same block pool,
    the block table from that row on."""

    def __init__(self, kv, seq):
        self.kv, self.seq = kv, seq

    def struct(self):
        s = self.kv.struct()
        s.block_table = self.kv.table[self.seq:].data_ptr()
        s.block_table_host = self.kv.table_host[self.seq:].ctypes.data
        return s


def _row_view(kv, seq):
    """A cache a batch-1 decode step can continue sequence `seq` in: row 0 of
    any cache, or a paged row through its block table."""
    if seq == 0:
        return kv
    assert kv.paged, "contiguous rows other than 0 have no one-sequence view"
    return _RowView(kv, seq)


@pytest.mark.parametrize("shape,T,start,paged,seq", [
    (synth.TINY, 37, 0, False, 0),          # a chunk from position 0, ragged token tile
    (synth.TINY, 20, 5, True, 1),           # after 5 cached positions, second sequence, paged
    (synth.TINY_QKNORM, 70, 0, True, 1),    # q/k norm, D = 128, two token tiles
    (synth.TINY_QKNORM, 9, 130, False, 0),  # short chunk after a longer cache
    (synth.TINY, 16, 3, False, 1),          # the other contiguous row (no decode after)
])
def test_prefill_tiny(shape, T, start, paged, seq):
    worst = _run(shape, T, start, paged, seq=seq)
    print(f"prefill {shape.hidden} T={T} start={start}: worst rel-L2 {worst:.3e}")


def test_prefill_0p5b_prompt32():
    """The 0.5B model's 32-token prompt in one pass, then 8 greedy steps."""
    worst = _run(synth.QWEN2_0P5B, 32, 0, False, decode_steps=8, seq=0)
    print(f"prefill 0.5B T=32: worst rel-L2 {worst:.3e}")


def test_prefill_0p5b_chunk300_after_past():
    """300 tokens (three token tiles of 128, ragged) after 200 cached positions,
    paged, the second sequence."""
    worst = _run(synth.QWEN2_0P5B.with_layers(4), 300, 200, True, seq=1)
    print(f"prefill 0.5B (4 layers) T=300 after 200: worst rel-L2 {worst:.3e}")


def test_prefill_8b_shape_two_layers():
    worst = _run(synth.QWEN3_8B.with_layers(2), 130, 64, False, seq=0)
    print(f"prefill 8B shape (2 layers) T=130: worst rel-L2 {worst:.3e}")


def test_prefill_8b_shape_paired_blocks():
    """330 tokens at the 8B shape: 21 token blocks of 16 x 8 kv heads outnumber
    the SMs, so each attention CTA takes an early and a late block (the middle
    one alone, the last one partial)."""
    worst = _run(synth.QWEN3_8B.with_layers(2), 330, 0, False, decode_steps=2, seq=0)
    print(f"prefill 8B shape (2 layers) T=330, paired blocks: worst rel-L2 {worst:.3e}")


def test_prefill_rejects_bad_arguments():
    shape = synth.TINY
    wd, _ = weights_both(shape)
    model = nc.Model(shape, wd, max_batch=2, max_ctx=64)
    kv = nc.KVCache(shape, 2, max_ctx=64)
    logits = torch.empty(shape.vocab, device="cuda")
    toks = torch.zeros(40, dtype=torch.int32, device="cuda")
    E = {n: nc.STATUS.index(n) for n in nc.STATUS}
    with pytest.raises(nc.NCError) as e:
        model.prefill(0, toks, 30, kv, logits)     # 30 + 40 > 64 slots
    assert e.value.code == E["NC_ERR_POSITION"]
    with pytest.raises(nc.NCError) as e:
        model.prefill(2, toks, 0, kv, logits)      # sequence 2 of a 2-sequence cache
    assert e.value.code == E["NC_ERR_CAPACITY"]
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nc.NCError) as e:
        model.prefill(0, toks, 0, kv, logits, scratch=small)
    assert e.value.code == E["NC_ERR_CAPACITY"]
    assert not kv.k.any()
    model.close()
