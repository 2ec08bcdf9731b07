"""GPU parity of whole blocks and whole decode steps against the CPU oracle,
through the C ABI (nc_block_forward, nc_decode_step)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from helpers import REL_L2_GATE, bf16_bits, f32, rel_l2, to_device, token_agrees, weights_both
from transformer_decode_gb300 import nc, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nc.load()
    oracle.build()


def test_generator_same_bits_on_gpu_and_cpu():
    a = synth.normal_bf16(0, 42, (3, 1_000_003), 0.02, device="cuda")
    b = synth.normal_bf16(0, 42, (3, 1_000_003), 0.02, device="cpu")
    assert torch.equal(a.cpu().view(torch.int16), b.view(torch.int16))
    assert torch.equal(synth.token_ids(999, 151936, device="cuda").cpu(), synth.token_ids(999, 151936))


def _fill_past(kv, okv, shape, positions, layers):
    """Synthetic past K/V (seed 4) for slots 0..p-1 of every sequence, written
    into both caches."""
    for l in range(layers):
        for b, p in enumerate(positions):
            if p == 0:
                continue
            for g in range(shape.n_kv_heads):
                kr = synth.synthetic_kv_rows(shape, l, b, g, 0, p, device="cuda")
                vr = synth.synthetic_kv_rows(shape, l, b, g, 1, p, device="cuda")
                kv.write_sequence(l, b, g, kr, vr)
                if okv.bf16:
                    okv.k[l, b, g, :p] = bf16_bits(kr).reshape(p, -1)
                    okv.v[l, b, g, :p] = bf16_bits(vr).reshape(p, -1)
                else:
                    okv.k[l, b, g, :p] = f32(kr).reshape(p, -1)
                    okv.v[l, b, g, :p] = f32(vr).reshape(p, -1)


# ------------------------------------------------------------------ one block (C0 shape)
@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("kv_bf16", [False, True])
def test_block_forward_0p5b_past16(paged, kv_bf16):
    shape = dataclasses.replace(synth.QWEN2_0P5B.with_layers(1), vocab=1024)
    wd, wc = weights_both(shape)
    model = nc.Model(shape, wd, max_batch=1, max_ctx=64)
    om = oracle.OracleModel(shape, wc)
    pos = 16
    kdt = torch.bfloat16 if kv_bf16 else torch.float32
    if paged:
        table, nblk = synth.block_tables([pos], 1, 16)
        kv = nc.KVCache(shape, 1, paged=True, block_table=table, num_blocks=nblk, dtype=kdt)
    else:
        kv = nc.KVCache(shape, 1, max_ctx=64, dtype=kdt)
    okv = om.new_kv(1, 64, bf16=kv_bf16)
    _fill_past(kv, okv, shape, [pos], 1)
    x0 = synth.normal_bf16(0, 9999, (1, shape.hidden), 1.0).float()
    x = x0.cuda()
    p = torch.tensor([pos], dtype=torch.int32)
    model.block_forward(0, x, p.cuda(), p, kv)
    torch.cuda.synchronize()
    ref = om.block_decode(0, okv, 0, pos, x0[0].numpy())
    assert rel_l2(f32(x[0]), ref) < REL_L2_GATE / 10
    widen = oracle.bf16_to_f32 if kv_bf16 else (lambda a: a)
    for g in range(shape.n_kv_heads):
        ks, vs = kv.slot_view(0, 0, g, pos)
        tol = 1e-3 if kv_bf16 else 1e-5
        assert rel_l2(f32(ks), widen(okv.k[0, 0, g, pos])) < tol
        assert rel_l2(f32(vs), widen(okv.v[0, 0, g, pos])) < tol
    model.close()


def test_block_forward_w8a8_codes_on_identical_input():
    """W8A8 blocks of the 0.5B shape at 512 past positions, each run on the
    same fp32 input on both sides (nc_block_forward and the oracle's block,
    layer by layer through the model): every activation code of the four
    products equals the oracle's except boundary cases (neighbours, from a
    quotient within CODE_BOUNDARY_TOL of .5; counted and checked), and with
    those forced each block output is within 5e-4."""
    shape = synth.QWEN2_0P5B
    wd, wc = weights_both(shape)
    model = nc.Model(shape, wd, max_batch=1, max_ctx=600, w8a8=True)
    om = oracle.OracleModel(shape, wc, w8a8=True)
    pos = 512
    kv = nc.KVCache(shape, 1, max_ctx=600)
    okv = om.new_kv(1, 600)
    _fill_past(kv, okv, shape, [pos], shape.n_layers)
    H, qd, F = shape.hidden, shape.q_dim, shape.ffn
    per_layer = 2 * H + qd + F
    codes = torch.empty(shape.n_layers * per_layer, dtype=torch.int8, device="cuda")
    model.debug_w8a8_codes(codes)
    x = synth.normal_bf16(0, 9999, (shape.hidden,), 1.0).float().numpy()
    p = torch.tensor([pos], dtype=torch.int32)
    worst, nd = 0.0, 0
    for l in range(shape.n_layers):
        xg = torch.from_numpy(x).view(1, -1).cuda()
        model.block_forward(l, xg, p.cuda(), p, kv)
        torch.cuda.synchronize()
        c = codes.cpu().numpy()[l * per_layer:(l + 1) * per_layer]
        qkv, o, gu, d = c[:H], c[H:H + qd], c[H + qd:2 * H + qd], c[2 * H + qd:]
        force = np.concatenate([qkv, qkv, qkv, o, gu, gu, d])
        tr = oracle.OracleTrace(5 * H + qd + F, 0, force_codes=force)
        ref = om.block_decode(l, okv, 0, pos, x, trace=tr)
        assert tr.complete
        nd += _check_forced_codes(tr.codes, force, tr.quot)
        e = rel_l2(f32(xg[0]), ref)
        worst = max(worst, e)
        assert e < REL_L2_GATE, (l, e)
        x = ref  # the next block starts from the oracle's output on both sides
    model.debug_w8a8_codes(None)
    model.close()
    print(f"W8A8 blocks: worst rel-L2 {worst:.3e}, boundary codes forced {nd}")


# ------------------------------------------------------------------ greedy decode
def _greedy_compare(shape, wd, wc, prompt, steps, batch=1, past=None, paged=False,
                    use_graph=True, gate=REL_L2_GATE, staged=False, int4_group=0):
    """Teacher-forced greedy decode: both sides consume the oracle's token.
    Every step's logits within `gate` (rel-L2) and the greedy tokens equal
    under the near-tie rule. Returns the worst logit rel-L2 seen. (Paths with
    a rounding step inside the model, W8A8 codes or bf16 K/V, use
    _traced_compare.)"""
    om = oracle.OracleModel(shape, wc, int4_group=int4_group)
    past = past or [0] * batch
    n_total = len(prompt[0]) + steps if prompt is not None else steps
    max_ctx = max(past) + n_total + 1
    model = nc.Model(shape, wd, max_batch=batch, max_ctx=max_ctx + 16, int4_group=int4_group)
    if paged:
        table, nblk = synth.block_tables(past, n_total, 16)
        kv = nc.KVCache(shape, batch, paged=True, block_table=table, num_blocks=nblk)
    else:
        kv = nc.KVCache(shape, batch, max_ctx=max_ctx)
    okv = om.new_kv(batch, max_ctx)
    _fill_past(kv, okv, shape, past, shape.n_layers)
    logits = torch.empty(batch, shape.vocab, device="cuda")
    nxt = torch.empty(batch, dtype=torch.int32, device="cuda")
    pos = np.array(past, np.int32)
    tok = np.array([prompt[b][0] for b in range(batch)] if prompt is not None else
                   synth.token_ids(batch, shape.vocab, stream=77).tolist(), np.int32)
    worst = 0.0
    n_prompt = len(prompt[0]) if prompt is not None else 0
    tok_d = torch.empty(batch, dtype=torch.int32, device="cuda")
    pos_d = torch.empty(batch, dtype=torch.int32, device="cuda")
    for i in range(n_total):
        tok_d.copy_(torch.from_numpy(tok))
        pos_d.copy_(torch.from_numpy(pos))
        model.decode_step(tok_d, pos_d, pos, kv, logits, nxt, use_graph=use_graph, staged=staged)
        ol, on = om.decode_step(okv, tok, pos)
        torch.cuda.synchronize()
        gl, gn = logits.cpu().numpy(), nxt.cpu().numpy()
        for b in range(batch):
            e = rel_l2(gl[b], ol[b])
            worst = max(worst, e)
            assert e < gate, (i, b, e, gate)
            assert gn[b] == int(np.argmax(gl[b]))
            assert token_agrees(int(gn[b]), ol[b], e), (i, b, gn[b], on[b])
        pos = pos + 1
        if i + 1 < n_prompt:
            tok = np.array([prompt[b][i + 1] for b in range(batch)], np.int32)
        else:
            tok = on.astype(np.int32)
    assert model.device_status() == 0
    model.close()
    return worst


# Rounding steps inside the model (nanoinfer "Quantization": activation codes
# rounded half away from zero; bf16 K/V rounded to nearest even on store) are
# discontinuities: two correct fp32 evaluations whose inputs differ in the
# last bits can round a value that sits on a boundary to neighbouring results.
# _traced_compare therefore runs the oracle with the GPU's rounded values
# forced in (oracle.OracleTrace) and checks each forced value that differs from
# the oracle's own: it must be the neighbouring code (or bf16 value), and the
# oracle's unrounded value must lie within these distances of the boundary
# between the two. The GPU and oracle inputs of a rounding step agree to fp32
# drift: relative 4e-6 or better of the vector's scale over a whole model on
# the CUDA-core paths (the measured logit rel-L2), and 3e-5 on the tensor-core
# path of batch 9..16 (its activations enter as bf16 hi / lo planes: 2^-18 of
# each input element is lost). A quotient v / s of at most 127 code units
# then moves by at most 127 * 2 * 4e-6 = 1e-3 = 2^-10 units (W8A8 runs on the
# CUDA cores), and a K/V value by 3e-5 of its head vector's largest
# magnitude (the bound below leaves a factor 8).
CODE_BOUNDARY_TOL = 2.0 ** -10   # code units from a .5 boundary
KV_BOUNDARY_TOL = 2.0 ** -12     # distance from the rounding interval, in units of the
                                 # head vector's largest magnitude


def _check_forced_codes(own, forced, quot):
    """Differing codes: neighbours, from a quotient within CODE_BOUNDARY_TOL
    of the .5 boundary between them. Returns the number of differences."""
    d = np.nonzero(own != forced)[0]
    if d.size:
        assert np.all(np.abs(own[d].astype(np.int32) - forced[d].astype(np.int32)) == 1), d[:8]
        q = np.abs(quot[d].astype(np.float64))
        dist = np.abs(q - np.floor(q) - 0.5)
        assert np.all(dist <= CODE_BOUNDARY_TOL), (d[:8], quot[d][:8], dist.max())
    return int(d.size)


def _check_forced_kv(own, forced, val, D):
    """Differing bf16 K/V bits: the GPU's stored value must be the rounding
    (to nearest even) of a value within KV_BOUNDARY_TOL x the largest
    magnitude of its head vector (D values) from the oracle's fp32 value: the
    drift of an fp32 evaluation is relative to the vector's scale, so a small
    element may sit several bf16 steps from the oracle's and still be a
    correct result. Returns the number of differences."""
    d = np.nonzero(own != forced)[0]
    if d.size:
        vmax = np.abs(val.astype(np.float64)).reshape(-1, D).max(axis=1)[d // D]
        g = oracle.bf16_to_f32(forced[d]).astype(np.float64)
        # the interval of fp32 values that round to g: half a bf16 step each way
        e = np.floor(np.log2(np.maximum(np.abs(g), 2.0 ** -126)))
        half = 2.0 ** (e - 8)
        v = val[d].astype(np.float64)
        gap = np.maximum(np.abs(v - g) - half, 0.0)
        assert np.all(gap <= KV_BOUNDARY_TOL * vmax), (d[:8], v[:8], g[:8])
    return int(d.size)


def _traced_compare(shape, wd, wc, steps, batch=1, past=None, paged=False, w8a8=False,
                    kv_bf16=False, prompt=None, staged=False):
    """Teacher-forced greedy decode with the oracle's rounding steps forced
    to the GPU's results (each difference checked to be a boundary case, see
    above), so both sides compute on identical codes and cache bits: then
    every step's logits meet the plain 5e-4 gate and the tokens agree.
    Returns (worst logit rel-L2, differing codes, differing K/V values)."""
    b32 = w8a8 == "b32"
    om = oracle.OracleModel(shape, wc, w8a8=bool(w8a8), act_block=32 if b32 else 0,
                            int8_embed=b32)
    past = past or [0] * batch
    n_total = (len(prompt[0]) if prompt is not None else 0) + steps
    max_ctx = max(past) + n_total + 1
    model = nc.Model(shape, wd, max_batch=batch, max_ctx=max_ctx + 16, w8a8=w8a8)
    kdt = torch.bfloat16 if kv_bf16 else torch.float32
    if paged:
        table, nblk = synth.block_tables(past, n_total, 16)
        kv = nc.KVCache(shape, batch, paged=True, block_table=table, num_blocks=nblk, dtype=kdt)
    else:
        kv = nc.KVCache(shape, batch, max_ctx=max_ctx, dtype=kdt)
    okv = om.new_kv(batch, max_ctx, bf16=kv_bf16)
    _fill_past(kv, okv, shape, past, shape.n_layers)
    H, qd, F, L = shape.hidden, shape.q_dim, shape.ffn, shape.n_layers
    D, Hkv = shape.head_dim, shape.n_kv_heads
    per_layer = batch * (2 * H + qd + F)
    codes = scales = None
    if w8a8:
        codes = torch.empty(L * per_layer + (batch * H if b32 else 0), dtype=torch.int8,
                            device="cuda")
        model.debug_w8a8_codes(codes)
    # per sequence and layer q, k, v, o, gate, up, down; the blocked mode's
    # int8 head after the layers
    n_codes = batch * (L * (5 * H + qd + F) + (H if b32 else 0)) if w8a8 else 0
    n_kv = batch * L * Hkv * 2 * D if kv_bf16 else 0
    logits = torch.empty(batch, shape.vocab, device="cuda")
    nxt = torch.empty(batch, dtype=torch.int32, device="cuda")
    pos = np.array(past, np.int32)
    n_prompt = len(prompt[0]) if prompt is not None else 0
    tok = np.array([prompt[b][0] for b in range(batch)] if prompt is not None else
                   synth.token_ids(batch, shape.vocab, stream=77).tolist(), np.int32)
    tok_d = torch.empty(batch, dtype=torch.int32, device="cuda")
    pos_d = torch.empty(batch, dtype=torch.int32, device="cuda")
    worst, n_code_diff, n_kv_diff = 0.0, 0, 0
    for i in range(n_total):
        tok_d.copy_(torch.from_numpy(tok))
        pos_d.copy_(torch.from_numpy(pos))
        model.decode_step(tok_d, pos_d, pos, kv, logits, nxt, staged=staged)
        torch.cuda.synchronize()
        force_codes = force_kv = None
        if w8a8:
            call = codes.cpu().numpy()
            c = call[:L * per_layer].reshape(L, per_layer)
            parts = []
            for b in range(batch):
                for l in range(L):
                    qkv_b = c[l, b * H:(b + 1) * H]
                    o0 = batch * H
                    o_b = c[l, o0 + b * qd:o0 + (b + 1) * qd]
                    g0 = o0 + batch * qd
                    gu_b = c[l, g0 + b * H:g0 + (b + 1) * H]
                    d0 = g0 + batch * H
                    d_b = c[l, d0 + b * F:d0 + (b + 1) * F]
                    parts += [qkv_b, qkv_b, qkv_b, o_b, gu_b, gu_b, d_b]
                if b32:
                    parts.append(call[L * per_layer + b * H:L * per_layer + (b + 1) * H])
            force_codes = np.concatenate(parts)
        if kv_bf16:
            rows = []
            for b in range(batch):
                for l in range(L):
                    for g in range(Hkv):
                        ks, vs = kv.slot_view(l, b, g, int(pos[b]))
                        rows += [bf16_bits(ks), bf16_bits(vs)]
            force_kv = np.concatenate(rows)
        tr = oracle.OracleTrace(n_codes, n_kv, force_codes, force_kv)
        ol, on = om.decode_step(okv, tok, pos, trace=tr)
        assert tr.complete
        if w8a8:
            n_code_diff += _check_forced_codes(tr.codes, force_codes, tr.quot)
        if kv_bf16:
            n_kv_diff += _check_forced_kv(tr.kv_own, force_kv, tr.kv_val, D)
        gl, gn = logits.cpu().numpy(), nxt.cpu().numpy()
        for b in range(batch):
            e = rel_l2(gl[b], ol[b])
            worst = max(worst, e)
            assert e < REL_L2_GATE, (i, b, e)
            assert gn[b] == int(np.argmax(gl[b]))
            assert token_agrees(int(gn[b]), ol[b], e), (i, b, gn[b], on[b])
        pos = pos + 1
        if i + 1 < n_prompt:
            tok = np.array([prompt[b][i + 1] for b in range(batch)], np.int32)
        else:
            tok = on.astype(np.int32)
    if w8a8:
        model.debug_w8a8_codes(None)
    assert model.device_status() == 0
    model.close()
    return worst, n_code_diff, n_kv_diff


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_QKNORM])
@pytest.mark.parametrize("path", ["persistent", "staged-graph", "staged-eager"])
def test_decode_tiny(shape, path):
    """Both step paths: the persistent kernel (default at these sizes) and the
    per-stage kernels, replayed from a graph or launched directly."""
    wd, wc = weights_both(shape)
    prompt = [synth.token_ids(5, shape.vocab, stream=11).tolist()]
    _greedy_compare(shape, wd, wc, prompt, steps=20, use_graph=path != "staged-eager",
                    staged=path != "persistent")


def test_decode_path_dispatch():
    """nc_decode_path reports the implementation a step would run: the
    persistent kernel up to batch 4 at any cache length, else the stage
    kernels; NC_STEP_STAGED forces the latter."""
    shape = synth.TINY
    wd, _ = weights_both(shape)
    model = nc.Model(shape, wd, max_batch=8, max_ctx=8192)
    small = nc.KVCache(shape, 8, max_ctx=64)
    big = nc.KVCache(shape, 1, max_ctx=8192)
    assert model.decode_path(1, small) == "persistent"
    assert model.decode_path(4, small) == "persistent"
    assert model.decode_path(5, small) == "staged"
    assert model.decode_path(1, small, staged=True) == "staged"
    assert model.decode_path(1, big) == "persistent"
    model.close()


def test_decode_group6_d128_runs_staged():
    """Six query heads per kv head at D = 128 are beyond the persistent
    kernel's attention instances (groups of at most 4 at that head size): the
    step runs on the stage kernels, and its tokens still match the oracle."""
    shape = dataclasses.replace(synth.TINY_QKNORM, n_q_heads=6, n_kv_heads=1)
    wd, wc = weights_both(shape)
    model = nc.Model(shape, wd, max_batch=1, max_ctx=64)
    assert model.decode_path(1, nc.KVCache(shape, 1, max_ctx=64)) == "staged"
    model.close()
    _greedy_compare(shape, wd, wc, None, steps=6, past=[20])


@pytest.mark.parametrize("batch", [2, 4])
def test_decode_tiny_persistent_batch(batch):
    """The persistent kernel at batch 2 and 4, mixed positions."""
    shape = synth.TINY
    wd, wc = weights_both(shape)
    _greedy_compare(shape, wd, wc, None, steps=10, batch=batch, past=[0, 7, 19, 3][:batch])


@pytest.mark.parametrize("paged", [False, True])
def test_decode_tiny_persistent_splits(paged):
    """Attention split over positions (scans longer than 128 positions, one
    split per 128 positions up to the grid's share of each (sequence, kv
    head); the last split to finish merges): past lengths 300, 200, 129 and
    5 give 3, 2, 2 and 1 splits."""
    shape = synth.TINY
    wd, wc = weights_both(shape)
    _greedy_compare(shape, wd, wc, None, steps=6, batch=4, past=[300, 200, 129, 5], paged=paged)


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_QKNORM])
@pytest.mark.parametrize("batch,paged", [(9, False), (16, True)])
def test_decode_tiny_tensor_cores(shape, batch, paged):
    """Batch 9..16: the projections and the LM head run on the tensor cores
    (tcgen05 with the accumulator in tensor memory, activations as bf16
    hi / lo planes); ragged output rows (TINY_QKNORM's 328-token vocabulary,
    2.6 tiles of 128) and a batch that fills 9 of the 16 token columns."""
    wd, wc = weights_both(shape)
    past = [(7 * b) % 37 for b in range(batch)]
    _greedy_compare(shape, wd, wc, None, steps=6, batch=batch, past=past, paged=paged)


def test_decode_tiny_batch_paged():
    shape = synth.TINY
    wd, wc = weights_both(shape)
    _greedy_compare(shape, wd, wc, None, steps=12, batch=5, past=[0, 3, 16, 31, 70], paged=True)


@pytest.mark.parametrize("staged", [False, True])
def test_decode_0p5b_prompt32_greedy64(staged):
    """The full 24-layer 0.5B-shaped model: a 32-token prompt then 64 greedy
    tokens, contiguous cache; the persistent kernel and the per-stage path."""
    shape = synth.QWEN2_0P5B
    wd, wc = weights_both(shape)
    prompt = [synth.token_ids(32, shape.vocab).tolist()]
    worst = _greedy_compare(shape, wd, wc, prompt, steps=64, staged=staged)
    print(f"0.5B greedy (staged {staged}): worst logit rel-L2 {worst:.3e}")


def test_decode_0p5b_w8a8_past512():
    """The W8A8 configuration at full size: 512 past positions, 64 greedy
    steps. Every activation code of every step equals the oracle's except
    boundary cases (each checked), and with those forced the logits meet the
    plain 5e-4 gate at every step. The integer arithmetic itself is checked
    bit-exact in test_gpu_stages."""
    shape = synth.QWEN2_0P5B
    wd, wc = weights_both(shape)
    worst, nd, _ = _traced_compare(shape, wd, wc, steps=64, past=[512], w8a8=True)
    print(f"0.5B W8A8: worst logit rel-L2 {worst:.3e}, boundary codes forced {nd}")


@pytest.mark.parametrize("shape,past,steps", [(synth.TINY, 0, 12),
                                               (synth.QWEN2_0P5B, 512, 64)])
def test_decode_w8a8_b32(shape, past, steps):
    """W8A8 with activations in blocks of 32 and the int8 embedding as the
    tied head (NC_INT8_B32) against the oracle's same mode: every activation
    code, the head's included, equals the oracle's except boundary cases
    (checked and forced), and the logits meet the plain 5e-4 gate."""
    wd, wc = weights_both(shape)
    worst, nd, _ = _traced_compare(shape, wd, wc, steps=steps, past=[past], w8a8="b32")
    print(f"W8A8 blocks of 32 ({shape.hidden}): worst logit rel-L2 {worst:.3e}, "
          f"boundary codes forced {nd}")


@pytest.mark.parametrize("shape,group,past,steps", [(synth.TINY, 32, 0, 12),
                                                     (synth.TINY, 128, 5, 12),
                                                     (synth.QWEN2_0P5B, 128, 512, 64)])
def test_decode_int4(shape, group, past, steps):
    """INT4 group-wise projections (NC_INT4_G32 / NC_INT4_G128) against the
    oracle's INT4 mode. Only weights are quantised (on the device, by the
    same operations as the oracle's quantiser), so the plain 5e-4 gate holds."""
    wd, wc = weights_both(shape)
    worst = _greedy_compare(shape, wd, wc, None, steps=steps, past=[past], int4_group=group)
    print(f"INT4 group {group} ({shape.hidden}): worst logit rel-L2 {worst:.3e}")


def test_decode_0p5b_batch16_paged():
    """The batch-16 paged configuration at full size: 16 sequences with past
    lengths U[256, 4096], shuffled block tables, 8 teacher-forced steps."""
    shape = synth.QWEN2_0P5B
    wd, wc = weights_both(shape)
    past = synth.past_lengths(16, 256, 4096).tolist()
    worst = _greedy_compare(shape, wd, wc, None, steps=8, batch=16, past=past, paged=True)
    print(f"0.5B B16 paged: worst logit rel-L2 {worst:.3e}")


def test_decode_0p5b_batch16_paged_bf16_kv():
    """The same with a bf16 cache: each step's stored K/V equal the oracle's
    except boundary cases (checked), forced so the plain gate holds."""
    shape = synth.QWEN2_0P5B
    wd, wc = weights_both(shape)
    past = synth.past_lengths(16, 256, 4096).tolist()
    worst, _, nd = _traced_compare(shape, wd, wc, steps=4, batch=16, past=past, paged=True,
                                   kv_bf16=True)
    print(f"0.5B B16 paged bf16 KV: worst logit rel-L2 {worst:.3e}, boundary K/V forced {nd}")


@pytest.mark.parametrize("staged", [False, True])
def test_decode_0p5b_bf16_kv_prompt(staged):
    """bf16 K/V from position 0 (an 8-token prompt, then 8 greedy tokens), on
    the persistent kernel and the stage kernels: stored values equal the
    oracle's except boundary cases (checked and forced)."""
    shape = synth.QWEN2_0P5B
    wd, wc = weights_both(shape)
    prompt = [synth.token_ids(8, shape.vocab).tolist()]
    worst, _, nd = _traced_compare(shape, wd, wc, steps=8, kv_bf16=True, prompt=prompt,
                                   staged=staged)
    print(f"0.5B bf16 KV (staged {staged}): worst logit rel-L2 {worst:.3e}, "
          f"boundary K/V forced {nd}")


@pytest.mark.parametrize("staged", [False, True])
def test_decode_8b_shape_two_layers_past4096(staged):
    """Two 8B-shaped layers at 4096 past positions: the persistent kernel
    (the attention split over the whole grid, merged by the last split) and
    the per-stage kernels."""
    shape = synth.QWEN3_8B.with_layers(2)
    wd, wc = weights_both(shape)
    worst = _greedy_compare(shape, wd, wc, None, steps=3, past=[4096], staged=staged)
    print(f"8B-shaped (2 layers, staged {staged}): worst logit rel-L2 {worst:.3e}")


def test_decode_8b_shape_full_past4096():
    """The whole 36-layer 8B-shaped model at 4096 past positions, 4
    teacher-forced greedy steps on the path the benchmark times (the
    persistent kernel)."""
    shape = synth.QWEN3_8B
    wd, wc = weights_both(shape)
    worst = _greedy_compare(shape, wd, wc, None, steps=4, past=[4096])
    print(f"8B-shaped (36 layers): worst logit rel-L2 {worst:.3e}")


def test_invalid_inputs_leave_state_untouched():
    shape = synth.TINY
    wd, _ = weights_both(shape)
    model = nc.Model(shape, wd, max_batch=2, max_ctx=32)
    kv = nc.KVCache(shape, 2, max_ctx=32)
    logits = torch.empty(2, shape.vocab, device="cuda")
    tok = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(nc.NCError) as e:
        model.decode_step(tok, tok, np.array([0, 32], np.int32), kv, logits)
    assert e.value.code == nc.STATUS.index("NC_ERR_POSITION")
    with pytest.raises(nc.NCError) as e:
        model.decode_step(torch.zeros(3, dtype=torch.int32, device="cuda"),
                          torch.zeros(3, dtype=torch.int32, device="cuda"), [0, 0, 0], kv,
                          torch.empty(3, shape.vocab, device="cuda"))
    assert e.value.code == nc.STATUS.index("NC_ERR_CAPACITY")
    big = nc.KVCache(shape, 2, max_ctx=64)
    with pytest.raises(nc.NCError) as e:
        model.decode_step(tok, tok, [0, 0], big, logits)
    assert e.value.code == nc.STATUS.index("NC_ERR_CAPACITY")
    # paged: a hole in the block table is refused on the host
    table = torch.tensor([[0, 1], [2, -1]], dtype=torch.int32)
    pk = nc.KVCache(shape, 2, paged=True, block_table=table, num_blocks=3)
    with pytest.raises(nc.NCError) as e:
        model.decode_step(tok, tok, [3, 17], pk, logits)
    assert e.value.code == nc.STATUS.index("NC_ERR_POSITION")
    assert not kv.k.any() and not pk.k.any()
    # an out-of-range token id is caught on the device without a fault
    bad = torch.tensor([shape.vocab + 5, 1], dtype=torch.int32, device="cuda")
    model.decode_step(bad, tok, [0, 0], kv, logits, use_graph=False)
    torch.cuda.synchronize()
    assert model.device_status() != 0
    model.close()
