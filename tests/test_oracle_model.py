"""Model-level pins of the oracle on tiny shapes: grouped-query repeat (not
tile), the causal mask, the KV-cache invariant under five chunkings, the
planted position bug, and fp32 against fp64 agreement."""
import numpy as np
import pytest
import torch

from transformer_decode_gb300 import synth


def _rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.fixture(scope="module")
def tiny(orc):
    w = synth.model_weights(synth.TINY, seed=0)
    return orc.OracleModel(synth.TINY, w), w


@pytest.fixture(scope="module")
def tiny_qk(orc):
    w = synth.model_weights(synth.TINY_QKNORM, seed=0)
    return orc.OracleModel(synth.TINY_QKNORM, w), w


def _bf16(t):
    return torch.tensor(t, dtype=torch.float32).to(torch.bfloat16)


def test_gqa_repeats_kv_heads(orc):
    """nanoinfer "Model architecture": query head h reads kv head h // G, so
    kv head 0 serves query heads 0..G-1 (repeat, not tile).

    Construction: W_v = 0 and the v bias of kv head g is the constant c_g, and
    every cached V of head g is c_g too, so attention returns c_g for every
    query head that reads kv head g whatever the scores. W_o = I and W_d = 0
    make the block output x + a."""
    s = synth.TINY
    D, G = s.head_dim, s.group
    w = synth.model_weights(s, seed=0)
    lw = w["layers"][0]
    consts = [0.5, -1.25]
    lw["wv"] = torch.zeros_like(lw["wv"])
    lw["bv"] = _bf16(np.repeat(consts, D))
    lw["wo"] = _bf16(np.eye(s.hidden, s.q_dim))
    lw["wd"] = torch.zeros_like(lw["wd"])
    m = orc.OracleModel(s, w)
    kv = m.new_kv(1, 8)
    pos = 5
    for g, c in enumerate(consts):
        kv.v[0, 0, g, :pos] = c
    kv.k[0, 0, :, :pos] = synth.normal_bf16(0, 99, (s.n_kv_heads, pos, D), 0.5).float().numpy()
    x = np.random.default_rng(0).standard_normal(s.hidden)
    out = m.block_decode(0, kv, 0, pos, x, "f64")
    a = (out - x).reshape(s.n_q_heads, D)
    for h in range(s.n_q_heads):
        assert np.allclose(a[h], consts[h // G], rtol=1e-12), h
    # the tiled pairing (h % Hkv) would differ
    assert any(consts[h // G] != consts[h % s.n_kv_heads] for h in range(s.n_q_heads))


def test_causal_mask(tiny):
    """Row i of the uncached forward does not depend on tokens after i, and a
    token attends to itself (row 0 depends on token 0)."""
    m, _ = tiny
    toks = synth.token_ids(9, synth.TINY.vocab, stream=3)
    a = m.forward_full(toks, "f64")
    t2 = toks.clone()
    t2[6:] = (t2[6:] + 17) % synth.TINY.vocab
    b = m.forward_full(t2, "f64")
    assert np.array_equal(a[:6], b[:6])
    assert not np.allclose(a[6:], b[6:])
    t3 = toks.clone()
    t3[0] = (t3[0] + 1) % synth.TINY.vocab
    assert not np.allclose(m.forward_full(t3, "f64")[0], a[0])


@pytest.mark.parametrize("which", ["tiny", "tiny_qk"])
@pytest.mark.parametrize("prec", ["f32", "f64"])
@pytest.mark.parametrize("kv_bf16", [False, True])
def test_cache_invariant_five_chunkings(which, prec, kv_bf16, request):
    """nanoinfer "KV cache": the same 8 tokens under five chunkings (one shot,
    one at a time, prompt then decode, halves, ragged) give what one uncached
    pass gives, for a cache that stores fp32 or bf16."""
    m, _ = request.getfixturevalue(which)
    toks = synth.token_ids(8, m.shape.vocab, stream=4)
    ref = m.forward_full(toks, prec, kv_bf16=kv_bf16)
    for chunks in ([8], [1] * 8, [5, 1, 1, 1], [4, 4], [3, 2, 3]):
        kv = m.new_kv(1, 8, bf16=kv_bf16)
        rows, start = [], 0
        for n in chunks:
            rows.append(m.forward_chunk(kv, 0, toks[start:start + n], start, prec))
            start += n
        got = np.concatenate(rows)
        assert _rel_l2(got, ref) < (1e-6 if prec == "f32" else 1e-14), chunks
    # token-major decode steps (the decode path proper)
    kv = m.new_kv(1, 8, bf16=kv_bf16)
    for i in range(8):
        logits, nxt = m.decode_step(kv, toks[i:i + 1], np.array([i], np.int32), prec)
    assert _rel_l2(logits[0], ref[-1]) < (1e-6 if prec == "f32" else 1e-14)
    assert nxt[0] == int(np.argmax(ref[-1]))


def test_decode_batch_rows_are_independent(tiny):
    """Two sequences in one batch give what each gives alone."""
    m, _ = tiny
    toks = synth.token_ids(6, m.shape.vocab, stream=5).numpy()
    kv = m.new_kv(2, 8)
    kva, kvb = m.new_kv(1, 8), m.new_kv(1, 8)
    for i in range(3):
        both, _ = m.decode_step(kv, toks[[i, 3 + i]], np.array([i, i], np.int32))
        la, _ = m.decode_step(kva, toks[[i]], np.array([i], np.int32))
        lb, _ = m.decode_step(kvb, toks[[3 + i]], np.array([i], np.int32))
        assert np.array_equal(both[0], la[0]) and np.array_equal(both[1], lb[0])


def test_planted_position_bug_changes_output(tiny):
    """nanoinfer "KV cache": a decode step at position 0 instead of the cache
    length gives finite but different numbers (the bug that must be caught by
    comparison, since it raises nothing)."""
    m, _ = tiny
    toks = synth.token_ids(6, m.shape.vocab, stream=6)
    kv = m.new_kv(1, 8)
    m.forward_chunk(kv, 0, toks[:5], 0)
    kv_bug = kv.copy()
    good, _ = m.decode_step(kv, toks[5:6], np.array([5], np.int32))
    bad, _ = m.decode_step(kv_bug, toks[5:6], np.array([0], np.int32))
    assert np.all(np.isfinite(bad)) and _rel_l2(bad, good) > 1e-3


def test_invalid_position_rejected(tiny):
    m, _ = tiny
    kv = m.new_kv(1, 4)
    with pytest.raises(ValueError):
        m.decode_step(kv, np.array([1], np.int32), np.array([4], np.int32))


@pytest.mark.parametrize("which", ["tiny", "tiny_qk"])
def test_f32_oracle_close_to_f64(which, request):
    """The oracle's own rounding is far below the 5e-4 parity gate."""
    m, _ = request.getfixturevalue(which)
    toks = synth.token_ids(12, m.shape.vocab, stream=7)
    a = m.forward_full(toks, "f32")
    b = m.forward_full(toks, "f64")
    assert _rel_l2(a, b) < 1e-5


def test_hidden_states_drift_per_layer(tiny):
    """The per-layer residual stream is reported and the last entry feeds the
    head: logits equal the head applied to hidden[-1]."""
    m, w = tiny
    kv = m.new_kv(1, 4)
    logits, nxt, hid = m.decode_step(kv, np.array([3], np.int32), np.array([0], np.int32),
                                     "f64", hidden=True)
    import oracle
    n = oracle.rmsnorm(hid[0, -1], w["g_final"], m.shape.rms_eps, "f64")
    assert np.allclose(oracle.matvec_bf16(w["embed"], n, "f64"), logits[0], rtol=1e-14)
    e = oracle.bf16_to_f32(w["embed"][3].view(torch.int16).numpy())
    assert np.array_equal(hid[0, 0], e.astype(np.float64))


def test_w8a8_model_close_to_bf16(orc, tiny):
    """The W8A8 model is the bf16 model up to quantisation error."""
    _, w = tiny
    m8 = orc.OracleModel(synth.TINY, w, w8a8=True)
    m16 = orc.OracleModel(synth.TINY, w)
    toks = synth.token_ids(6, synth.TINY.vocab, stream=8)
    a = m8.forward_full(toks, "f64")
    b = m16.forward_full(toks, "f64")
    assert 0 < _rel_l2(a, b) < 0.1
    kv = m8.new_kv(1, 8)
    for i in range(6):
        lg, _ = m8.decode_step(kv, toks[i:i + 1], np.array([i], np.int32), "f64")
    assert _rel_l2(lg[0], a[-1]) < 1e-14


def _torch_forward(shape, w, tokens):
    """The whole decoder from torch's library routines in fp64, written from
    the architecture (nanoinfer, "Model architecture"): pre-norm blocks with
    residual adds, QKV bias or per-head q/k RMSNorm, half-split RoPE as a
    complex rotation of (x_i, x_{i+D/2}), causal grouped-query SDPA (query
    head h reads kv head h // G), SwiGLU, final norm, tied or untied head."""
    F = torch.nn.functional
    d = lambda t: None if t is None else t.double()
    H, D, G = shape.hidden, shape.head_dim, shape.group
    T = len(tokens)
    x = d(w["embed"])[torch.as_tensor(tokens, dtype=torch.long)]
    half = D // 2
    inv = torch.tensor([1.0 / shape.rope_theta ** (2 * i / D) for i in range(half)],
                       dtype=torch.float64)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :])

    def rope(t):  # t [heads, T, D]
        z = torch.complex(t[..., :half], t[..., half:]) * rot
        return torch.cat([z.real, z.imag], -1)

    for lw in w["layers"]:
        lw = {k: d(v) for k, v in lw.items()}
        n = F.rms_norm(x, (H,), lw["g_attn"], shape.rms_eps)
        q = F.linear(n, lw["wq"], lw["bq"]).view(T, -1, D).transpose(0, 1)
        k = F.linear(n, lw["wk"], lw["bk"]).view(T, -1, D).transpose(0, 1)
        v = F.linear(n, lw["wv"], lw["bv"]).view(T, -1, D).transpose(0, 1)
        if shape.qk_norm:
            q = F.rms_norm(q, (D,), lw["g_q"], shape.rms_eps)
            k = F.rms_norm(k, (D,), lw["g_k"], shape.rms_eps)
        q, k = rope(q), rope(k)
        k = k.repeat_interleave(G, 0)
        v = v.repeat_interleave(G, 0)
        a = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True)[0]
        x = x + F.linear(a.transpose(0, 1).reshape(T, -1), lw["wo"])
        n2 = F.rms_norm(x, (H,), lw["g_mlp"], shape.rms_eps)
        x = x + F.linear(F.silu(F.linear(n2, lw["wg"])) * F.linear(n2, lw["wu"]), lw["wd"])
    head = d(w["lm_head"]) if w.get("lm_head") is not None else d(w["embed"])
    return F.linear(F.rms_norm(x, (H,), d(w["g_final"]), shape.rms_eps), head).numpy()


@pytest.fixture(scope="module")
def qwen_dims(orc):
    """The 0.5B layer shape (14 query heads, group 7, H 896, F 4864) with two
    layers and a 1000-token vocabulary, so fp64 torch stays small."""
    import dataclasses
    s = dataclasses.replace(synth.QWEN2_0P5B, n_layers=2, vocab=1000)
    w = synth.model_weights(s, seed=0)
    return orc.OracleModel(s, w), w


@pytest.mark.parametrize("which", ["tiny", "tiny_qk", "qwen_dims"])
def test_whole_model_matches_torch_library_composition(which, request):
    """The oracle's wiring of the pieces (which gain feeds which norm, the
    residual order, bias or q/k norm before RoPE, the head) against the same
    model composed from torch's own routines: one shape carries the QKV bias
    and the tied head, the other q/k norm, no bias and an untied head."""
    m, w = request.getfixturevalue(which)
    toks = synth.token_ids(10, m.shape.vocab, stream=11)
    ref = _torch_forward(m.shape, w, toks.tolist())
    got = m.forward_full(toks, "f64")
    assert _rel_l2(got, ref) < 1e-6
    # a planted wiring mistake (the MLP norm reading the attention gain) is seen
    w2 = dict(w)
    w2["layers"] = [dict(lw, g_mlp=lw["g_attn"]) for lw in w["layers"]]
    assert _rel_l2(got, _torch_forward(m.shape, w2, toks.tolist())) > 1e-4


def _w8a8_composition(s, w, toks, block=None, int8_embed=False, wrong_row=False):
    """The architecture from torch routines in fp64 with every projection (and,
    with int8_embed, the embedding and the tied head) replaced by the numpy
    quantiser's W8A8 product: per-row int8 weights, activations per token
    (block None) or per block, int32 sums, float(acc) * (s_w * s_x) + bias."""
    from oracle import quant
    F = torch.nn.functional

    def lin8(Wf, b, X, bad=False):
        wq, sw = quant.quantize_rows_i8(Wf)
        if bad:
            sw = sw[::-1].copy()  # row j dequantised with row N-1-j's scale
        bias = None if b is None else b.float().numpy()
        out = [quant.linear_w8a8_blocked(wq, sw, bias, x, block=block or x.size)[0]
               for x in X.numpy().astype(np.float32)]
        return torch.tensor(np.stack(out), dtype=torch.float64)

    f = lambda t: t.float().numpy()
    H, D, G, T = s.hidden, s.head_dim, s.group, len(toks)
    idx = torch.as_tensor(toks.tolist(), dtype=torch.long)
    if int8_embed:
        eq, es = quant.quantize_rows_i8(f(w["embed"]))
        x = torch.tensor(np.stack([quant.embed_i8(eq, es, int(t)) for t in toks]),
                         dtype=torch.float64)
    else:
        x = w["embed"].double()[idx]
    half = D // 2
    inv = torch.tensor([1.0 / s.rope_theta ** (2 * i / D) for i in range(half)],
                       dtype=torch.float64)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :])
    rope = lambda t: torch.cat([(z := torch.complex(t[..., :half], t[..., half:]) * rot).real,
                                z.imag], -1)
    bad = wrong_row
    for lw in w["layers"]:
        n = F.rms_norm(x, (H,), lw["g_attn"].double(), s.rms_eps)
        q = lin8(f(lw["wq"]), lw["bq"], n, bad).view(T, -1, D).transpose(0, 1)
        k = lin8(f(lw["wk"]), lw["bk"], n, bad).view(T, -1, D).transpose(0, 1)
        v = lin8(f(lw["wv"]), lw["bv"], n, bad).view(T, -1, D).transpose(0, 1)
        q, k = rope(q), rope(k)
        a = F.scaled_dot_product_attention(q[None], k.repeat_interleave(G, 0)[None],
                                           v.repeat_interleave(G, 0)[None], is_causal=True)[0]
        x = x + lin8(f(lw["wo"]), None, a.transpose(0, 1).reshape(T, -1), bad)
        n2 = F.rms_norm(x, (H,), lw["g_mlp"].double(), s.rms_eps)
        x = x + lin8(f(lw["wd"]), None, F.silu(lin8(f(lw["wg"]), None, n2, bad))
                     * lin8(f(lw["wu"]), None, n2, bad), bad)
    nf = F.rms_norm(x, (H,), w["g_final"].double(), s.rms_eps)
    if int8_embed:
        return lin8(f(w["embed"]), None, nf).numpy()
    return F.linear(nf, w["embed"].double()).numpy()


@pytest.mark.parametrize("block,int8_embed", [(None, False), (32, True)])
def test_w8a8_model_matches_composition_with_the_numpy_quantiser(orc, block, int8_embed):
    """The C oracle's W8A8 models (activations per token; per 32 with the
    embedding and tied head int8 too) against the composition above. The two
    reach the quantised activations by different summation orders, so a code
    can flip at a rounding boundary: the gate is 1e-2, while a wiring mistake
    (a scale of the wrong row) moves the logits by far more."""
    s = synth.TINY
    w = synth.model_weights(s, seed=0)
    m8 = orc.OracleModel(s, w, w8a8=True, act_block=block or 0, int8_embed=int8_embed)
    toks = synth.token_ids(6, s.vocab, stream=12)
    got = m8.forward_full(toks, "f32")
    err = _rel_l2(got, _w8a8_composition(s, w, toks, block, int8_embed))
    assert err < 1e-2, err
    bad = _rel_l2(got, _w8a8_composition(s, w, toks, block, int8_embed, wrong_row=True))
    assert bad > 10 * max(err, 1e-3)


def test_oracle_bits_do_not_depend_on_the_thread_count(orc, tiny, tiny_qk):
    """The oracle parallelises only over independent output rows, each sum in
    index order, so its output is bit-identical for 1, 2, 3 and 8 threads
    (nanocompile's thread-count sweep)."""
    before = orc.get_threads()
    try:
        for m, _ in (tiny, tiny_qk):
            toks = synth.token_ids(7, m.shape.vocab, stream=13)
            outs = []
            for n in (1, 2, 3, 8):
                orc.set_threads(n)
                outs.append(m.forward_full(toks, "f32"))
            for o in outs[1:]:
                assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    finally:
        orc.set_threads(before)


def test_blocked_w8a8_int8_embedding_model(orc):
    """The oracle's int8 embedding / head with activations in blocks of 32:
    the residual row is q * s exactly, the cached decode equals the uncached
    forward, the head is the blocked W8A8 product of the final norm, and the
    model stays near the bf16 one."""
    from oracle import quant
    s = synth.TINY
    w = synth.model_weights(s, seed=0)
    m = orc.OracleModel(s, w, w8a8=True, act_block=32, int8_embed=True)
    eq, es = m.q8_embed
    toks = synth.token_ids(6, s.vocab, stream=14)
    kv = m.new_kv(1, 8)
    for i in range(6):
        lg, _, hid = m.decode_step(kv, toks[i:i + 1], np.array([i], np.int32), "f64",
                                   hidden=True)
    assert np.array_equal(hid[0, 0], quant.embed_i8(eq, es, int(toks[5])).astype(np.float64))
    full = m.forward_full(toks, "f64")
    assert _rel_l2(lg[0], full[-1]) < 1e-14
    n = orc.rmsnorm(hid[0, -1], w["g_final"], s.rms_eps, "f64")
    assert np.allclose(orc.linear_w8a8_blocked(eq, es, None, n, 32, "f64"), lg[0], rtol=1e-14,
                       atol=1e-14)
    bf = orc.OracleModel(s, w).forward_full(toks, "f64")
    assert 0 < _rel_l2(full, bf) < 0.1
    # per-32 blocks sit closer to the bf16 model than one scale per token
    per_tok = orc.OracleModel(s, w, w8a8=True, int8_embed=True).forward_full(toks, "f64")
    assert _rel_l2(full, bf) < _rel_l2(per_tok, bf)


def _int4_composition(s, w, toks, group, shift_scales=False):
    """The architecture from torch routines in fp64 with every projection
    replaced by the numpy INT4 product of the same weights (oracle/quant.py,
    its fp64 form): W_deq x with W_deq = q * s rounded to fp32."""
    from oracle import quant
    F = torch.nn.functional
    f = lambda t: t.float().numpy()

    def lin4(Wt, b, X):
        q, sc = quant.quantize_int4(f(Wt), group)
        if shift_scales:
            sc = np.roll(sc, 1, axis=1)  # each group dequantised with its neighbour's scale
        wd = torch.tensor(quant.dequant_int4(q, sc, group), dtype=torch.float64)
        return F.linear(X, wd, None if b is None else b.double())

    H, D, G, T = s.hidden, s.head_dim, s.group, len(toks)
    x = w["embed"].double()[torch.as_tensor(toks.tolist(), dtype=torch.long)]
    half = D // 2
    inv = torch.tensor([1.0 / s.rope_theta ** (2 * i / D) for i in range(half)],
                       dtype=torch.float64)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * inv[None, :])
    rope = lambda t: torch.cat([(z := torch.complex(t[..., :half], t[..., half:]) * rot).real,
                                z.imag], -1)
    for lw in w["layers"]:
        n = F.rms_norm(x, (H,), lw["g_attn"].double(), s.rms_eps)
        q = lin4(lw["wq"], lw["bq"], n).view(T, -1, D).transpose(0, 1)
        k = lin4(lw["wk"], lw["bk"], n).view(T, -1, D).transpose(0, 1)
        v = lin4(lw["wv"], lw["bv"], n).view(T, -1, D).transpose(0, 1)
        q, k = rope(q), rope(k)
        a = F.scaled_dot_product_attention(q[None], k.repeat_interleave(G, 0)[None],
                                           v.repeat_interleave(G, 0)[None], is_causal=True)[0]
        x = x + lin4(lw["wo"], None, a.transpose(0, 1).reshape(T, -1))
        n2 = F.rms_norm(x, (H,), lw["g_mlp"].double(), s.rms_eps)
        x = x + lin4(lw["wd"], None, F.silu(lin4(lw["wg"], None, n2)) * lin4(lw["wu"], None, n2))
    return F.linear(F.rms_norm(x, (H,), w["g_final"].double(), s.rms_eps),
                    w["embed"].double()).numpy()


@pytest.mark.parametrize("group", [32, 128])
def test_int4_model(orc, group):
    """The oracle's INT4 model mode: no activation is quantised, so it meets
    the torch composition with the numpy product at fp64 rounding (a shifted
    group scale is caught), the cached decode equals the uncached forward,
    and it stays near the bf16 model."""
    s = synth.TINY
    w = synth.model_weights(s, seed=0)
    m = orc.OracleModel(s, w, int4_group=group)
    toks = synth.token_ids(6, s.vocab, stream=15)
    full = m.forward_full(toks, "f64")
    ref = _int4_composition(s, w, toks, group)
    assert _rel_l2(full, ref) < 1e-6
    assert _rel_l2(full, _int4_composition(s, w, toks, group, shift_scales=True)) > 1e-3
    kv = m.new_kv(1, 8)
    for i in range(6):
        lg, _ = m.decode_step(kv, toks[i:i + 1], np.array([i], np.int32), "f64")
    assert _rel_l2(lg[0], full[-1]) < 1e-14
    assert 0 < _rel_l2(full, orc.OracleModel(s, w).forward_full(toks, "f64")) < 0.5


def test_int4_group_32_is_closer_to_bf16_than_128(orc):
    """Smaller groups confine each large weight to fewer neighbours (the page:
    group 32 cuts weight error from 12.3% to 9.9%)."""
    s = synth.TINY
    w = synth.model_weights(s, seed=0)
    toks = synth.token_ids(6, s.vocab, stream=16)
    bf = orc.OracleModel(s, w).forward_full(toks, "f64")
    e32 = _rel_l2(orc.OracleModel(s, w, int4_group=32).forward_full(toks, "f64"), bf)
    e128 = _rel_l2(orc.OracleModel(s, w, int4_group=128).forward_full(toks, "f64"), bf)
    assert e32 < e128
