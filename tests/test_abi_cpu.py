"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/nc.h declares, and rejects invalid input before
any CUDA call (nothing here reaches a kernel)."""
import ctypes as C
import os
import re

import pytest

from transformer_decode_gb300 import nc, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "nc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nc_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return nc.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(nc.EXPORTS)
    assert lib.nc_abi_version() == 1


def test_status_strings(lib):
    for code, name in enumerate(nc.STATUS):
        assert lib.nc_status_string(code).decode() == name


def _cfg(**kw):
    s = synth.QWEN2_0P5B
    c = nc.Config(s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.ffn, s.n_layers, s.vocab,
                  1e-6, 1e6, 1, 0, 1, 0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value", [("head_dim", 96), ("n_kv_heads", 3), ("hidden", 900),
                                          ("rms_eps", 0.0), ("wtype", 7), ("vocab", 0)])
def test_model_create_rejects_bad_config(lib, field, value):
    cfg = _cfg(**{field: value})
    layers = (nc.LayerWeights * cfg.n_layers)()
    w = nc.Weights(16, 0, 16, layers)
    h = C.c_void_p()
    rc = lib.nc_model_create(C.byref(cfg), C.byref(w), 1, 128, None, C.byref(h))
    assert rc == nc.STATUS.index("NC_ERR_SHAPE"), lib.nc_last_error_message()
    assert h.value is None


def test_model_create_rejects_null_and_misaligned_weights(lib):
    cfg = _cfg()
    layers = (nc.LayerWeights * cfg.n_layers)()
    h = C.c_void_p()
    rc = lib.nc_model_create(C.byref(cfg), C.byref(nc.Weights(0, 0, 16, layers)), 1, 128, None,
                             C.byref(h))
    assert rc == nc.STATUS.index("NC_ERR_INVALID_ARGUMENT")
    rc = lib.nc_model_create(C.byref(cfg), C.byref(nc.Weights(24, 0, 16, layers)), 1, 128, None,
                             C.byref(h))
    assert rc == nc.STATUS.index("NC_ERR_INVALID_ARGUMENT")
    assert b"aligned" in lib.nc_last_error_message()
    # a layer pointer missing
    rc = lib.nc_model_create(C.byref(cfg), C.byref(nc.Weights(16, 0, 16, layers)), 1, 128, None,
                             C.byref(h))
    assert rc == nc.STATUS.index("NC_ERR_INVALID_ARGUMENT")
    # capacity
    rc = lib.nc_model_create(C.byref(cfg), C.byref(nc.Weights(16, 0, 16, layers)), 17, 128, None,
                             C.byref(h))
    assert rc == nc.STATUS.index("NC_ERR_CAPACITY")


def test_stage_entry_points_reject_bad_shapes(lib):
    P = C.c_void_p(4096)
    BF, I8 = nc.NC_BF16, nc.NC_INT8
    assert lib.nc_rmsnorm_gemv(None, None, 1e-6, P, BF, None, None, 1, 64, 8, P, None, None) == 1
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, BF, None, None, 1, 60, 8, P, None, None) == 2   # K % 8
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, BF, None, None, 17, 64, 8, P, None, None) == 2  # B > 16
    assert lib.nc_rmsnorm_gemv(C.c_void_p(4100), None, 1e-6, P, BF, None, None, 1, 64, 8, P, None,
                               None) == 1
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, BF, None, 0, 64, 8, P, None) == 2
    assert lib.nc_gemv_residual(P, P, BF, None, 1, 64, 0, P, None) == 2
    # the weight type: unknown -> NC_ERR_DTYPE; scales and accumulators belong to NC_INT8;
    # NC_INT8 needs its scales and K a multiple of 16
    E = {n: nc.STATUS.index(n) for n in nc.STATUS}
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, 7, None, None, 1, 64, 8, P, None, None) == E["NC_ERR_DTYPE"]
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, 7, None, 1, 64, 8, P, None) == E["NC_ERR_DTYPE"]
    assert lib.nc_gemv_residual(P, P, 7, None, 1, 64, 8, P, None) == E["NC_ERR_DTYPE"]
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, BF, P, None, 1, 64, 8, P, None, None) == 1
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, BF, None, None, 1, 64, 8, P, P, None) == 1
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, BF, P, 1, 64, 8, P, None) == 1
    assert lib.nc_gemv_residual(P, P, BF, P, 1, 64, 8, P, None) == 1
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, I8, None, None, 1, 64, 8, P, None, None) == 1
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, I8, None, 1, 64, 8, P, None) == 1
    assert lib.nc_gemv_residual(P, P, I8, None, 1, 64, 8, P, None) == 1
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, I8, P, None, 1, 40, 8, P, None, None) == 2  # K % 16
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, I8, P, 17, 64, 8, P, None) == 2
    assert lib.nc_gemv_residual(P, P, I8, P, 1, 64, 0, P, None) == 2
    assert lib.nc_w8a8_gemv(P, None, 1e-6, P, P, None, 1, 40, 8, P, None, None, None, None) == 2
    assert lib.nc_quantize_weight(P, 0, 8, P, P, None) == 2
    assert lib.nc_decode_step(None, 1, P, P, P, None, P, None, 1, None) == 1
    assert lib.nc_model_destroy(None) == 1


def test_sample_rejects_bad_arguments_before_any_launch(lib):
    P = C.c_void_p(4096)
    V = 151936
    need = lib.nc_sample_scratch_bytes(16, V)
    assert need == 16 * 5 * ((V + 63) // 64 * 64) * 4
    assert lib.nc_sample_scratch_bytes(0, V) == 0 and lib.nc_sample_scratch_bytes(1, 0) == 0
    E = {n: nc.STATUS.index(n) for n in nc.STATUS}

    def call(logits=P, B=16, V=V, T=0.7, k=20, p=0.8, u=P, tok=P, kept=None, scratch=P,
             nbytes=need):
        return lib.nc_sample(logits, B, V, T, k, p, u, tok, kept, scratch, nbytes, None)

    assert call(logits=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(tok=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(B=0) == E["NC_ERR_SHAPE"] and call(B=65536) == E["NC_ERR_SHAPE"]
    assert call(V=0) == E["NC_ERR_SHAPE"] and call(V=(1 << 24) + 1) == E["NC_ERR_SHAPE"]
    for T in (-0.5, float("nan"), float("inf")):
        assert call(T=T) == E["NC_ERR_INVALID_ARGUMENT"], T
    assert call(k=-1) == E["NC_ERR_INVALID_ARGUMENT"]
    for p in (0.0, -0.1, 1.01, float("nan")):
        assert call(p=p) == E["NC_ERR_INVALID_ARGUMENT"], p
    assert call(u=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(scratch=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(scratch=C.c_void_p(4100)) == E["NC_ERR_INVALID_ARGUMENT"]  # misaligned
    assert call(nbytes=need - 1) == E["NC_ERR_CAPACITY"]
    assert b"needed" in lib.nc_last_error_message()


def test_static_attention_validates_cache_and_positions_on_the_host(lib):
    """nc_attn_decode_static needs no model: every rejection below is decided
    from host data (sizes, positions_host, block_table_host) before anything
    touches the device. Every call here must be rejected: the pointers are
    fake and must never reach a kernel."""
    import numpy as np
    E = {n: nc.STATUS.index(n) for n in nc.STATUS}
    P = C.c_void_p(4096)

    def kv(**kw):
        d = dict(paged=0, dtype=nc.NC_KV_F32, batch_capacity=2, max_ctx=64, block_size=16,
                 num_blocks=8, max_blocks_per_seq=4, k=4096, v=8192, block_table=None,
                 block_table_host=None)
        d.update(kw)
        return nc.KVStruct(**d)

    def call(pos=(3, 5), B=2, Hq=14, Hkv=2, D=64, L=24, layer=0, cache=None, q=P, out=P):
        ph = np.ascontiguousarray(np.asarray(pos, np.int32))
        c = cache if cache is not None else kv()
        return lib.nc_attn_decode_static(Hq, Hkv, D, L, layer, B, q, P,
                                         ph.ctypes.data_as(C.c_void_p), C.byref(c), out, None)

    assert call(q=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(out=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(cache=kv(k=0)) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(D=96) == E["NC_ERR_SHAPE"]
    assert call(Hq=15) == E["NC_ERR_SHAPE"]                 # not a multiple of Hkv
    assert call(Hq=18, Hkv=2) == E["NC_ERR_SHAPE"]          # group 9 > 8
    assert call(layer=24) == E["NC_ERR_SHAPE"] and call(layer=-1) == E["NC_ERR_SHAPE"]
    assert call(B=0, pos=()) == E["NC_ERR_CAPACITY"]
    assert call(B=17, pos=[0] * 17) == E["NC_ERR_CAPACITY"]
    assert call(cache=kv(dtype=5)) == E["NC_ERR_DTYPE"]
    assert call(cache=kv(k=4100)) == E["NC_ERR_INVALID_ARGUMENT"]   # misaligned
    assert call(cache=kv(batch_capacity=1)) == E["NC_ERR_CAPACITY"]
    assert call(pos=(3, 64)) == E["NC_ERR_POSITION"]        # slot 64 of a 64-slot cache
    assert call(pos=(-1, 0)) == E["NC_ERR_POSITION"]
    # paged: tables required; every block up to the position must be in the pool
    assert call(cache=kv(paged=1)) == E["NC_ERR_INVALID_ARGUMENT"]
    table = np.array([[0, 1, 2, 3], [4, 5, -1, 7]], np.int32)
    pk = kv(paged=1, block_table=4096, block_table_host=table.ctypes.data)
    assert call(pos=(63, 32), cache=pk) == E["NC_ERR_POSITION"]       # block 2 of row 1 is a hole
    table[0, 3] = 8                                                   # outside the 8-block pool
    assert call(pos=(63, 0), cache=pk) == E["NC_ERR_POSITION"]
    assert call(pos=(64, 0), cache=pk) == E["NC_ERR_POSITION"]        # past 4 blocks x 16
    # the static merge tickets bound batch x kv heads
    assert call(B=16, pos=[0] * 16, Hq=128, Hkv=128,
                cache=kv(batch_capacity=16)) == E["NC_ERR_CAPACITY"]
    assert b"tickets" in lib.nc_last_error_message()
    # the status reader refuses a null destination before touching the device
    assert lib.nc_attn_decode_static_status(None, None) == E["NC_ERR_INVALID_ARGUMENT"]


def test_entry_points_reject_misaligned_pointers(lib):
    """Each pointer must meet the widest access its kernels make through it
    (16-byte weight and activation streams, 8-byte gain pairs, scalar fp32 /
    int32 / fp64 elements); a misaligned one is refused on the host, before
    any launch."""
    E = nc.STATUS.index("NC_ERR_INVALID_ARGUMENT")
    P, P2, P4 = C.c_void_p(4096), C.c_void_p(4098), C.c_void_p(4100)
    # gamma read 8 bytes at a time, bias per bf16, y per fp32
    BF, I8 = nc.NC_BF16, nc.NC_INT8
    assert lib.nc_rmsnorm_gemv(P, P4, 1e-6, P, BF, None, None, 1, 64, 8, P, None, None) == E
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, BF, None, C.c_void_p(4097), 1, 64, 8, P, None,
                               None) == E
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, BF, None, None, 1, 64, 8, P2, None, None) == E
    assert lib.nc_swiglu_gemv(P, P4, 1e-6, P, BF, None, 1, 64, 8, P, None) == E
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, BF, None, 1, 64, 8, P2, None) == E
    assert lib.nc_gemv_residual(P, P, BF, None, 1, 64, 8, P2, None) == E
    # NC_INT8: 16-byte int8 rows, 4-byte scales, accumulators and outputs
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P2, I8, P, None, 1, 64, 8, P, None, None) == E
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, I8, P2, None, 1, 64, 8, P, None, None) == E
    assert lib.nc_rmsnorm_gemv(P, None, 1e-6, P, I8, P, None, 1, 64, 8, P, P2, None) == E
    assert lib.nc_swiglu_gemv(P, None, 1e-6, P, I8, P2, 1, 64, 8, P, None) == E
    assert lib.nc_gemv_residual(P, P, I8, P, 1, 64, 8, P2, None) == E
    assert lib.nc_w8a8_gemv(P2, None, 1e-6, P, P, None, 1, 64, 8, P, None, None, None, None) == E
    assert lib.nc_w8a8_gemv(P, None, 1e-6, P, P2, None, 1, 64, 8, P, None, None, None, None) == E
    assert lib.nc_w8a8_gemv(P, None, 1e-6, P, P, None, 1, 64, 8, P, None, P2, None, None) == E
    # the sampler: fp32 logits, int32 tokens and counts, fp64 uniforms
    n = lib.nc_sample_scratch_bytes(1, 1000)
    assert lib.nc_sample(P2, 1, 1000, 0.7, 20, 0.8, P, P, None, P, n, None) == E
    assert lib.nc_sample(P, 1, 1000, 0.7, 20, 0.8, P4, P, None, P, n, None) == E
    assert lib.nc_sample(P, 1, 1000, 0.7, 20, 0.8, P, P2, None, P, n, None) == E
    assert lib.nc_sample(P, 1, 1000, 0.7, 20, 0.8, P, P, P2, P, n, None) == E


def test_w8a8_b32_rejects_bad_arguments(lib):
    E = {n: nc.STATUS.index(n) for n in nc.STATUS}
    P = C.c_void_p(4096)
    call = lambda x=P, W=P, B=1, K=896, N=8, y=P, sx=None: lib.nc_w8a8_gemv_b32(
        x, None, 1e-6, W, P, None, B, K, N, y, None, sx, None, None)
    assert call(x=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(W=C.c_void_p(4104)) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(sx=C.c_void_p(4098)) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(B=0) == E["NC_ERR_SHAPE"] and call(B=9) == E["NC_ERR_SHAPE"]
    assert call(K=880) == E["NC_ERR_SHAPE"] and call(K=16) == E["NC_ERR_SHAPE"]


def test_int4_gemv_rejects_bad_arguments(lib):
    E = {n: nc.STATUS.index(n) for n in nc.STATUS}
    P = C.c_void_p(4096)
    call = lambda x=P, W=P, sc=P, group=32, B=1, K=896, N=8, y=P, g=None: lib.nc_int4_gemv(
        x, g, 1e-6, W, sc, group, B, K, N, y, None)
    assert call(x=None) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(W=C.c_void_p(4104)) == E["NC_ERR_INVALID_ARGUMENT"]  # packed rows need 16 bytes
    assert call(g=C.c_void_p(4097)) == E["NC_ERR_INVALID_ARGUMENT"]
    assert call(B=0) == E["NC_ERR_SHAPE"] and call(B=9) == E["NC_ERR_SHAPE"]
    assert call(group=48) == E["NC_ERR_SHAPE"]
    assert call(K=880, group=32) == E["NC_ERR_SHAPE"]             # not a multiple of the group
    assert call(K=960, group=128) == E["NC_ERR_SHAPE"]            # 960 is not a multiple of 128
    assert call(N=0) == E["NC_ERR_SHAPE"]
