"""Python access to the CPU oracle (liboracle.so).

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline use this package. It builds liboracle.so from oracle.c with gcc (no
CUDA, no shared code with the CUDA library) and exposes thin ctypes wrappers
that take numpy arrays or CPU torch tensors.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = [os.path.join(_HERE, f) for f in ("oracle.c", "oracle_impl.h", "oracle.h")]
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
          "-std=c11", "-Wall"]


def build(force: bool = False) -> str:
    """Compile liboracle.so if it is missing or older than its sources."""
    stale = force or not os.path.exists(_SO) or any(
        os.path.getmtime(s) > os.path.getmtime(_SO) for s in _SRC)
    if stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC[0], "-lm"])
        os.replace(tmp, _SO)
    return _SO


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("n_layers", C.c_int),
                ("vocab", C.c_int), ("rms_eps", C.c_double), ("rope_theta", C.c_double),
                ("qkv_bias", C.c_int), ("qk_norm", C.c_int), ("tie_embeddings", C.c_int)]


_LAYER_U16 = ["wq", "wk", "wv", "bq", "bk", "bv", "wo", "wg", "wu", "wd",
              "g_attn", "g_mlp", "g_q", "g_k"]
_LAYER_I8 = ["q8_wq", "q8_wk", "q8_wv", "q8_wo", "q8_wg", "q8_wu", "q8_wd"]
_LAYER_F32 = ["s_wq", "s_wk", "s_wv", "s_wo", "s_wg", "s_wu", "s_wd"]
_LAYER_U8_4 = ["q4_wq", "q4_wk", "q4_wv", "q4_wo", "q4_wg", "q4_wu", "q4_wd"]
_LAYER_F32_4 = ["s4_wq", "s4_wk", "s4_wv", "s4_wo", "s4_wg", "s4_wu", "s4_wd"]
PROJ = ["wq", "wk", "wv", "wo", "wg", "wu", "wd"]


class Layer(C.Structure):
    _fields_ = ([(n, C.POINTER(C.c_uint16)) for n in _LAYER_U16]
                + [(n, C.POINTER(C.c_int8)) for n in _LAYER_I8]
                + [(n, C.POINTER(C.c_float)) for n in _LAYER_F32]
                + [(n, C.POINTER(C.c_uint8)) for n in _LAYER_U8_4]
                + [(n, C.POINTER(C.c_float)) for n in _LAYER_F32_4])


class Model(C.Structure):
    _fields_ = [("cfg", Config), ("embed", C.POINTER(C.c_uint16)),
                ("lm_head", C.POINTER(C.c_uint16)), ("g_final", C.POINTER(C.c_uint16)),
                ("layers", C.POINTER(Layer)), ("w8a8", C.c_int), ("act_block", C.c_int),
                ("q8_embed", C.POINTER(C.c_int8)), ("s_embed", C.POINTER(C.c_float)),
                ("int4_group", C.c_int)]


class KV(C.Structure):
    _fields_ = [("batch", C.c_int), ("max_ctx", C.c_int), ("bf16", C.c_int),
                ("k", C.c_void_p), ("v", C.c_void_p)]


def _p(a, ct):
    return None if a is None else a.ctypes.data_as(C.POINTER(ct))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


def _declare(L):
    u16p, i8p, f32p, f64p = (C.POINTER(C.c_uint16), C.POINTER(C.c_int8),
                             C.POINTER(C.c_float), C.POINTER(C.c_double))
    i32p = C.POINTER(C.c_int32)
    L.orc_bf16_to_f32_n.argtypes = [u16p, f32p, C.c_long]
    L.orc_f32_to_bf16_n.argtypes = [f32p, u16p, C.c_long]
    L.orc_quantize_row_f32.argtypes = [f32p, C.c_int, i8p]
    L.orc_quantize_row_f32.restype = C.c_float
    L.orc_quantize_weight_f32.argtypes = [u16p, C.c_int, C.c_int, i8p, f32p]
    L.orc_matvec_i8.argtypes = [i8p, C.c_int, C.c_int, i8p, i32p]
    L.orc_argmax_f32.argtypes = [f32p, C.c_int]
    L.orc_argmax_f64.argtypes = [f64p, C.c_int]
    L.orc_rope_inv_freq.argtypes = [C.c_double, C.c_int, f32p]
    L.orc_set_threads.argtypes = [C.c_int]
    L.orc_get_threads.restype = C.c_int
    for sfx, rp, rt in (("f32", f32p, C.c_float), ("f64", f64p, C.c_double)):
        g = lambda n: getattr(L, f"orc_{n}_{sfx}")
        g("rmsnorm").argtypes = [rp, C.c_int, u16p, C.c_double, rp]
        g("matvec_bf16").argtypes = [u16p, C.c_int, C.c_int, rp, rp]
        g("rope").argtypes = [rp, C.c_int, C.c_int, C.c_double]
        g("rope_interleaved").argtypes = [rp, C.c_int, C.c_int, C.c_double]
        g("silu").argtypes = [rt]
        g("silu").restype = rt
        g("softmax").argtypes = [rp, C.c_int, rp]
        g("attention_head").argtypes = [rp, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, rp]
        g("linear_w8a8").argtypes = [i8p, f32p, u16p, C.c_int, C.c_int, rp, rp]
        g("linear_w8a8_blocked").argtypes = [i8p, f32p, u16p, C.c_int, C.c_int, C.c_int, rp, rp]
        g("linear_int4").argtypes = [C.POINTER(C.c_uint8), f32p, C.c_int, u16p, C.c_int,
                                     C.c_int, rp, rp]
        g("block_decode").argtypes = [C.POINTER(Model), C.c_int, C.POINTER(KV), C.c_int,
                                      C.c_int, rp]
        g("decode_step").argtypes = [C.POINTER(Model), C.POINTER(KV), C.c_int, i32p, i32p,
                                     rp, i32p, rp]
        g("decode_step").restype = C.c_int
        g("forward_chunk").argtypes = [C.POINTER(Model), C.POINTER(KV), C.c_int, C.c_int,
                                       i32p, C.c_int, rp]
        g("forward_chunk").restype = C.c_int
        g("forward_full").argtypes = [C.POINTER(Model), C.c_int, i32p, C.c_int, rp]
        g("forward_full").restype = C.c_int


# --------------------------------------------------------------------------
# numpy helpers
# --------------------------------------------------------------------------
def _np(t, dtype):
    """A C-contiguous numpy array of dtype from a numpy array or CPU tensor
    (bf16 tensors are reinterpreted as their uint16 bit patterns)."""
    if t is None:
        return None
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" \
                and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _real(prec):
    return (np.float32, C.c_float) if prec == "f32" else (np.float64, C.c_double)


def bf16_to_f32(bits) -> np.ndarray:
    b = _np(bits, np.uint16)
    out = np.empty(b.shape, np.float32)
    lib().orc_bf16_to_f32_n(_p(b, C.c_uint16), _p(out, C.c_float), b.size)
    return out


def f32_to_bf16(x) -> np.ndarray:
    f = _np(x, np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().orc_f32_to_bf16_n(_p(f, C.c_float), _p(out, C.c_uint16), f.size)
    return out


def rmsnorm(x, g, eps, prec="f32"):
    dt, ct = _real(prec)
    x = _np(x, dt)
    g = _np(g, np.uint16)
    out = np.empty_like(x)
    getattr(lib(), f"orc_rmsnorm_{prec}")(_p(x, ct), x.size, _p(g, C.c_uint16), eps, _p(out, ct))
    return out


def matvec_bf16(w, x, prec="f32"):
    dt, ct = _real(prec)
    w = _np(w, np.uint16)
    x = _np(x, dt)
    n, k = w.shape
    y = np.empty(n, dt)
    getattr(lib(), f"orc_matvec_bf16_{prec}")(_p(w, C.c_uint16), n, k, _p(x, ct), _p(y, ct))
    return y


def rope(v, pos, theta, prec="f32", interleaved=False):
    dt, ct = _real(prec)
    v = _np(v, dt).copy()
    fn = "rope_interleaved" if interleaved else "rope"
    getattr(lib(), f"orc_{fn}_{prec}")(_p(v, ct), v.size, pos, theta)
    return v


def silu(x, prec="f32"):
    return getattr(lib(), f"orc_silu_{prec}")(float(x))


def softmax(s, prec="f32"):
    dt, ct = _real(prec)
    s = _np(s, dt)
    p = np.empty_like(s)
    getattr(lib(), f"orc_softmax_{prec}")(_p(s, ct), s.size, _p(p, ct))
    return p


def attention_head(q, k, v, prec="f32"):
    """q [D]; k, v [n_pos, D] as bf16 bits (uint16 arrays, bf16 tensors) or
    fp32 values (float32 arrays or tensors)."""
    dt, ct = _real(prec)
    q = _np(q, dt)
    bf16 = _is_bf16(k)
    k = _np(k, np.uint16 if bf16 else np.float32)
    v = _np(v, np.uint16 if bf16 else np.float32)
    out = np.empty(q.size, dt)
    getattr(lib(), f"orc_attention_head_{prec}")(_p(q, ct), k.ctypes.data, v.ctypes.data, int(bf16),
                                                k.shape[0], q.size, _p(out, ct))
    return out


def _is_bf16(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.dtype == torch.bfloat16
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a).dtype == np.uint16


def quantize_row(v):
    v = _np(v, np.float32)
    q = np.empty(v.size, np.int8)
    s = lib().orc_quantize_row_f32(_p(v, C.c_float), v.size, _p(q, C.c_int8))
    return q, np.float32(s)


def quantize_weight(w):
    w = _np(w, np.uint16)
    n, k = w.shape
    q = np.empty((n, k), np.int8)
    s = np.empty(n, np.float32)
    lib().orc_quantize_weight_f32(_p(w, C.c_uint16), n, k, _p(q, C.c_int8), _p(s, C.c_float))
    return q, s


def matvec_i8(w, x):
    w = _np(w, np.int8)
    x = _np(x, np.int8)
    n, k = w.shape
    acc = np.empty(n, np.int32)
    rc = lib().orc_matvec_i8(_p(w, C.c_int8), n, k, _p(x, C.c_int8), _p(acc, C.c_int32))
    if rc != 0:
        raise OverflowError("int8 dot product left the int32 range")
    return acc


def linear_w8a8(w8, sw, bias, x, prec="f32"):
    dt, ct = _real(prec)
    w8 = _np(w8, np.int8)
    sw = _np(sw, np.float32)
    bias = _np(bias, np.uint16)
    x = _np(x, dt)
    n, k = w8.shape
    y = np.empty(n, dt)
    getattr(lib(), f"orc_linear_w8a8_{prec}")(_p(w8, C.c_int8), _p(sw, C.c_float),
                                             _p(bias, C.c_uint16), n, k, _p(x, ct), _p(y, ct))
    return y


def linear_w8a8_blocked(w8, sw, bias, x, block=32, prec="f32"):
    """W8A8 with activations quantised per block of `block` values."""
    dt, ct = _real(prec)
    w8 = _np(w8, np.int8)
    sw = _np(sw, np.float32)
    bias = _np(bias, np.uint16)
    x = _np(x, dt)
    n, k = w8.shape
    y = np.empty(n, dt)
    getattr(lib(), f"orc_linear_w8a8_blocked_{prec}")(_p(w8, C.c_int8), _p(sw, C.c_float),
                                                     _p(bias, C.c_uint16), n, k, int(block),
                                                     _p(x, ct), _p(y, ct))
    return y


def linear_int4(packed, s4, group, bias, x, prec="f32"):
    """y = the INT4 group-wise rows (packed [N, K/2] uint8, scales [N, K/group])
    times x, + bias."""
    dt, ct = _real(prec)
    packed = _np(packed, np.uint8)
    s4 = _np(s4, np.float32)
    bias = _np(bias, np.uint16)
    x = _np(x, dt)
    n = packed.shape[0]
    k = 2 * packed.shape[1]
    y = np.empty(n, dt)
    getattr(lib(), f"orc_linear_int4_{prec}")(_p(packed, C.c_uint8), _p(s4, C.c_float),
                                             int(group), _p(bias, C.c_uint16), n, k,
                                             _p(x, ct), _p(y, ct))
    return y


def argmax(v):
    v = np.ascontiguousarray(v)
    if v.dtype == np.float64:
        return lib().orc_argmax_f64(_p(v, C.c_double), v.size)
    v = v.astype(np.float32, copy=False)
    return lib().orc_argmax_f32(_p(v, C.c_float), v.size)


def rope_inv_freq(theta, d):
    out = np.empty(d // 2, np.float32)
    lib().orc_rope_inv_freq(theta, d, _p(out, C.c_float))
    return out


def set_threads(n: int):
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return lib().orc_get_threads()


# --------------------------------------------------------------------------
# Whole model
# --------------------------------------------------------------------------
class OracleModel:
    """A model held as numpy arrays plus the ctypes structs that point at them.

    weights: the dict produced by the seeded generator (torch or numpy, bf16).
    w8a8: if True, each layer's seven projections are quantised per output
    row by the oracle's own weight quantiser and the int8 path is used.
    act_block: with w8a8, 0 quantises each token's activations with one
    scale; 32 uses one scale per block of 32 values.
    int8_embed: the embedding (and the tied head) is stored int8 per row too.
    int4_group: > 0 stores the seven projections as INT4 with one scale per
    group of that many weights (quantised by oracle/quant.py), fp32 activations.
    """

    def __init__(self, shape, weights, w8a8=False, act_block=0, int8_embed=False,
                 int4_group=0):
        self.shape = shape
        self._keep = []
        cfg = Config(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                     shape.ffn, shape.n_layers, shape.vocab, shape.rms_eps, shape.rope_theta,
                     int(shape.qkv_bias), int(shape.qk_norm), int(shape.tie_embeddings))
        layers = (Layer * shape.n_layers)()
        self.q8 = []
        for l, lw in enumerate(weights["layers"]):
            q8l = {}
            for n in _LAYER_U16:
                a = _np(lw.get(n), np.uint16)
                self._keep.append(a)
                setattr(layers[l], n, _p(a, C.c_uint16))
            if int4_group:
                from . import quant
                for n in PROJ:
                    wf = bf16_to_f32(_np(lw[n], np.uint16))
                    q4, s4 = quant.quantize_int4(wf, int4_group)
                    p4 = quant.pack_int4(q4)
                    q8l["int4_" + n] = (p4, s4)
                    self._keep += [p4, s4]
                    setattr(layers[l], "q4_" + n, _p(p4, C.c_uint8))
                    setattr(layers[l], "s4_" + n, _p(s4, C.c_float))
            if w8a8:
                for n in PROJ:
                    q, s = quantize_weight(lw[n])
                    q8l[n] = (q, s)
                    self._keep += [q, s]
                    setattr(layers[l], "q8_" + n, _p(q, C.c_int8))
                    setattr(layers[l], "s_" + n, _p(s, C.c_float))
            self.q8.append(q8l)
        emb = _np(weights["embed"], np.uint16)
        head = _np(weights.get("lm_head"), np.uint16)
        gf = _np(weights["g_final"], np.uint16)
        self._keep += [emb, head, gf, layers]
        self.layers = layers
        q8e = se = None
        if int8_embed:
            q8e, se = quantize_weight(emb)
            self._keep += [q8e, se]
        self.q8_embed = (q8e, se)
        self.struct = Model(cfg, _p(emb, C.c_uint16), _p(head, C.c_uint16),
                            _p(gf, C.c_uint16), layers, int(w8a8), int(act_block),
                            _p(q8e, C.c_int8), _p(se, C.c_float), int(int4_group))

    def new_kv(self, batch, max_ctx, bf16=False):
        return OracleKV(self.shape, batch, max_ctx, bf16)

    def decode_step(self, kv, tokens, positions, prec="f32", hidden=False):
        dt, ct = _real(prec)
        tokens = _np(tokens, np.int32)
        positions = _np(positions, np.int32)
        B = tokens.size
        logits = np.empty((B, self.shape.vocab), dt)
        nxt = np.empty(B, np.int32)
        hid = np.empty((B, self.shape.n_layers + 1, self.shape.hidden), dt) if hidden else None
        rc = getattr(lib(), f"orc_decode_step_{prec}")(
            C.byref(self.struct), C.byref(kv.struct), B, _p(tokens, C.c_int32),
            _p(positions, C.c_int32), _p(logits, ct), _p(nxt, C.c_int32), _p(hid, ct))
        if rc != 0:
            raise ValueError("oracle decode step rejected its input (position or NaN)")
        return (logits, nxt, hid) if hidden else (logits, nxt)

    def block_decode(self, layer, kv, b, pos, x, prec="f32"):
        dt, ct = _real(prec)
        x = _np(x, dt).copy()
        getattr(lib(), f"orc_block_decode_{prec}")(C.byref(self.struct), layer,
                                                  C.byref(kv.struct), b, pos, _p(x, ct))
        return x

    def forward_chunk(self, kv, b, tokens, start_pos, prec="f32"):
        dt, ct = _real(prec)
        tokens = _np(tokens, np.int32)
        logits = np.empty((tokens.size, self.shape.vocab), dt)
        rc = getattr(lib(), f"orc_forward_chunk_{prec}")(
            C.byref(self.struct), C.byref(kv.struct), b, tokens.size, _p(tokens, C.c_int32),
            start_pos, _p(logits, ct))
        if rc != 0:
            raise ValueError("chunk does not fit the cache")
        return logits

    def forward_full(self, tokens, prec="f32", kv_bf16=False):
        dt, ct = _real(prec)
        tokens = _np(tokens, np.int32)
        logits = np.empty((tokens.size, self.shape.vocab), dt)
        getattr(lib(), f"orc_forward_full_{prec}")(C.byref(self.struct), tokens.size,
                                                  _p(tokens, C.c_int32), int(kv_bf16),
                                                  _p(logits, ct))
        return logits


class OracleKV:
    """Logical KV cache [L][B][Hkv][max_ctx][D]: fp32 values, or bf16 bits
    (uint16) when bf16=True."""

    def __init__(self, shape, batch, max_ctx, bf16=False):
        dims = (shape.n_layers, batch, shape.n_kv_heads, max_ctx, shape.head_dim)
        dt = np.uint16 if bf16 else np.float32
        self.bf16 = bool(bf16)
        self.k = np.zeros(dims, dt)
        self.v = np.zeros(dims, dt)
        self.struct = KV(batch, max_ctx, int(bf16), self.k.ctypes.data, self.v.ctypes.data)

    def copy(self):
        o = OracleKV.__new__(OracleKV)
        o.bf16 = self.bf16
        o.k = self.k.copy()
        o.v = self.v.copy()
        o.struct = KV(self.struct.batch, self.struct.max_ctx, int(o.bf16), o.k.ctypes.data,
                      o.v.ctypes.data)
        return o
