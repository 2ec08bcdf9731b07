"""Python binding of libnc (include/nc.h): argument marshalling only.

Every function here checks tensor devices, dtypes and shapes, then calls the
C entry point of the same name; all arithmetic runs in libnc's CUDA kernels.
There is no fallback: if libnc.so cannot be loaded the import of this module
still succeeds but the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

NC_OK = 0
STATUS = ["NC_OK", "NC_ERR_INVALID_ARGUMENT", "NC_ERR_SHAPE", "NC_ERR_DTYPE", "NC_ERR_CAPACITY",
          "NC_ERR_POSITION", "NC_ERR_CUDA", "NC_ERR_TIMEOUT", "NC_ERR_UNHEALTHY",
          "NC_ERR_UNSUPPORTED"]
NC_BF16, NC_INT8, NC_INT8_B32, NC_INT4_G32, NC_INT4_G128 = 0, 1, 2, 3, 4
NC_STEP_GRAPH, NC_STEP_ADVANCE, NC_STEP_STAGED = 1, 2, 4
NC_KV_F32, NC_KV_BF16 = 0, 1

EXPORTS = [
    "nc_status_string", "nc_last_error_message", "nc_abi_version", "nc_model_create",
    "nc_model_destroy", "nc_model_memory", "nc_decode_step", "nc_block_forward",
    "nc_get_device_status", "nc_rmsnorm_gemv", "nc_gemv_residual", "nc_swiglu_gemv",
    "nc_rope_qkv", "nc_attn_decode", "nc_lm_head_argmax", "nc_quantize_weight", "nc_w8a8_gemv",
    "nc_attn_decode_static", "nc_profile_phases", "nc_read_phase_profile", "nc_decode_path",
    "nc_sample", "nc_sample_scratch_bytes", "nc_attn_decode_static_status",
    "nc_debug_w8a8_codes", "nc_w8a8_gemv_b32",
    "nc_int4_gemv", "nc_prefill", "nc_prefill_scratch_bytes",
]


class NCError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS[code] if 0 <= code < len(STATUS) else code}: {msg}")
        self.code = code


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("n_layers", C.c_int),
                ("vocab", C.c_int), ("rms_eps", C.c_float), ("rope_theta", C.c_float),
                ("qkv_bias", C.c_int), ("qk_norm", C.c_int), ("tie_embeddings", C.c_int),
                ("wtype", C.c_int)]


_LW = ["wq", "wk", "wv", "bq", "bk", "bv", "wo", "wg", "wu", "wd", "g_attn", "g_mlp", "g_q", "g_k"]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _LW]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("g_final", C.c_void_p),
                ("layers", C.POINTER(LayerWeights))]


class KVStruct(C.Structure):
    _fields_ = [("paged", C.c_int), ("dtype", C.c_int), ("batch_capacity", C.c_int),
                ("max_ctx", C.c_int),
                ("block_size", C.c_int), ("num_blocks", C.c_int),
                ("max_blocks_per_seq", C.c_int), ("k", C.c_void_p), ("v", C.c_void_p),
                ("block_table", C.c_void_p), ("block_table_host", C.c_void_p)]


def lib_path() -> str:
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libnc.so (building it first when sources are newer and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_stale:
                try:
                    _build.build()
                except RuntimeError:
                    if not os.path.exists(_build.LIB):
                        raise
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libnc.so not found at {_build.LIB}; run "
                                   "transformer_decode_gb300.build.build()")
            L = C.CDLL(_build.LIB)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    vp, i, f = C.c_void_p, C.c_int, C.c_float
    L.nc_status_string.restype = C.c_char_p
    L.nc_status_string.argtypes = [i]
    L.nc_last_error_message.restype = C.c_char_p
    L.nc_abi_version.restype = i
    L.nc_model_create.argtypes = [C.POINTER(Config), C.POINTER(Weights), i, i, vp, C.POINTER(vp)]
    L.nc_model_destroy.argtypes = [vp]
    L.nc_model_memory.argtypes = [vp, C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)]
    L.nc_decode_step.argtypes = [vp, i, vp, vp, vp, C.POINTER(KVStruct), vp, vp, i, vp]
    L.nc_block_forward.argtypes = [vp, i, i, vp, vp, vp, C.POINTER(KVStruct), vp]
    L.nc_get_device_status.argtypes = [vp, vp, C.POINTER(C.c_int)]
    L.nc_rmsnorm_gemv.argtypes = [vp, vp, f, vp, i, vp, vp, i, i, i, vp, vp, vp]
    L.nc_gemv_residual.argtypes = [vp, vp, i, vp, i, i, i, vp, vp]
    L.nc_swiglu_gemv.argtypes = [vp, vp, f, vp, i, vp, i, i, i, vp, vp]
    L.nc_rope_qkv.argtypes = [vp, i, i, vp, vp, vp, vp, C.POINTER(KVStruct), vp]
    L.nc_attn_decode.argtypes = [vp, i, i, vp, vp, vp, C.POINTER(KVStruct), vp, vp]
    L.nc_lm_head_argmax.argtypes = [vp, vp, vp, f, vp, i, i, i, vp, vp, vp]
    L.nc_quantize_weight.argtypes = [vp, i, i, vp, vp, vp]
    L.nc_w8a8_gemv.argtypes = [vp, vp, f, vp, vp, vp, i, i, i, vp, vp, vp, vp, vp]
    L.nc_attn_decode_static.argtypes = [i, i, i, i, i, i, vp, vp, vp, C.POINTER(KVStruct), vp, vp]
    L.nc_attn_decode_static_status.argtypes = [vp, C.POINTER(i)]
    L.nc_prefill.argtypes = [vp, i, i, vp, i, C.POINTER(KVStruct), vp, vp, vp, C.c_size_t, vp]
    L.nc_prefill_scratch_bytes.argtypes = [vp, i]
    L.nc_debug_w8a8_codes.argtypes = [vp, vp, C.c_size_t, vp, C.c_size_t]
    L.nc_profile_phases.argtypes = [vp, i]
    L.nc_decode_path.argtypes = [vp, i, vp, i, C.POINTER(i)]
    L.nc_read_phase_profile.argtypes = [vp, vp, C.POINTER(C.c_ulonglong), i, C.POINTER(i)]
    L.nc_sample.argtypes = [vp, i, i, f, i, f, vp, vp, vp, vp, C.c_size_t, vp]
    L.nc_sample_scratch_bytes.argtypes = [i, i]
    L.nc_w8a8_gemv_b32.argtypes = [vp, vp, f, vp, vp, vp, i, i, i, vp, vp, vp, vp, vp]
    L.nc_int4_gemv.argtypes = [vp, vp, f, vp, vp, i, i, i, i, vp, vp]
    for n in EXPORTS:
        if n not in ("nc_status_string", "nc_last_error_message", "nc_sample_scratch_bytes",
                     "nc_prefill_scratch_bytes"):
            getattr(L, n).restype = C.c_int
    L.nc_sample_scratch_bytes.restype = C.c_size_t
    L.nc_prefill_scratch_bytes.restype = C.c_size_t


def _check(rc):
    if rc != NC_OK:
        raise NCError(rc, load().nc_last_error_message().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _ptr(t, dtype=None, name="tensor", numel=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return C.c_void_p(t.data_ptr())


def _host_i32(a):
    import numpy as np
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ------------------------------------------------------------------ stage entry points
def _weights(W, w_scale, rows, K, name):
    """(pointer, weight type, scale pointer) of a stage GEMV's weights: bf16
    rows, or int8 rows with their fp32 per-row scales."""
    if W.dtype == torch.int8:
        if w_scale is None:
            raise TypeError(f"int8 {name} needs its per-row scales")
        return (_ptr(W, torch.int8, name, rows * K), NC_INT8,
                _ptr(w_scale, torch.float32, "w_scale", rows))
    if w_scale is not None:
        raise TypeError(f"scales apply to int8 {name} only")
    return _ptr(W, torch.bfloat16, name, rows * K), NC_BF16, None


def rmsnorm_gemv(x, gamma, eps, W, bias, y, w_scale=None, acc=None, stream=None):
    """nc_rmsnorm_gemv. W bf16, or int8 with w_scale (W8A8); acc [B, N] int32
    (int8 only) receives the accumulators."""
    B, K = x.shape
    N = W.shape[0]
    wp, wt, sp = _weights(W, w_scale, N, K, "W")
    _check(load().nc_rmsnorm_gemv(_ptr(x, torch.float32, "x"), _ptr(gamma, torch.bfloat16, "gamma"),
                                  float(eps), wp, wt, sp, _ptr(bias, torch.bfloat16, "bias"), B, K,
                                  N, _ptr(y, torch.float32, "y", B * N),
                                  _ptr(acc, torch.int32, "acc", B * N), _stream(stream)))


def gemv_residual(a, W, x, w_scale=None, stream=None):
    B, K = a.shape
    N = W.shape[0]
    wp, wt, sp = _weights(W, w_scale, N, K, "W")
    _check(load().nc_gemv_residual(_ptr(a, torch.float32, "a"), wp, wt, sp, B, K, N,
                                   _ptr(x, torch.float32, "x", B * N), _stream(stream)))


def swiglu_gemv(x, gamma, eps, W_gu, h, s_gu=None, stream=None):
    B, K = x.shape
    F = W_gu.shape[0] // 2
    wp, wt, sp = _weights(W_gu, s_gu, 2 * F, K, "W_gu")
    _check(load().nc_swiglu_gemv(_ptr(x, torch.float32, "x"), _ptr(gamma, torch.bfloat16, "gamma"),
                                 float(eps), wp, wt, sp, B, K, F,
                                 _ptr(h, torch.float32, "h", B * F), _stream(stream)))


def quantize_weight(W, q, scale, stream=None):
    N, K = W.shape
    _check(load().nc_quantize_weight(_ptr(W, torch.bfloat16, "W"), N, K,
                                     _ptr(q, torch.int8, "q", N * K),
                                     _ptr(scale, torch.float32, "scale", N), _stream(stream)))


def w8a8_gemv(x, gamma, eps, Wq, w_scale, bias, y, xq_out=None, sx_out=None, acc_out=None,
              stream=None):
    B, K = x.shape
    N = Wq.shape[0]
    _check(load().nc_w8a8_gemv(_ptr(x, torch.float32, "x"), _ptr(gamma, torch.bfloat16, "gamma"),
                               float(eps), _ptr(Wq, torch.int8, "Wq", N * K),
                               _ptr(w_scale, torch.float32, "w_scale", N),
                               _ptr(bias, torch.bfloat16, "bias"), B, K, N,
                               _ptr(y, torch.float32, "y", B * N),
                               _ptr(xq_out, torch.int8, "xq_out"), _ptr(sx_out, torch.float32, "sx_out"),
                               _ptr(acc_out, torch.int32, "acc_out"), _stream(stream)))


def w8a8_gemv_b32(x, gamma, eps, Wq, w_scale, bias, y, xq_out=None, sx_out=None, acc_out=None,
                  stream=None):
    """nc_w8a8_gemv_b32: the W8A8 product with activations in blocks of 32."""
    B, K = x.shape
    N = Wq.shape[0]
    _check(load().nc_w8a8_gemv_b32(
        _ptr(x, torch.float32, "x"), _ptr(gamma, torch.bfloat16, "gamma"), float(eps),
        _ptr(Wq, torch.int8, "Wq", N * K), _ptr(w_scale, torch.float32, "w_scale", N),
        _ptr(bias, torch.bfloat16, "bias"), B, K, N, _ptr(y, torch.float32, "y", B * N),
        _ptr(xq_out, torch.int8, "xq_out"), _ptr(sx_out, torch.float32, "sx_out"),
        _ptr(acc_out, torch.int32, "acc_out"), _stream(stream)))


def attn_decode_static(shape, layer, q, positions, positions_host, kv, out, stream=None):
    """nc_attn_decode_static: split-K decode attention that allocates nothing
    (its scratch is a static device array). For callers that cannot allocate
    device memory; see include/nc.h for the size limit and the set-up rule."""
    B = q.shape[0]
    ph = _host_i32(positions_host)
    s = kv.struct()
    _check(load().nc_attn_decode_static(
        shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.n_layers, layer, B,
        _ptr(q, torch.float32, "q", B * shape.q_dim), _ptr(positions, torch.int32, "positions", B),
        ph.ctypes.data_as(C.c_void_p), C.byref(s),
        _ptr(out, torch.float32, "out", B * shape.q_dim), _stream(stream)))


def attn_decode_static_status(stream=None):
    """nc_attn_decode_static_status: synchronise the stream, read and clear
    the device-side error word of attn_decode_static (0 = none)."""
    code = C.c_int(0)
    _check(load().nc_attn_decode_static_status(_stream(stream), C.byref(code)))
    return code.value


def int4_gemv(x, gamma, eps, Wq, scales, group, y, stream=None):
    """nc_int4_gemv: y = dequantised INT4 weights (packed [N, K/2] uint8, fp32
    scales [N, K/group]) times the (normed) activations x [B, K]."""
    B, K = x.shape
    N = Wq.shape[0]
    _check(load().nc_int4_gemv(_ptr(x, torch.float32, "x"), _ptr(gamma, torch.bfloat16, "gamma"),
                               float(eps), _ptr(Wq, torch.uint8, "Wq", N * K // 2),
                               _ptr(scales, torch.float32, "scales", N * (K // group)),
                               int(group), B, K, N, _ptr(y, torch.float32, "y", B * N),
                               _stream(stream)))


# ------------------------------------------------------------------ sampling
def sample_scratch_bytes(B, V):
    return int(load().nc_sample_scratch_bytes(int(B), int(V)))


def sample(logits, temperature, top_k, top_p, u, tokens, kept=None, scratch=None, stream=None):
    """nc_sample: one token per row of logits [B, V] (temperature -> top-k ->
    top-p -> inverse-CDF draw with the uniforms u [B] fp64). kept [B, 2] int32
    receives the kept counts; scratch is a caller-owned device buffer of
    sample_scratch_bytes(B, V) bytes (any dtype), needed when temperature > 0."""
    B, V = logits.shape
    sp = None
    nbytes = 0
    if scratch is not None:
        sp = _ptr(scratch, None, "scratch")
        nbytes = scratch.numel() * scratch.element_size()
    _check(load().nc_sample(_ptr(logits, torch.float32, "logits"), B, V, float(temperature),
                            int(top_k), float(top_p), _ptr(u, torch.float64, "u", B),
                            _ptr(tokens, torch.int32, "tokens", B),
                            _ptr(kept, torch.int32, "kept", 2 * B), sp, nbytes, _stream(stream)))


class Sampler:
    """A scratch buffer sized for up to max_batch rows of V logits, and the
    nc_sample call that uses it."""

    def __init__(self, max_batch, vocab, device="cuda"):
        self.max_batch, self.vocab = int(max_batch), int(vocab)
        n = sample_scratch_bytes(self.max_batch, self.vocab)
        self.scratch = torch.empty(n, dtype=torch.uint8, device=device)

    def __call__(self, logits, temperature, top_k, top_p, u, tokens, kept=None, stream=None):
        if logits.shape[0] > self.max_batch or logits.shape[1] != self.vocab:
            raise ValueError("logits larger than this sampler's scratch")
        sample(logits, temperature, top_k, top_p, u, tokens, kept, self.scratch, stream)


# ------------------------------------------------------------------ KV cache
class KVCache:
    """Caller-owned KV storage in the layouts nc.h describes, fp32 (default)
    or bf16 elements.

    contiguous: k, v [L, batch, Hkv, max_ctx, D];
    paged:      k, v [L, num_blocks, Hkv, block_size, D] with an int32
                block table [batch, max_blocks_per_seq] (device + host copy).
    """

    def __init__(self, shape, batch, max_ctx=None, paged=False, block_table=None,
                 num_blocks=None, block_size=16, dtype=torch.float32, device="cuda"):
        if dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("KV cache dtype must be torch.float32 or torch.bfloat16")
        self.shape = shape
        self.batch = batch
        self.paged = bool(paged)
        self.dtype = dtype
        L, Hkv, D = shape.n_layers, shape.n_kv_heads, shape.head_dim
        if not paged:
            self.max_ctx = int(max_ctx)
            dims = (L, batch, Hkv, self.max_ctx, D)
            self.block_size = self.num_blocks = self.max_blocks = 0
            self.table = self.table_host = None
        else:
            bt = block_table.to(torch.int32).cpu().contiguous()
            self.table_host = bt.numpy().copy()
            self.table = bt.to(device)
            self.block_size = int(block_size)
            self.num_blocks = int(num_blocks)
            self.max_blocks = bt.shape[1]
            self.max_ctx = self.max_blocks * self.block_size
            dims = (L, self.num_blocks, Hkv, self.block_size, D)
        self.k = torch.zeros(dims, dtype=dtype, device=device)
        self.v = torch.zeros(dims, dtype=dtype, device=device)

    def struct(self):
        s = KVStruct(int(self.paged), NC_KV_BF16 if self.dtype == torch.bfloat16 else NC_KV_F32,
                     self.batch, self.max_ctx, self.block_size, self.num_blocks,
                     self.max_blocks, self.k.data_ptr(), self.v.data_ptr(),
                     self.table.data_ptr() if self.paged else None,
                     self.table_host.ctypes.data if self.paged else None)
        return s

    def slot_view(self, layer, b, kv_head, pos):
        """(k, v) views of one cached position: [D] each, in the cache dtype."""
        if not self.paged:
            return self.k[layer, b, kv_head, pos], self.v[layer, b, kv_head, pos]
        blk = int(self.table_host[b, pos // self.block_size])
        o = pos % self.block_size
        return self.k[layer, blk, kv_head, o], self.v[layer, blk, kv_head, o]

    def write_sequence(self, layer, b, kv_head, k_rows, v_rows):
        """Store positions 0..n-1 of one (layer, sequence, kv head) from [n, D] rows (converted to the cache dtype)."""
        n = k_rows.shape[0]
        if not self.paged:
            self.k[layer, b, kv_head, :n] = k_rows
            self.v[layer, b, kv_head, :n] = v_rows
            return
        bs = self.block_size
        for j in range(0, n, bs):
            blk = int(self.table_host[b, j // bs])
            m = min(bs, n - j)
            self.k[layer, blk, kv_head, :m] = k_rows[j:j + m]
            self.v[layer, blk, kv_head, :m] = v_rows[j:j + m]

    def read_sequence(self, layer, b, kv_head, n):
        """Positions 0..n-1 of one (layer, sequence, kv head) as [n, D] rows."""
        if not self.paged:
            return self.k[layer, b, kv_head, :n], self.v[layer, b, kv_head, :n]
        bs = self.block_size
        ks, vs = [], []
        for j in range(0, n, bs):
            blk = int(self.table_host[b, j // bs])
            m = min(bs, n - j)
            ks.append(self.k[layer, blk, kv_head, :m])
            vs.append(self.v[layer, blk, kv_head, :m])
        return torch.cat(ks), torch.cat(vs)


# ------------------------------------------------------------------ model
class Model:
    """A libnc model built from checkpoint-layout weights on the GPU.

    weights: dict as produced by the seeded generator (bf16 CUDA tensors).
    The model keeps its own packed copy; the caller may free the originals.
    """

    def __init__(self, shape, weights, max_batch=1, max_ctx=4096, w8a8=False, int4_group=0,
                 stream=None):
        L = load()
        self.shape = shape
        self.max_batch = max_batch
        self.max_ctx = max_ctx
        cfg = Config(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                     shape.n_layers, shape.vocab, shape.rms_eps, shape.rope_theta,
                     int(shape.qkv_bias), int(shape.qk_norm), int(shape.tie_embeddings),
                     {False: NC_BF16, True: NC_INT8, "b32": NC_INT8_B32}[w8a8] if w8a8 else
                     {0: NC_BF16, 32: NC_INT4_G32, 128: NC_INT4_G128}[int4_group])
        layers = (LayerWeights * shape.n_layers)()
        for l, lw in enumerate(weights["layers"]):
            for n in _LW:
                t = lw.get(n)
                setattr(layers[l], n, None if t is None else _ptr(t, torch.bfloat16, n).value)
        w = Weights(_ptr(weights["embed"], torch.bfloat16, "embed").value,
                    None if weights.get("lm_head") is None else
                    _ptr(weights["lm_head"], torch.bfloat16, "lm_head").value,
                    _ptr(weights["g_final"], torch.bfloat16, "g_final").value, layers)
        h = C.c_void_p()
        _check(L.nc_model_create(C.byref(cfg), C.byref(w), max_batch, max_ctx, _stream(stream),
                                 C.byref(h)))
        self._h = h
        self.w8a8 = w8a8

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("model is closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            load().nc_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def memory(self):
        wb, ws = C.c_size_t(), C.c_size_t()
        _check(load().nc_model_memory(self.handle, C.byref(wb), C.byref(ws)))
        return wb.value, ws.value

    def decode_step(self, tokens, positions, positions_host, kv, logits, next_tokens=None,
                    use_graph=True, advance=False, staged=False, stream=None):
        """One decode step (nc_decode_step). advance=True: the device then sets
        tokens = greedy token and positions += 1 for the next call.
        staged=True forces the per-stage kernels instead of the persistent one."""
        B = tokens.numel()
        ph = _host_i32(positions_host)
        s = kv.struct()
        flags = ((NC_STEP_GRAPH if use_graph else 0) | (NC_STEP_ADVANCE if advance else 0)
                 | (NC_STEP_STAGED if staged else 0))
        _check(load().nc_decode_step(self.handle, B, _ptr(tokens, torch.int32, "tokens"),
                                     _ptr(positions, torch.int32, "positions", B),
                                     ph.ctypes.data_as(C.c_void_p), C.byref(s),
                                     _ptr(logits, torch.float32, "logits", B * self.shape.vocab),
                                     _ptr(next_tokens, torch.int32, "next_tokens"),
                                     flags, _stream(stream)))

    def decode_path(self, batch, kv, staged=False):
        """'persistent' or 'staged': the implementation nc_decode_step runs for
        this batch and cache (nc_decode_path; nothing is launched)."""
        s = kv.struct()
        out = C.c_int()
        _check(load().nc_decode_path(self.handle, batch, C.byref(s),
                                     NC_STEP_STAGED if staged else 0, C.byref(out)))
        return "persistent" if out.value == 1 else "staged"

    def block_forward(self, layer, x, positions, positions_host, kv, stream=None):
        B = x.shape[0]
        ph = _host_i32(positions_host)
        s = kv.struct()
        _check(load().nc_block_forward(self.handle, layer, B, _ptr(x, torch.float32, "x"),
                                       _ptr(positions, torch.int32, "positions", B),
                                       ph.ctypes.data_as(C.c_void_p), C.byref(s), _stream(stream)))

    def rope_qkv(self, layer, qkv, positions, positions_host, q_out, kv, stream=None):
        B = qkv.shape[0]
        ph = _host_i32(positions_host)
        s = kv.struct()
        _check(load().nc_rope_qkv(self.handle, layer, B, _ptr(qkv, torch.float32, "qkv"),
                                  _ptr(positions, torch.int32, "positions", B),
                                  ph.ctypes.data_as(C.c_void_p), _ptr(q_out, torch.float32, "q_out"),
                                  C.byref(s), _stream(stream)))

    def attn_decode(self, layer, q, positions, positions_host, kv, out, stream=None):
        B = q.shape[0]
        ph = _host_i32(positions_host)
        s = kv.struct()
        _check(load().nc_attn_decode(self.handle, layer, B, _ptr(q, torch.float32, "q"),
                                     _ptr(positions, torch.int32, "positions", B),
                                     ph.ctypes.data_as(C.c_void_p), C.byref(s),
                                     _ptr(out, torch.float32, "out"), _stream(stream)))

    def lm_head_argmax(self, x, gamma, eps, W, logits, next_tokens=None, stream=None):
        B, K = x.shape
        V = W.shape[0]
        _check(load().nc_lm_head_argmax(self.handle, _ptr(x, torch.float32, "x"),
                                        _ptr(gamma, torch.bfloat16, "gamma"), float(eps),
                                        _ptr(W, torch.bfloat16, "W", V * K), B, K, V,
                                        _ptr(logits, torch.float32, "logits", B * V),
                                        _ptr(next_tokens, torch.int32, "next_tokens"),
                                        _stream(stream)))

    def prefill_scratch_bytes(self, T):
        return int(load().nc_prefill_scratch_bytes(self.handle, int(T)))

    def prefill(self, seq, tokens, start, kv, logits, next_tokens=None, scratch=None, stream=None):
        """nc_prefill: tokens [T] int32 (device) enter sequence seq at positions
        start .. start + T - 1 in one forward pass; logits [V] receives the last
        token's logits. scratch: a device buffer of prefill_scratch_bytes(T)
        bytes (allocated here when None)."""
        T = tokens.numel()
        need = self.prefill_scratch_bytes(T)
        if scratch is None:
            scratch = torch.empty(need, dtype=torch.uint8, device=tokens.device)
        s = kv.struct()
        _check(load().nc_prefill(self.handle, int(seq), T, _ptr(tokens, torch.int32, "tokens", T),
                                 int(start), C.byref(s),
                                 _ptr(logits, torch.float32, "logits", self.shape.vocab),
                                 _ptr(next_tokens, torch.int32, "next_tokens"),
                                 _ptr(scratch, None, "scratch"),
                                 scratch.numel() * scratch.element_size(), _stream(stream)))
        return scratch

    def debug_w8a8_codes(self, codes=None, scales=None):
        """nc_debug_w8a8_codes: while set, every step writes its W8A8
        activation codes (int8) and scales (fp32) to these device tensors
        (layout in include/nc.h); None, None turns it off."""
        self._dbg = (codes, scales)  # keep them alive while set
        _check(load().nc_debug_w8a8_codes(
            self.handle, _ptr(codes, torch.int8, "codes"), 0 if codes is None else codes.numel(),
            _ptr(scales, torch.float32, "scales"), 0 if scales is None else scales.numel()))

    def profile_phases(self, enable=True):
        _check(load().nc_profile_phases(self.handle, int(enable)))

    def read_phase_profile(self, stream=None):
        """Last persistent step's phase timestamps (ns), one row per CTA: a
        dict of int64 tensors 'start' [ncta, 5L+1], 'input' [ncta, 5L+1]
        (input arrived), 'cta_start' [ncta], 'cta_end' [ncta], and
        'attn' [ncta, L, 8]: per layer, for the CTA's first attention item,
        the scan combined, the output or partials published, the merge done
        (0 where the CTA did not merge), scan warp 0's first and last K/V
        chunk in, its scan done, and (head size 64) the first chunk's scores
        and weights done."""
        L = self.shape.n_layers
        nph = 5 * L + 1
        per = 2 * nph + 2 + 8 * L
        ncta = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        cap = ncta * per
        buf = (C.c_ulonglong * cap)()
        n = C.c_int()
        _check(load().nc_read_phase_profile(self.handle, _stream(stream), buf, cap, C.byref(n)))
        v = torch.tensor(list(buf)[:n.value], dtype=torch.int64).view(-1, per)
        return {"start": v[:, 0:2 * nph:2], "input": v[:, 1:2 * nph:2], "cta_start": v[:, 2 * nph],
                "cta_end": v[:, 2 * nph + 1], "attn": v[:, 2 * nph + 2:].reshape(-1, L, 8)}

    def device_status(self, stream=None):
        code = C.c_int()
        _check(load().nc_get_device_status(self.handle, _stream(stream), C.byref(code)))
        return code.value
