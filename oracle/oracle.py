"""ctypes front end of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg are the only callers.  Nothing here imports the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


class OrcConfig(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("vocab", "hidden", "layers", "n_heads", "n_kv_heads", "head_dim", "ff")] + [
        ("rope_theta", C.c_double), ("rms_eps", C.c_double), ("rope_llama3", C.c_int),
        ("rs_factor", C.c_double), ("rs_low", C.c_double), ("rs_high", C.c_double),
        ("rs_orig_max_pos", C.c_int), ("qkv_bias", C.c_int), ("qk_norm", C.c_int),
        ("causal", C.c_int), ("n_labels", C.c_int)]


_LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "bq", "bk", "bv", "q_norm", "k_norm", "wo",
                 "mlp_norm", "w_gate", "w_up", "w_down")


class OrcLayer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _LAYER_FIELDS]


class OrcModel(C.Structure):
    _fields_ = [("cfg", OrcConfig), ("embed", C.c_void_p), ("final_norm", C.c_void_p),
                ("cls_w", C.c_void_p), ("cls_b", C.c_void_p), ("layers", C.POINTER(OrcLayer))]


class OrcCache(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("layers", "n_kv_heads", "head_dim", "max_len", "len", "kv_bf16")] + [
        ("k", C.c_void_p), ("v", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.orc_bf16_decode.argtypes = [P, P, C.c_size_t]
        L.orc_bf16_round.argtypes = [C.c_double]
        L.orc_bf16_round.restype = C.c_uint16
        L.orc_rmsnorm.argtypes = [P, P, C.c_int, C.c_double, P]
        L.orc_rope_inv_freq.argtypes = [C.POINTER(OrcConfig), P]
        L.orc_rope_apply.argtypes = [P, C.c_int, P, C.c_long]
        L.orc_rope_table_f32.argtypes = [C.POINTER(OrcConfig), C.c_long, C.c_int, P, P]
        L.orc_rope_store_bf16_f32.argtypes = [P, C.c_int, C.c_int, P, P, P]
        L.orc_softmax.argtypes = [P, C.c_int]
        L.orc_silu.argtypes = [C.c_double]
        L.orc_silu.restype = C.c_double
        L.orc_argmax.argtypes = [P, C.c_long]
        L.orc_argmax.restype = C.c_long
        L.orc_attention.argtypes = [P, P, P, C.c_int, C.c_int, C.c_int, C.c_long, C.c_long, P]
        L.orc_validate.argtypes = [C.POINTER(OrcConfig)]
        L.orc_forward_full.argtypes = [C.POINTER(OrcModel), P, C.c_int, P, P, P]
        L.orc_forward_activations.argtypes = [C.POINTER(OrcModel), P, C.c_int, P, P]
        L.orc_mean_pooled_head.argtypes = [P, C.c_int, C.c_int, P, P, C.c_int, P]
        L.orc_f16_round.argtypes = [C.c_float]
        L.orc_f16_round.restype = C.c_uint16
        L.orc_f16_decode.argtypes = [C.c_uint16]
        L.orc_f16_decode.restype = C.c_float
        L.orc_q8_0_dequant.argtypes = [P, C.c_long, P]
        L.orc_q8_0_quantize.argtypes = [P, C.c_long, P]
        L.orc_cache_new.argtypes = [C.POINTER(OrcConfig), C.c_int, C.c_int]
        L.orc_cache_new.restype = C.POINTER(OrcCache)
        L.orc_cache_free.argtypes = [C.POINTER(OrcCache)]
        L.orc_forward_cached.argtypes = [C.POINTER(OrcModel), C.POINTER(OrcCache), P, C.c_int,
                                         C.c_int, P, P]
        L.orc_greedy.argtypes = [C.POINTER(OrcModel), C.POINTER(OrcCache), P, C.c_int, C.c_int,
                                 P, P, P, P]
        L.orc_num_threads.restype = C.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def make_config(shape) -> OrcConfig:
    d = shape if isinstance(shape, dict) else shape.asdict()
    c = OrcConfig()
    for name, _ in OrcConfig._fields_:
        setattr(c, name, d[name])
    return c


# ---- primitives -------------------------------------------------------------

def bf16_decode(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    lib().orc_bf16_decode(_p(bits), _p(out), bits.size)
    return out


def bf16_round(x: float) -> int:
    return int(lib().orc_bf16_round(float(x)))


def rmsnorm(x, w, eps):
    x = _f64(x)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(w), x.size, float(eps), _p(y))
    return y


def rope_inv_freq(shape) -> np.ndarray:
    cfg = make_config(shape)
    out = np.empty(cfg.head_dim // 2, dtype=np.float64)
    lib().orc_rope_inv_freq(C.byref(cfg), _p(out))
    return out


def rope_apply(v, inv_freq, pos):
    v = _f64(v).copy()
    inv = _f64(inv_freq)
    lib().orc_rope_apply(_p(v), v.size, _p(inv), int(pos))
    return v


def rope_table_f32(shape, pos0, npos):
    cfg = make_config(shape)
    half = cfg.head_dim // 2
    cos_t = np.empty((npos, half), dtype=np.float32)
    sin_t = np.empty((npos, half), dtype=np.float32)
    lib().orc_rope_table_f32(C.byref(cfg), int(pos0), int(npos), _p(cos_t), _p(sin_t))
    return cos_t, sin_t


def rope_store_bf16_f32(x, n_heads, head_dim, cos_row, sin_row):
    x = np.ascontiguousarray(x, dtype=np.float32)
    c = np.ascontiguousarray(cos_row, dtype=np.float32)
    s = np.ascontiguousarray(sin_row, dtype=np.float32)
    out = np.empty(n_heads * head_dim, dtype=np.uint16)
    lib().orc_rope_store_bf16_f32(_p(x), n_heads, head_dim, _p(c), _p(s), _p(out))
    return out


def softmax(s):
    s = _f64(s).copy()
    lib().orc_softmax(_p(s), s.size)
    return s


def silu(g: float) -> float:
    return float(lib().orc_silu(float(g)))


def argmax(v) -> int:
    v = _f64(v)
    return int(lib().orc_argmax(_p(v), v.size))


def attention(q, k, v, n_heads, n_kv_heads, head_dim, n_keys=None):
    """q: [NH*D]; k, v: [NKV, S, D]; attends over the first n_keys rows."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = k.shape[1]
    n_keys = S if n_keys is None else n_keys
    out = np.empty(n_heads * head_dim, dtype=np.float64)
    lib().orc_attention(_p(q), _p(k), _p(v), n_heads, n_kv_heads, head_dim, S * head_dim,
                        int(n_keys), _p(out))
    return out


def f16_round(x: float) -> int:
    return int(lib().orc_f16_round(float(x)))


def f16_decode(h: int) -> float:
    return float(lib().orc_f16_decode(int(h)))


def q8_0_quantize(x) -> np.ndarray:
    """[EI] q8_0 blocks (uint8 [n/32, 34]) of f32 values x (n a multiple of 32)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert x.size % 32 == 0
    out = np.empty((x.size // 32, 34), dtype=np.uint8)
    lib().orc_q8_0_quantize(_p(x), x.size, _p(out))
    return out


def q8_0_dequant(blocks) -> np.ndarray:
    """f32 values of q8_0 blocks (uint8 [n_blocks, 34])."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 34)
    out = np.empty(b.shape[0] * 32, dtype=np.float32)
    lib().orc_q8_0_dequant(_p(b), b.shape[0], _p(out))
    return out


LAYER_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def q8_0_layer_weights(weights: dict, layers: int) -> dict:
    """A model's weights with every layer matrix replaced by the f32 decode of
    its q8_0 encoding (embedding, head, norms and biases as given): the
    values a q8_0 model computes with."""
    out = dict(weights)
    for l in range(layers):
        for m in LAYER_MATRICES:
            k = f"layers.{l}.{m}"
            a = out[k]
            a = bf16_decode(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float32)
            out[k] = q8_0_dequant(q8_0_quantize(a)).reshape(a.shape)
    return out


def mean_pooled_head(hidden, w, b=None):
    """[PII] forward() sensitivity head over final-normed states hidden [T, H]:
    mean over positions, then . w[j] + b[j] for w [n_out, H] (f32 values)."""
    h = np.ascontiguousarray(hidden, dtype=np.float64)
    T, H = h.shape
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1, H)
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    out = np.empty(w.shape[0], dtype=np.float64)
    lib().orc_mean_pooled_head(_p(h), T, H, _p(w), _p(bb), w.shape[0], _p(out))
    return out


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ---- whole model ------------------------------------------------------------

class OracleModel:
    """The oracle's view of one model: f32 weights decoded from bf16 bits by
    the oracle's own decode (or given as f32 directly)."""

    def __init__(self, shape, weights: dict):
        self.shape = shape
        self.cfg = make_config(shape)
        if lib().orc_validate(C.byref(self.cfg)) != 0:
            raise ValueError("invalid config")
        self._keep = {}
        for name, arr in weights.items():
            if arr.dtype == np.uint16:
                self._keep[name] = bf16_decode(arr)
            else:
                self._keep[name] = np.ascontiguousarray(arr, dtype=np.float32)
        L = self.cfg.layers
        self._layers = (OrcLayer * L)()
        for l in range(L):
            for f in _LAYER_FIELDS:
                a = self._keep.get(f"layers.{l}.{f}")
                setattr(self._layers[l], f, None if a is None else a.ctypes.data)
        m = OrcModel()
        m.cfg = self.cfg
        m.embed = self._keep["embed"].ctypes.data
        m.final_norm = self._keep["final_norm"].ctypes.data
        m.cls_w = self._keep["cls_w"].ctypes.data if "cls_w" in self._keep else None
        m.cls_b = self._keep["cls_b"].ctypes.data if "cls_b" in self._keep else None
        m.layers = self._layers
        self._m = m

    @property
    def H(self):
        return self.cfg.hidden

    @property
    def V(self):
        return self.cfg.vocab

    def forward_full(self, ids, logits=True, cls=False):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T = ids.size
        hid = np.empty((T, self.H), dtype=np.float64)
        lg = np.empty((T, self.V), dtype=np.float64) if logits else None
        cl = np.empty((T, self.cfg.n_labels), dtype=np.float64) if cls else None
        rc = lib().orc_forward_full(C.byref(self._m), _p(ids), T, _p(hid), _p(lg), _p(cl))
        if rc != 0:
            raise RuntimeError(f"orc_forward_full rc={rc}")
        return hid, lg, cl

    def forward_activations(self, ids, logits=True):
        """[EI] forward_with_activations: the residual stream at the last
        position after every block [L, H], and the last position's logits."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        acts = np.empty((self.cfg.layers, self.H), dtype=np.float64)
        lg = np.empty(self.V, dtype=np.float64) if logits else None
        rc = lib().orc_forward_activations(C.byref(self._m), _p(ids), ids.size, _p(acts), _p(lg))
        if rc != 0:
            raise RuntimeError(f"orc_forward_activations rc={rc}")
        return acts, lg

    def new_cache(self, max_len, kv_bf16=False):
        return OracleCache(self, max_len, kv_bf16)

    def forward_cached(self, cache, ids, start_pos=None, logits=True):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        n = ids.size
        sp = cache.len if start_pos is None else start_pos
        hid = np.empty((n, self.H), dtype=np.float64)
        lg = np.empty(self.V, dtype=np.float64) if logits else None
        rc = lib().orc_forward_cached(C.byref(self._m), cache.ptr, _p(ids), n, int(sp), _p(hid),
                                      _p(lg))
        return rc, hid, lg

    def greedy(self, prompt, n_steps, forced=None, kv_bf16=False, max_len=None, logits=True,
               hidden=True):
        prompt = np.ascontiguousarray(prompt, dtype=np.int32)
        cache = self.new_cache(max_len or (prompt.size + n_steps + 1), kv_bf16)
        toks = np.empty(n_steps + 1, dtype=np.int32)
        lg = np.empty((n_steps + 1, self.V), dtype=np.float64) if logits else None
        hd = np.empty((n_steps + 1, self.H), dtype=np.float64) if hidden else None
        fz = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        rc = lib().orc_greedy(C.byref(self._m), cache.ptr, _p(prompt), prompt.size, n_steps,
                              _p(fz), _p(toks), _p(lg), _p(hd))
        if rc != 0:
            raise RuntimeError(f"orc_greedy rc={rc}")
        return toks, lg, hd


class OracleCache:
    def __init__(self, model: OracleModel, max_len: int, kv_bf16: bool):
        self.ptr = lib().orc_cache_new(C.byref(model.cfg), int(max_len), int(bool(kv_bf16)))
        if not self.ptr:
            raise MemoryError("orc_cache_new failed")
        c = model.cfg
        self._shape = (c.layers, c.n_kv_heads, max_len, c.head_dim)

    @property
    def len(self):
        return self.ptr.contents.len

    def load(self, k_bits, v_bits, length):
        """Start from a given cache: rows [0, length) of K and V (bf16 bit
        patterns [L, NKV, >= length, D], decoded exactly by the oracle's own
        bf16 decode) become the cache contents and the cursor becomes length
        ([EI] kv cache: the cursor counts the rows every layer has stored).  A
        cached step then computes the next token from exactly that history."""
        L, NKV, max_len, D = self._shape
        if not 0 <= length <= max_len:
            raise ValueError("length outside the cache")
        k, v = self.arrays()
        for dst, src in ((k, k_bits), (v, v_bits)):
            src = np.asarray(src).view(np.uint16)[:, :, :length]
            if src.shape != (L, NKV, length, D):
                raise ValueError(f"cache rows of shape {src.shape}, want {(L, NKV, length, D)}")
            dst[:, :, :length] = bf16_decode(np.ascontiguousarray(src))
            dst[:, :, length:] = 0.0
        self.ptr.contents.len = int(length)

    def arrays(self):
        """(K, V) as float64 views [L, NKV, max_len, D] of the oracle's cache."""
        n = int(np.prod(self._shape))
        k = np.ctypeslib.as_array(C.cast(self.ptr.contents.k, C.POINTER(C.c_double)), (n,))
        v = np.ctypeslib.as_array(C.cast(self.ptr.contents.v, C.POINTER(C.c_double)), (n,))
        return k.reshape(self._shape), v.reshape(self._shape)

    def __del__(self):
        if getattr(self, "ptr", None):
            lib().orc_cache_free(self.ptr)
            self.ptr = None
