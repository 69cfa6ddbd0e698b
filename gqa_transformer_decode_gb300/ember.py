"""ctypes binding of the C ABI in include/ember.h (argument marshalling only).

Every step of the forward runs in the CUDA library ``_build/libember.so``;
this module only builds the C structs, passes device pointers and raises on
a non-zero status.  Importing it on a machine without the built library and
without nvcc fails loudly: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

P = C.c_void_p

EMBER_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "CAPACITY", 3: "STATE", 4: "TOKEN", 5: "TIMEOUT",
                6: "CUDA", 7: "OOM", 8: "UNSUPPORTED"}


class EmberError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")


class ember_config(C.Structure):
    _fields_ = [("vocab", C.c_int32), ("hidden", C.c_int32), ("layers", C.c_int32),
                ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("ff", C.c_int32), ("rope_theta", C.c_double), ("rms_eps", C.c_double),
                ("rope_llama3", C.c_int32), ("rs_factor", C.c_double), ("rs_low", C.c_double),
                ("rs_high", C.c_double), ("rs_orig_max_pos", C.c_int32), ("qkv_bias", C.c_int32),
                ("qk_norm", C.c_int32), ("causal", C.c_int32), ("n_labels", C.c_int32),
                ("max_tokens", C.c_int32), ("max_positions", C.c_int32),
                ("weights_q8", C.c_int32)]


LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "bq", "bk", "bv", "q_norm", "k_norm", "wo",
                "mlp_norm", "w_gate", "w_up", "w_down")


class ember_layer_weights(C.Structure):
    _fields_ = [(n, P) for n in LAYER_FIELDS]


class ember_weights(C.Structure):
    _fields_ = [("embed", P), ("final_norm", P), ("cls_w", P), ("cls_b", P),
                ("layers", C.POINTER(ember_layer_weights))]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libember.so, building it first if the sources are newer."""
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("EMBER_LIB")   # an alternative build of the same sources
    if not path:
        if not _build.up_to_date():
            _build.build()
        path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing and could not be built")
    L = C.CDLL(path)
    st = C.c_int
    sig = {
        "ember_model_create": (st, [C.POINTER(ember_config), C.POINTER(ember_weights), C.POINTER(P)]),
        "ember_model_destroy": (None, [P]),
        "ember_kv_bytes": (C.c_size_t, [C.POINTER(ember_config), C.c_int32, C.c_int32]),
        "ember_kv_alloc": (st, [P, C.c_int32, C.c_int32, C.POINTER(P)]),
        "ember_kv_free": (None, [P]),
        "ember_kv_reset": (st, [P, C.c_int32, P]),
        "ember_kv_set_cursor": (st, [P, C.c_int32, C.c_int32, P]),
        "ember_kv_layout": (st, [P, C.POINTER(P), C.POINTER(P), C.POINTER(C.c_int64)]),
        "ember_prefill": (st, [P, P, C.c_int32, P, C.c_int32, C.c_int32, P, P, P, P]),
        "ember_decode_step": (st, [P, P, C.c_int32, P, P, P, P, P, P]),
        "ember_decode_step_traced": (st, [P, P, C.c_int32, P, P, P, P, P, P, C.POINTER(C.c_float),
                                          C.POINTER(C.c_char_p), C.c_int32, C.POINTER(C.c_int32)]),
        "ember_encode": (st, [P, P, C.c_int32, C.c_int32, P, P, P]),
        "ember_sync_status": (st, [P, P]),
        "ember_last_error": (C.c_char_p, []),
        "ember_rope_store": (st, [P, C.c_int32, C.c_int32, C.c_int32, P, P, P, P]),
        "ember_gemm_bf16": (st, [P, P, P, C.c_int32, C.c_int32, C.c_int32, P]),
        "ember_gemv_bf16": (st, [P, C.c_int32, C.c_int32, P, C.c_int32, P, P]),
        "ember_q8_0_quantize": (st, [P, C.c_int64, P, P, P]),
        "ember_gemv_q8_0": (st, [P, P, C.c_int32, C.c_int32, P, C.c_int32, P, P]),
        "ember_gemv_argmax_noalloc": (st, [P, C.c_int32, C.c_int32, P, C.c_int32, P, P, P]),
        "ember_sample": (st, [P, C.c_int32, C.c_int32, C.c_int32, C.c_float, C.c_int32, C.c_float, P, P,
                              P]),
        "ember_prefill_activations": (st, [P, P, C.c_int32, P, C.c_int32, C.c_int32, P, P, P, P]),
        "ember_mean_pooled_head": (st, [P, C.c_int32, C.c_int32, C.c_int32, P, P, C.c_int32, P, P]),
        "ember_test_bounded_wait": (st, [P, C.c_int32, C.c_int64, P]),
        "ember_kernel_launches": (C.c_uint64, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def last_error() -> str:
    return load().ember_last_error().decode(errors="replace")


def check(status: int, where: str):
    if status != EMBER_OK:
        raise EmberError(status, where, last_error())


def make_config(shape, max_tokens: int = 0, max_positions: int = 0, weights_q8: int = 0) -> ember_config:
    d = shape if isinstance(shape, dict) else shape.asdict()
    c = ember_config()
    for name, _ in ember_config._fields_:
        if name in d:
            setattr(c, name, d[name])
    c.max_tokens = max_tokens
    c.max_positions = max_positions
    c.weights_q8 = weights_q8
    return c


# Names of the C ABI, re-exported with the same spelling.
def ember_model_create(cfg, weights):
    out = P()
    check(load().ember_model_create(C.byref(cfg), C.byref(weights), C.byref(out)),
          "ember_model_create")
    return out


def ember_model_destroy(m):
    load().ember_model_destroy(m)


def ember_kv_bytes(cfg, max_seqs, max_len) -> int:
    return int(load().ember_kv_bytes(C.byref(cfg), max_seqs, max_len))


def ember_kv_alloc(m, max_seqs, max_len):
    out = P()
    check(load().ember_kv_alloc(m, max_seqs, max_len, C.byref(out)), "ember_kv_alloc")
    return out


def ember_kv_free(kv):
    load().ember_kv_free(kv)


def ember_kv_reset(kv, seq, stream=None):
    check(load().ember_kv_reset(kv, seq, stream), "ember_kv_reset")


def ember_kv_set_cursor(kv, seq, pos, stream=None):
    check(load().ember_kv_set_cursor(kv, seq, pos, stream), "ember_kv_set_cursor")


def ember_kv_layout(kv):
    k, v = P(), P()
    strides = (C.c_int64 * 4)()
    check(load().ember_kv_layout(kv, C.byref(k), C.byref(v), strides), "ember_kv_layout")
    return k.value, v.value, list(strides)


def ember_prefill(m, kv, seq, ids, n, start_pos, logits, argmax, hidden, stream):
    return load().ember_prefill(m, kv, seq, ids, n, start_pos, logits, argmax, hidden, stream)


def ember_decode_step(m, kv, batch, seqs, ids, positions, logits, argmax, stream):
    return load().ember_decode_step(m, kv, batch, seqs, ids, positions, logits, argmax, stream)


def ember_decode_step_traced(m, kv, batch, seqs, ids, positions, logits, argmax, stream, cap=4096):
    """-> (status, [(mangled kernel name, device us)] in launch order)."""
    us = (C.c_float * cap)()
    names = (C.c_char_p * cap)()
    n = C.c_int32(0)
    st = load().ember_decode_step_traced(m, kv, batch, seqs, ids, positions, logits, argmax, stream,
                                         us, names, cap, C.byref(n))
    k = min(n.value, cap) if st == EMBER_OK else 0
    return st, [(names[i].decode(errors="replace"), float(us[i])) for i in range(k)]


def kernel_name(mangled: str) -> str:
    """k_fused_attn<64,4> from the runtime's mangled name of an ember kernel."""
    import re
    m = re.match(r"_ZN5ember(\d+)", mangled)
    if not m:
        return mangled
    n = int(m.group(1))
    name, rest = mangled[m.end():m.end() + n], mangled[m.end() + n:]
    t = re.match(r"I((?:L[a-z]\d+E)+)E", rest)
    if not t:
        return name
    return name + "<" + ",".join(re.findall(r"L[a-z](\d+)E", t.group(1))) + ">"


def ember_encode(m, ids, B, T, out, hidden, stream):
    return load().ember_encode(m, ids, B, T, out, hidden, stream)


def ember_sync_status(m, stream) -> int:
    return load().ember_sync_status(m, stream)


def ember_rope_store(x, n_tok, n_heads, head_dim, cos_t, sin_t, out, stream):
    return load().ember_rope_store(x, n_tok, n_heads, head_dim, cos_t, sin_t, out, stream)


def ember_gemm_bf16(A, B, D, M, N, K, stream):
    return load().ember_gemm_bf16(A, B, D, M, N, K, stream)


def ember_gemv_bf16(W, N, K, x, nb, y, stream):
    return load().ember_gemv_bf16(W, N, K, x, nb, y, stream)


def ember_gemv_argmax_noalloc(W, N, K, x, nb, y, argmax, stream):
    return load().ember_gemv_argmax_noalloc(W, N, K, x, nb, y, argmax, stream)


def ember_q8_0_quantize(w, n, q, d, stream):
    return load().ember_q8_0_quantize(w, n, q, d, stream)


def ember_gemv_q8_0(q, d, N, K, x, nb, y, stream):
    return load().ember_gemv_q8_0(q, d, N, K, x, nb, y, stream)


def ember_sample(logits, B, V, ldl, temperature, top_k, top_p, r, out, stream):
    return load().ember_sample(logits, B, V, ldl, temperature, top_k, top_p, r, out, stream)


def ember_prefill_activations(m, kv, seq, ids, n, start_pos, acts, logits, argmax, stream):
    return load().ember_prefill_activations(m, kv, seq, ids, n, start_pos, acts, logits, argmax, stream)


def ember_mean_pooled_head(hidden, B, T, H, w, b, n_out, out, stream):
    return load().ember_mean_pooled_head(hidden, B, T, H, w, b, n_out, out, stream)


def ember_kernel_launches() -> int:
    return int(load().ember_kernel_launches())
