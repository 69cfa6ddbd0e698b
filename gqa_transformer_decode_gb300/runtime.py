"""Torch-side convenience wrapper around the C ABI.

PyTorch only provides device memory and streams here: weights are uploaded as
int16 tensors holding the bf16 bit patterns, handed to ember_model_create (which
copies them into the library's own layout) and released.  Every forward step
runs in libember.so.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import ember as E


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


class Model:
    """One model on the current CUDA device."""

    def __init__(self, shape, weights: dict, max_tokens: int = 0, max_positions: int = 0,
                 device="cuda", weights_q8: int = 0):
        self.shape = shape
        self.device = torch.device(device)
        self.cfg = E.make_config(shape, max_tokens, max_positions, weights_q8)
        up = {}
        for name, a in weights.items():
            a = np.ascontiguousarray(a)
            assert a.dtype == np.uint16, name
            up[name] = torch.from_numpy(a.view(np.int16)).to(self.device)
        L = shape.layers
        self._lw = (E.ember_layer_weights * L)()
        for l in range(L):
            for f in E.LAYER_FIELDS:
                t = up.get(f"layers.{l}.{f}")
                setattr(self._lw[l], f, None if t is None else t.data_ptr())
        w = E.ember_weights()
        w.embed = up["embed"].data_ptr()
        w.final_norm = up["final_norm"].data_ptr()
        w.cls_w = up["cls_w"].data_ptr() if "cls_w" in up else None
        w.cls_b = up["cls_b"].data_ptr() if "cls_b" in up else None
        w.layers = self._lw
        torch.cuda.synchronize()
        self.handle = E.ember_model_create(self.cfg, w)
        del up
        self.V, self.H = shape.vocab, shape.hidden

    def close(self):
        if getattr(self, "handle", None):
            E.ember_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_alloc(self, max_seqs: int, max_len: int) -> "KVCache":
        return KVCache(self, max_seqs, max_len)

    # -- calls (asynchronous on `stream`; check status with sync_status) ------
    def prefill(self, kv, seq, ids, start_pos, logits=None, argmax=None, hidden=None, stream=None):
        st = E.ember_prefill(self.handle, kv.handle, seq, _ptr(ids), ids.numel(), start_pos,
                             _ptr(logits), _ptr(argmax), _ptr(hidden), _stream_ptr(stream))
        E.check(st, "ember_prefill")

    def prefill_activations(self, kv, seq, ids, start_pos, acts, logits=None, argmax=None, stream=None):
        """Prefill that also writes the residual after every block at the last
        position into acts [layers, hidden] (f32 device tensor)."""
        st = E.ember_prefill_activations(self.handle, kv.handle, seq, _ptr(ids), ids.numel(), start_pos,
                                         _ptr(acts), _ptr(logits), _ptr(argmax), _stream_ptr(stream))
        E.check(st, "ember_prefill_activations")

    def decode_step(self, kv, seqs, ids, positions, logits=None, argmax=None, stream=None):
        st = E.ember_decode_step(self.handle, kv.handle, ids.numel(), _ptr(seqs), _ptr(ids),
                                 _ptr(positions), _ptr(logits), _ptr(argmax), _stream_ptr(stream))

        E.check(st, "ember_decode_step")

    def decode_step_traced(self, kv, seqs, ids, positions, logits=None, argmax=None, stream=None):
        """The same step run eagerly, one kernel at a time, each launch timed
        with CUDA events: [(kernel name, device us)] in launch order."""
        st, tr = E.ember_decode_step_traced(self.handle, kv.handle, ids.numel(), _ptr(seqs), _ptr(ids),
                                            _ptr(positions), _ptr(logits), _ptr(argmax),
                                            _stream_ptr(stream))
        E.check(st, "ember_decode_step_traced")
        return [(E.kernel_name(n), us) for n, us in tr]

    def encode(self, ids, B, T, out=None, hidden=None, stream=None):
        st = E.ember_encode(self.handle, _ptr(ids), B, T, _ptr(out), _ptr(hidden),
                            _stream_ptr(stream))
        E.check(st, "ember_encode")

    def sync_status(self, stream=None) -> int:
        return E.ember_sync_status(self.handle, _stream_ptr(stream))


class KVCache:
    def __init__(self, model: Model, max_seqs: int, max_len: int):
        self.model = model
        self.max_seqs, self.max_len = max_seqs, max_len
        self.handle = E.ember_kv_alloc(model.handle, max_seqs, max_len)

    def reset(self, seq, stream=None):
        E.ember_kv_reset(self.handle, seq, _stream_ptr(stream))

    def set_cursor(self, seq, pos, stream=None):
        E.ember_kv_set_cursor(self.handle, seq, pos, _stream_ptr(stream))

    def tensors(self):
        """(K, V) int16 tensors [S, L, NKV, max_len, D] aliasing the cache (read only)."""
        k, v, strides = E.ember_kv_layout(self.handle)
        s = self.model.shape
        shape = (self.max_seqs, s.layers, s.n_kv_heads, self.max_len, s.head_dim)
        n = int(np.prod(shape))
        out = []
        for p in (k, v):
            buf = _wrap_device(p, n * 2, self.model.device)
            out.append(buf.view(torch.int16).view(shape))
        return tuple(out)

    def close(self):
        if getattr(self, "handle", None):
            E.ember_kv_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _wrap_device(ptr: int, nbytes: int, device) -> torch.Tensor:
    """A uint8 tensor viewing nbytes of device memory owned by the library."""
    class _Holder:
        pass

    h = _Holder()
    h.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False),
                                  "version": 3, "strides": None}
    return torch.as_tensor(h, device=device)
