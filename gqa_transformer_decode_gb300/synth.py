"""Seeded synthetic inputs: model shapes, random weights and token ids.

This module is the only thing the CUDA library's tests and the CPU oracle
share.  It holds no step of the forward pass: it draws numbers and rounds them
to the bf16 storage format, nothing else.

Generator: a counter-based SplitMix64 stream per tensor (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), keyed by
``seed`` mixed with the FNV-1a hash of the tensor name, so any chunk of any
tensor can be drawn independently and in parallel.  Normals come from the
Box-Muller transform in float64.  Everything is plain numpy uint64 arithmetic,
so the draws are identical on every machine and numpy version.

Weight recipe (the synthetic stand-in for the checkpoints the pages load):
matrices, biases and the classifier ~ N(0, 0.02); every norm weight
(input/post-attention/final/q/k norms) ~ 1 + N(0, 0.1); drawn in float64,
rounded to float32, then to bf16 with round-to-nearest-even.  Token ids are
uniform over [0, vocab).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, asdict, field

import numpy as np

WEIGHT_SEED = 20261202
IDS_SEED = WEIGHT_SEED + 1

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


@dataclass(frozen=True)
class ModelShape:
    """Hyper-parameters of one decoder (field names follow the C ``ember_config``)."""

    name: str
    vocab: int
    hidden: int
    layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ff: int
    rope_theta: float
    rms_eps: float = 1e-6
    rope_llama3: int = 0
    rs_factor: float = 1.0
    rs_low: float = 1.0
    rs_high: float = 4.0
    rs_orig_max_pos: int = 8192
    qkv_bias: int = 0
    qk_norm: int = 0
    causal: int = 1
    n_labels: int = 0

    def asdict(self):
        return asdict(self)

    def params(self) -> int:
        H, D, F = self.hidden, self.head_dim, self.ff
        q, kv = self.n_heads * D, self.n_kv_heads * D
        per = 2 * H + (q + 2 * kv) * H + q * H + 3 * F * H
        if self.qkv_bias:
            per += q + 2 * kv
        if self.qk_norm:
            per += 2 * D
        total = self.layers * per + self.vocab * H + H
        if self.n_labels:
            total += self.n_labels * H + self.n_labels
        return total


@dataclass(frozen=True)
class Workload:
    """One benchmark / parity workload: a model shape plus the token pattern."""

    key: str
    model: ModelShape
    batch: int
    prompt: int
    steps: int
    note: str = ""
    extra: dict = field(default_factory=dict)
    weights_q8: int = 0      # 1: the layer matrices run as q8_0 blocks


TINY = ModelShape("tiny-qwen2", vocab=256, hidden=64, layers=2, n_heads=4, n_kv_heads=2,
                  head_dim=16, ff=128, rope_theta=1e4, qkv_bias=1)
QWEN25_05B = ModelShape("qwen2.5-0.5b-shape", vocab=151936, hidden=896, layers=24, n_heads=14,
                        n_kv_heads=2, head_dim=64, ff=4864, rope_theta=1e6, qkv_bias=1)
LLAMA32_1B = ModelShape("llama-3.2-1b-shape", vocab=128256, hidden=2048, layers=16, n_heads=32,
                        n_kv_heads=8, head_dim=64, ff=8192, rope_theta=5e5, rope_llama3=1,
                        rs_factor=32.0, rs_low=1.0, rs_high=4.0, rs_orig_max_pos=8192)
QWEN3_ENC = ModelShape("qwen3-encoder-shape", vocab=151936, hidden=1024, layers=28, n_heads=16,
                       n_kv_heads=8, head_dim=128, ff=3072, rope_theta=1e6, qk_norm=1, causal=0,
                       n_labels=16)

WORKLOADS = {
    "tiny": Workload("tiny", TINY, batch=1, prompt=8, steps=16,
                     note="f32 weights N(0,0.02); bf16-rounded copy for the GPU"),
    "qwen2.5-0.5b": Workload("qwen2.5-0.5b", QWEN25_05B, batch=1, prompt=128, steps=128),
    "llama-3.2-1b": Workload("llama-3.2-1b", LLAMA32_1B, batch=1, prompt=2048, steps=256),
    "qwen2.5-0.5b-q8_0": Workload("qwen2.5-0.5b-q8_0", QWEN25_05B, batch=1, prompt=128, steps=128,
                                  note="layer matrices quantized to q8_0 at model creation",
                                  weights_q8=1),
    "qwen2.5-0.5b-b64": Workload("qwen2.5-0.5b-b64", QWEN25_05B, batch=64, prompt=4096, steps=64),
    "qwen3-encoder": Workload("qwen3-encoder", QWEN3_ENC, batch=8, prompt=512, steps=0),
}


def _fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, name: str) -> np.uint64:
    k = np.array([(seed ^ _fnv1a64(name)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(k + _GAMMA)[0]


def _words(key: np.uint64, start: int, count: int) -> np.ndarray:
    """SplitMix64 outputs start .. start+count-1 of the stream keyed by ``key``."""
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + ctr * _GAMMA)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


_CHUNK = 1 << 18


def normal(seed: int, name: str, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n float64 draws of N(mean, std^2) from the stream (seed, name)."""
    key = _key(seed, name)
    out = np.empty(n, dtype=np.float64)

    def fill(lo: int):
        hi = min(n, lo + _CHUNK)
        w = _words(key, 2 * lo, 2 * (hi - lo))
        u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        out[lo:hi] = mean + std * (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2))

    list(_pool().map(fill, range(0, n, _CHUNK)))
    return out


def uniform_ids(seed: int, name: str, n: int, vocab: int) -> np.ndarray:
    """n int32 token ids uniform over [0, vocab)."""
    w = _words(_key(seed, name), 0, n)
    return (((w >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)).astype(np.int32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _tensor_list(m: ModelShape):
    """(name, shape, kind) for every weight; kind 'w' = N(0,.02), 'n' = 1+N(0,.1)."""
    H, D, F = m.hidden, m.head_dim, m.ff
    q, kv = m.n_heads * D, m.n_kv_heads * D
    out = [("embed", (m.vocab, H), "w"), ("final_norm", (H,), "n")]
    if m.n_labels:
        out += [("cls_w", (m.n_labels, H), "w"), ("cls_b", (m.n_labels,), "w")]
    for l in range(m.layers):
        p = f"layers.{l}."
        out += [(p + "attn_norm", (H,), "n"), (p + "wq", (q, H), "w"), (p + "wk", (kv, H), "w"),
                (p + "wv", (kv, H), "w")]
        if m.qkv_bias:
            out += [(p + "bq", (q,), "w"), (p + "bk", (kv,), "w"), (p + "bv", (kv,), "w")]
        if m.qk_norm:
            out += [(p + "q_norm", (D,), "n"), (p + "k_norm", (D,), "n")]
        out += [(p + "wo", (H, q), "w"), (p + "mlp_norm", (H,), "n"), (p + "w_gate", (F, H), "w"),
                (p + "w_up", (F, H), "w"), (p + "w_down", (H, F), "w")]
    return out


def weights_f32(m: ModelShape, seed: int = WEIGHT_SEED) -> dict:
    """Unrounded float32 draws, name -> array (the 'f32 random weights' form)."""
    out = {}
    for name, shape, kind in _tensor_list(m):
        n = int(np.prod(shape))
        mean, std = (1.0, 0.1) if kind == "n" else (0.0, 0.02)
        out[name] = normal(seed, name, n, mean, std).astype(np.float32).reshape(shape)
    return out


def weights_bf16(m: ModelShape, seed: int = WEIGHT_SEED) -> dict:
    """bf16 bit patterns (uint16), name -> array: the stored weights both sides use."""
    out = {}
    for name, shape, kind in _tensor_list(m):
        n = int(np.prod(shape))
        mean, std = (1.0, 0.1) if kind == "n" else (0.0, 0.02)
        x = normal(seed, name, n, mean, std).astype(np.float32)
        out[name] = f32_to_bf16_bits(x).reshape(shape)
    return out


def prompt_ids(m: ModelShape, n: int, seq: int = 0, seed: int = IDS_SEED) -> np.ndarray:
    """The uniform prompt of sequence ``seq``."""
    return uniform_ids(seed, f"prompt.{seq}", n, m.vocab)
