"""Pins of the oracle's activation probe ([EI] forward_with_activations) and
mean-pooled sensitivity head ([PII] forward(): h.mean(0) @ W.T + b).

- The probe's residual after every block equals the residual stream of the
  independent torch-library composition (tests/test_oracle_forward.py) after
  that block, at the last position; a probe taken before the block, after
  the final norm, or at the wrong position fails it.
- Its last row, RMS-normalised with the final norm, is the forward's own last
  hidden state; with every layer matrix zero every row is the embedding of
  the last token (the residual never changes).
- The pooled head over one position is the per-token label head (the cls
  linear, a different code path); over T positions it is the mean of the
  one-position heads and does not depend on the order of the positions; and
  it equals F.linear of the torch mean.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from test_oracle_forward import SMALL_ENC, SMALL_LLAMA, SMALL_QWEN2, _torch_weights


def torch_residuals(m, w, ids):
    """The residual stream after every block (torch library routines, float64), [L, T, H]."""
    t = _torch_weights(w)
    ids = torch.from_numpy(np.asarray(ids, dtype=np.int64))
    T, H, D, NH, NKV = ids.numel(), m.hidden, m.head_dim, m.n_heads, m.n_kv_heads
    f = m.rope_theta ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
    if m.rope_llama3:
        z = ((m.rs_orig_max_pos * f / (2 * math.pi) - m.rs_low) / (m.rs_high - m.rs_low)).clip(0, 1)
        f = f * torch.lerp(torch.tensor(1 / m.rs_factor, dtype=torch.float64),
                           torch.tensor(1.0, dtype=torch.float64), z)
    rot = torch.polar(torch.ones(T, D // 2, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * f)

    def rope(x):
        zz = torch.complex(x[..., : D // 2], x[..., D // 2:]) * rot[:, None, :]
        return torch.cat([zz.real, zz.imag], -1)

    x = F.embedding(ids, t["embed"])
    out = []
    for l in range(m.layers):
        p = f"layers.{l}."
        xb = F.rms_norm(x, (H,), t[p + "attn_norm"], m.rms_eps)
        q = F.linear(xb, t[p + "wq"], t.get(p + "bq")).view(T, NH, D)
        k = F.linear(xb, t[p + "wk"], t.get(p + "bk")).view(T, NKV, D)
        v = F.linear(xb, t[p + "wv"], t.get(p + "bv")).view(T, NKV, D)
        if m.qk_norm:
            q = F.rms_norm(q, (D,), t[p + "q_norm"], m.rms_eps)
            k = F.rms_norm(k, (D,), t[p + "k_norm"], m.rms_eps)
        q, k = rope(q), rope(k)
        a = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                           v.transpose(0, 1)[None], is_causal=bool(m.causal),
                                           enable_gqa=True)
        x = x + F.linear(a[0].transpose(0, 1).reshape(T, NH * D), t[p + "wo"])
        xb = F.rms_norm(x, (H,), t[p + "mlp_norm"], m.rms_eps)
        x = x + F.linear(F.silu(F.linear(xb, t[p + "w_gate"])) * F.linear(xb, t[p + "w_up"]),
                         t[p + "w_down"])
        out.append(x.numpy().copy())
    return np.stack(out)


@pytest.mark.parametrize("shape,T", [(synth.TINY, 8), (SMALL_QWEN2, 13), (SMALL_LLAMA, 11),
                                     (SMALL_ENC, 9)])
def test_probe_matches_the_torch_residual_stream_after_every_block(shape, T):
    w = synth.weights_bf16(shape)
    ids = synth.prompt_ids(shape, T)
    om = O.OracleModel(shape, w)
    acts, lg = om.forward_activations(ids)
    ref = torch_residuals(shape, w, ids)
    assert acts.shape == (shape.layers, shape.hidden)
    assert np.allclose(acts, ref[:, -1], rtol=1e-10, atol=1e-11)
    # a probe one block early, or at another position, would not match
    if shape.layers > 1:
        assert not np.allclose(acts[1:], ref[:-1, -1], rtol=1e-6, atol=1e-8)
    assert not np.allclose(acts, ref[:, 0], rtol=1e-6, atol=1e-8)
    # the last row is the pre-norm state of the last position; logits are that position's
    h, lg_full, _ = om.forward_full(ids)
    g = O.bf16_decode(w["final_norm"])
    assert np.allclose(O.rmsnorm(acts[-1], g, shape.rms_eps), h[-1], rtol=1e-12, atol=1e-14)
    assert np.allclose(lg, lg_full[-1], rtol=1e-12, atol=1e-13)


def test_probe_of_zero_layers_is_the_embedding():
    shape = SMALL_QWEN2
    w = synth.weights_f32(shape)
    for k in list(w):
        if k.startswith("layers.") and not k.endswith("norm"):
            w[k] = np.zeros_like(w[k])
    ids = synth.prompt_ids(shape, 6)
    acts, _ = O.OracleModel(shape, w).forward_activations(ids, logits=False)
    e = w["embed"][ids[-1]].astype(np.float64)
    for l in range(shape.layers):
        assert np.array_equal(acts[l], e)


def test_mean_pooled_head():
    shape = SMALL_ENC
    w = synth.weights_bf16(shape)
    T = 10
    ids = synth.prompt_ids(shape, T)
    h, _, cls = O.OracleModel(shape, w).forward_full(ids, logits=False, cls=True)
    W = O.bf16_decode(w["cls_w"])
    b = O.bf16_decode(w["cls_b"])
    # one position: the token label head
    for t in (0, 4, T - 1):
        assert np.allclose(O.mean_pooled_head(h[t:t + 1], W, b), cls[t], rtol=1e-12, atol=1e-13)
    # T positions: the mean of the one-position heads, independent of order
    pooled = O.mean_pooled_head(h, W, b)
    assert np.allclose(pooled, cls.mean(0), rtol=1e-12, atol=1e-13)
    perm = np.random.default_rng(1).permutation(T)
    assert np.allclose(O.mean_pooled_head(h[perm], W, b), pooled, rtol=1e-13, atol=1e-14)
    ref = F.linear(torch.from_numpy(h).mean(0), torch.from_numpy(W).double(), torch.from_numpy(b).double())
    assert np.allclose(pooled, ref.numpy(), rtol=1e-12, atol=1e-13)
    # no bias
    assert np.allclose(O.mean_pooled_head(h, W), pooled - b, rtol=1e-12, atol=1e-13)
