"""Pins of the oracle's whole forward pass.

1. Against an independent composition of torch library routines in float64
   (F.embedding, F.rms_norm, F.linear, F.scaled_dot_product_attention with
   enable_gqa, F.silu) with RoPE written as complex multiplication: a dropped
   term, a swapped gate/up, a transposed weight or a wrong GQA mapping in the
   oracle fails it.
2. Invariants the pages fix: whole-sequence == prefill + one cached step per
   token (ember internals, the KV-cache prefill bug), token-by-token prefill ==
   batched prefill, causality, a bidirectional single token == causal, the
   all-zero-layers closed form, determinism across thread counts.
3. Boundary errors (Falcon-H1-0.5B-Rust validate() / logits()).
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Small shapes that exercise every branch: Qwen2-like with biases and G = 7,
# Llama-like with llama3 scaling, Qwen3-encoder-like with q/k norm and no mask.
SMALL_QWEN2 = synth.ModelShape("s-qwen2", vocab=300, hidden=112, layers=3, n_heads=14,
                               n_kv_heads=2, head_dim=16, ff=160, rope_theta=1e6, qkv_bias=1)
SMALL_LLAMA = synth.ModelShape("s-llama", vocab=200, hidden=128, layers=2, n_heads=8,
                               n_kv_heads=2, head_dim=32, ff=256, rope_theta=5e5,
                               rope_llama3=1, rs_factor=32.0, rs_low=1.0, rs_high=4.0,
                               rs_orig_max_pos=64)
SMALL_ENC = synth.ModelShape("s-enc", vocab=180, hidden=96, layers=2, n_heads=4, n_kv_heads=2,
                             head_dim=32, ff=128, rope_theta=1e6, qk_norm=1, causal=0,
                             n_labels=16)


def _torch_weights(w):
    out = {}
    for k, a in w.items():
        if a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).double()
        else:
            t = torch.from_numpy(a).double()
        out[k] = t
    return out


def torch_forward(m, w, ids):
    """The forward written with torch library routines only (float64)."""
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

    def rope(x):   # x [T, n, D]; element i pairs with i + D/2
        z = torch.complex(x[..., : D // 2], x[..., D // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    x = F.embedding(ids, t["embed"])
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
    h = F.rms_norm(x, (H,), t["final_norm"], m.rms_eps)
    logits = F.linear(h, t["embed"])
    cls = F.linear(h, t["cls_w"], t["cls_b"]) if m.n_labels else None
    return h.numpy(), logits.numpy(), None if cls is None else cls.numpy()


@pytest.mark.parametrize("shape,T", [(synth.TINY, 8), (SMALL_QWEN2, 13), (SMALL_LLAMA, 11),
                                     (SMALL_ENC, 9)])
@pytest.mark.parametrize("wdtype", ["bf16", "f32"])
def test_forward_full_matches_torch_library_composition(shape, T, wdtype):
    w = synth.weights_bf16(shape) if wdtype == "bf16" else synth.weights_f32(shape)
    ids = synth.prompt_ids(shape, T)
    om = O.OracleModel(shape, w)
    h, lg, cls = om.forward_full(ids, logits=True, cls=bool(shape.n_labels))
    rh, rlg, rcls = torch_forward(shape, w, ids)
    assert np.allclose(h, rh, rtol=1e-10, atol=1e-11)
    assert np.allclose(lg, rlg, rtol=1e-10, atol=1e-11)
    if shape.n_labels:
        assert np.allclose(cls, rcls, rtol=1e-10, atol=1e-11)


def test_mutated_weights_are_detected():
    """The comparison above is sensitive: swapping gate and up changes the output."""
    shape = SMALL_QWEN2
    w = synth.weights_bf16(shape)
    ids = synth.prompt_ids(shape, 6)
    _, lg, _ = O.OracleModel(shape, w).forward_full(ids)
    w2 = dict(w)
    w2["layers.1.w_gate"], w2["layers.1.w_up"] = w["layers.1.w_up"], w["layers.1.w_gate"]
    _, lg2, _ = O.OracleModel(shape, w2).forward_full(ids)
    assert np.abs(lg - lg2).max() > 1e-4


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_QWEN2, SMALL_LLAMA])
def test_full_sequence_equals_prefill_plus_cached_steps(shape):
    """ember internals, bug #5: a prefill that lost the cache rows would make
    later steps disagree with the brute-force whole-sequence forward."""
    w = synth.weights_bf16(shape)
    om = O.OracleModel(shape, w)
    prompt = synth.prompt_ids(shape, 7)
    toks, glg, ghd = om.greedy(prompt, 9)
    seq = np.concatenate([prompt, toks[:-1]])
    h, lg, _ = om.forward_full(seq)
    assert np.allclose(lg[6:], glg, rtol=1e-12, atol=1e-12)
    assert np.allclose(h[6:], ghd, rtol=1e-12, atol=1e-12)
    assert all(int(np.argmax(glg[i])) == toks[i] for i in range(len(toks)))


def test_token_by_token_prefill_equals_batched_prefill():
    shape = SMALL_QWEN2
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    ids = synth.prompt_ids(shape, 10)
    c1 = om.new_cache(16)
    rc, h1, lg1 = om.forward_cached(c1, ids)
    assert rc == 0 and c1.len == 10
    c2 = om.new_cache(16)
    for i, tok in enumerate(ids):
        rc, h2, lg2 = om.forward_cached(c2, ids[i:i + 1], start_pos=i)
        assert rc == 0
    assert np.allclose(lg1, lg2, rtol=1e-12, atol=1e-13)
    k1, v1 = c1.arrays()
    k2, v2 = c2.arrays()
    assert np.allclose(k1, k2, rtol=1e-12, atol=1e-13) and np.allclose(v1, v2, rtol=1e-12,
                                                                         atol=1e-13)


def test_causality_future_tokens_do_not_change_the_past():
    shape = SMALL_LLAMA
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    ids = synth.prompt_ids(shape, 12)
    ids2 = ids.copy()
    ids2[7:] = (ids2[7:] + 1) % shape.vocab
    h1, _, _ = om.forward_full(ids, logits=False)
    h2, _, _ = om.forward_full(ids2, logits=False)
    assert np.array_equal(h1[:7], h2[:7])
    assert not np.allclose(h1[7:], h2[7:])


def test_bidirectional_sees_the_future_and_single_token_equals_causal():
    shape = SMALL_ENC
    w = synth.weights_bf16(shape)
    om = O.OracleModel(shape, w)
    ids = synth.prompt_ids(shape, 6)
    ids2 = ids.copy()
    ids2[5] = (ids2[5] + 1) % shape.vocab
    h1, _, _ = om.forward_full(ids, logits=False)
    h2, _, _ = om.forward_full(ids2, logits=False)
    assert not np.allclose(h1[0], h2[0])          # token 0 attends to token 5
    causal = synth.ModelShape(**{**shape.asdict(), "causal": 1})
    hc, _, _ = O.OracleModel(causal, w).forward_full(ids[:1], logits=False)
    hb, _, _ = om.forward_full(ids[:1], logits=False)
    assert np.array_equal(hc, hb)


def test_zero_layers_closed_form():
    """With every projection zero the residual stream is the embedding row, so
    h = RMSNorm(E[id]) and logits = E h (tied head)."""
    shape = SMALL_QWEN2
    w = synth.weights_f32(shape)
    for k in list(w):
        if k.startswith("layers.") and not k.endswith("norm"):
            w[k] = np.zeros_like(w[k])
    ids = synth.prompt_ids(shape, 5)
    h, lg, _ = O.OracleModel(shape, w).forward_full(ids)
    E = w["embed"].astype(np.float64)
    g = w["final_norm"].astype(np.float64)
    for t, i in enumerate(ids):
        e = E[i]
        hh = e / math.sqrt((e * e).mean() + shape.rms_eps) * g
        assert np.allclose(h[t], hh, rtol=1e-13, atol=1e-15)
        assert np.allclose(lg[t], E @ hh, rtol=1e-12, atol=1e-13)


def test_kv_bf16_option_rounds_the_stored_rows():
    shape = synth.TINY
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    ids = synth.prompt_ids(shape, 6)
    ca, cb = om.new_cache(8, kv_bf16=False), om.new_cache(8, kv_bf16=True)
    om.forward_cached(ca, ids)
    om.forward_cached(cb, ids)
    ka, va = ca.arrays()
    kb, vb = cb.arrays()
    # layer 0 sees identical inputs, so its rows differ only by the rounding
    ref_k = torch.from_numpy(ka[0, :, :6]).to(torch.bfloat16).double().numpy()
    ref_v = torch.from_numpy(va[0, :, :6]).to(torch.bfloat16).double().numpy()
    assert np.array_equal(kb[0, :, :6], ref_k) and np.array_equal(vb[0, :, :6], ref_v)
    assert not np.array_equal(ka[0, :, :6], kb[0, :, :6])


def test_loaded_cache_continues_exactly_like_the_original():
    """OracleCache.load: a bf16 cache exported as bit patterns and loaded into
    a fresh cache continues with the same next-token logits, bit for bit; a
    wrong row count or a corrupted row is seen (the step is conditioned on the
    loaded history, as the conditional-parity GPU tests need)."""
    shape = SMALL_QWEN2
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    ids = synth.prompt_ids(shape, 12)
    a = om.new_cache(16, kv_bf16=True)
    om.forward_cached(a, ids[:11])
    ka, va = a.arrays()
    bits = lambda x: (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kb, vb = bits(ka), bits(va)
    assert np.array_equal(O.bf16_decode(kb), ka.astype(np.float32))   # the rows are bf16 values
    b = om.new_cache(16, kv_bf16=True)
    b.load(kb, vb, 11)
    assert b.len == 11
    rc1, h1, l1 = om.forward_cached(a, ids[11:])
    rc2, h2, l2 = om.forward_cached(b, ids[11:])
    assert rc1 == rc2 == 0
    assert np.array_equal(l1, l2) and np.array_equal(h1, h2)
    # a corrupted history row changes the step
    c = om.new_cache(16, kv_bf16=True)
    kc = kb.copy()
    kc[1, 0, 3] ^= np.uint16(0x4000)
    c.load(kc, vb, 11)
    _, _, l3 = om.forward_cached(c, ids[11:])
    assert not np.allclose(l1, l3, rtol=1e-6, atol=1e-6)
    with pytest.raises(ValueError):
        c.load(kb[:, :, :5], vb[:, :, :5], 11)


def test_cache_errors_and_validation():
    shape = synth.TINY
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    c = om.new_cache(4)
    ids = synth.prompt_ids(shape, 3)
    assert om.forward_cached(c, ids, start_pos=1)[0] == -3       # position != cursor
    assert om.forward_cached(c, ids)[0] == 0
    assert om.forward_cached(c, ids)[0] == -2                    # 3 + 3 > 4
    assert om.forward_cached(c, np.array([256], np.int32))[0] == -4   # token >= vocab
    assert c.len == 3
    bad = [dict(n_kv_heads=3), dict(head_dim=15), dict(hidden=0), dict(ff=0)]
    for b in bad:
        s = synth.ModelShape(**{**shape.asdict(), **b})
        with pytest.raises(ValueError):
            O.OracleModel(s, synth.weights_bf16(synth.TINY))


def test_greedy_teacher_forcing():
    shape = SMALL_QWEN2
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    prompt = synth.prompt_ids(shape, 4)
    forced = synth.uniform_ids(99, "forced", 5, shape.vocab)
    toks, lg, _ = om.greedy(prompt, 5, forced=forced)
    _, lg_full, _ = om.forward_full(np.concatenate([prompt, forced]))
    assert np.allclose(lg, lg_full[3:], rtol=1e-12, atol=1e-13)
    assert list(toks) == [int(np.argmax(r)) for r in lg]


def test_results_identical_across_thread_counts():
    code = ("import numpy as np, sys; sys.path.insert(0, %r);"
            "from gqa_transformer_decode_gb300 import synth; from oracle import oracle as O;"
            "s = synth.TINY; om = O.OracleModel(s, synth.weights_bf16(s));"
            "t, lg, h = om.greedy(synth.prompt_ids(s, 8), 4);"
            "sys.stdout.write(lg.tobytes().hex()[:4000] + h.tobytes().hex()[-4000:])" % ROOT)
    outs = []
    for n in ("1", "3"):
        env = dict(os.environ, OMP_NUM_THREADS=n)
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=300)
        assert r.returncode == 0, r.stderr
        outs.append(r.stdout)
    assert outs[0] == outs[1]


def test_full_size_qwen_shape_prefill_and_decode_agree():
    """The full Qwen2.5-0.5B shape runs through both oracle paths."""
    shape = synth.QWEN25_05B
    om = O.OracleModel(shape, synth.weights_bf16(shape))
    prompt = synth.prompt_ids(shape, 3)
    toks, glg, _ = om.greedy(prompt, 2)
    _, lg, _ = om.forward_full(np.concatenate([prompt, toks[:-1]]))
    assert np.allclose(lg[2:], glg, rtol=1e-11, atol=1e-12)
    assert np.all(np.isfinite(glg)) and glg.shape == (3, shape.vocab)
