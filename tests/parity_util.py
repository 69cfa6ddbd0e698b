"""Comparison metrics of the parity tests.

The metrics follow PII-Tracer-vLLM serving/reference_forward.py main(): max
and mean absolute delta, minimum per-row cosine and argmax agreement.  The
bar: every position's hidden state and logits within
max-abs 2e-2 and cosine >= 0.9999; greedy tokens identical wherever the
oracle's top-2 logit gap exceeds 1e-2.
"""
import numpy as np

MAX_ABS = 2e-2
MIN_COS = 0.9999
GAP = 1e-2


def metrics(ref, got):
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, np.asarray(ref).shape[-1])
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    d = np.abs(ref - got)
    num = (ref * got).sum(-1)
    den = np.linalg.norm(ref, axis=-1) * np.linalg.norm(got, axis=-1)
    cos = num / np.maximum(den, 1e-300)
    return {"max_abs": float(d.max()), "mean_abs": float(d.mean()), "min_cos": float(cos.min())}


def assert_close(ref, got, what, max_abs=MAX_ABS, min_cos=MIN_COS):
    m = metrics(ref, got)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert m["max_abs"] <= max_abs and m["min_cos"] >= min_cos, f"{what}: {m}"
    return m


def top2_gap(logits_row):
    s = np.sort(np.asarray(logits_row, dtype=np.float64))
    return s[-1] - s[-2]


def assert_tokens(ref_logits, ref_tokens, got_tokens, what):
    """Tokens must agree wherever the oracle's top-2 gap exceeds GAP."""
    checked = 0
    for i, (r, g) in enumerate(zip(ref_tokens, got_tokens)):
        if top2_gap(ref_logits[i]) > GAP:
            checked += 1
            assert int(r) == int(g), f"{what}: step {i} oracle {r} gpu {g}"
    return checked


def first_argmax(v):
    """np.argmax: first index of the maximum (NaN counts as the maximum)."""
    return int(np.argmax(np.asarray(v)))


def oracle_step_on_gpu_cache(om, kv, seq, length, token, max_len=None):
    """One oracle cached step of `token` at position `length`, starting from
    rows [0, length) of the GPU's bf16 cache of sequence `seq` (decoded
    exactly): conditional parity of a decode step at any context length.
    Returns (final-normed hidden [H], logits [V], oracle K / V rows at
    position `length` [L, NKV, D])."""
    K, V = kv.tensors()
    kb = K[seq][:, :, :length].cpu().numpy()
    vb = V[seq][:, :, :length].cpu().numpy()
    oc = om.new_cache(max_len or length + 1, kv_bf16=True)
    oc.load(kb, vb, length)
    rc, hid, lg = om.forward_cached(oc, np.array([token], np.int32))
    assert rc == 0, rc
    ok, ov = oc.arrays()
    return hid[0], lg, ok[:, :, length].copy(), ov[:, :, length].copy()
