"""The token sampler kernel (ember_sample, through the C ABI) against the
oracle's sampler ("ember internals" §sampler: temperature -> top-k -> top-p
-> softmax -> inverse CDF) on seeded logits and draws.

Both sides take every selection by exact comparisons of the same f32 values
(the IEEE division of stage 1 and the top-k threshold are bit-identical on
both).  The two decisions that read sums -- which descending prefix first
holds more than p of the mass, and which running sum first exceeds the draw
r -- are taken in f64 by the oracle and by the kernel from f32 exponentials
(<= 2 ulp each) quantised to 2^-40 and summed exactly, so the kernel's
normalised running sums lie within EPS = 3e-7 of the oracle's.  A row whose
oracle sum lies that close to p or to r is ambiguous: there the kernel's
token must still be one whose CDF interval reaches within EPS of r (or, for
p, a valid index); every other row must give the oracle's token."""
import ctypes as C

import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import ember as E
from oracle import sampler as S

pytestmark = pytest.mark.gpu

EPS = 3e-7


def gpu_sample(logits, t, k, p, r, stream=None):
    L = torch.as_tensor(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    R = torch.as_tensor(np.asarray(r, dtype=np.float32)).cuda()
    out = torch.full((L.shape[0],), -7, dtype=torch.int32, device="cuda")
    s = stream or torch.cuda.current_stream()
    P = lambda x: C.c_void_p(x.data_ptr())  # noqa: E731
    st = E.ember_sample(P(L), L.shape[0], L.shape[1], L.shape[1], float(t), int(k), float(p), P(R),
                        P(out), C.c_void_p(s.cuda_stream))
    assert st == 0, E.last_error()
    s.synchronize()
    return out.cpu().numpy()


def nucleus_margin(x, t, k, p):
    """Distance (f64) of the oracle's nucleus sums from p around its cutoff."""
    if not (0.0 < np.float32(p) < 1.0):
        return np.inf
    y = S.top_k_mask(S.temperature_scale(x, t), k)
    ordered = np.sort(S.softmax_f64(y))[::-1]
    cum = np.add.accumulate(ordered)
    pp = np.float64(np.float32(p))
    j = np.nonzero(cum > pp)[0]
    j = j[0] if j.size else len(cum) - 1
    return min(abs(cum[i] - pp) for i in range(max(0, j - 1), j + 1))


def check(logits, t, k, p, r, label):
    got = gpu_sample(logits, t, k, p, r)
    want = S.sample_rows(logits, t, k, p, r)
    amb = 0
    for b in range(len(r)):
        assert 0 <= got[b] < logits.shape[1], (label, b, got[b])
        if np.float32(t) <= 0 or got[b] == want[b]:
            assert got[b] == want[b], (label, b)
            continue
        # the tokens differ: legitimate only at a boundary within EPS
        if nucleus_margin(logits[b], t, k, p) < EPS:
            amb += 1
            continue
        dist = S.sample_distribution(logits[b], t, k, p)
        cum = np.add.accumulate(dist)
        lo = cum[got[b] - 1] if got[b] > 0 else 0.0
        rr = np.float64(np.float32(r[b]))
        near = dist[got[b]] > 0 and lo - EPS <= rr < cum[got[b]] + EPS
        assert near, f"{label} row {b}: gpu {got[b]} oracle {want[b]} (t={t} k={k} p={p} r={r[b]})"
        amb += 1
    assert amb <= max(1, len(r) // 4), f"{label}: {amb} of {len(r)} rows at a boundary"
    return got


V_QWEN = 151936


@pytest.mark.parametrize("t,k,p", [
    (1.0, 0, 1.0),      # plain softmax sampling
    (0.7, 0, 1.0),      # sharpened
    (1.3, 40, 1.0),     # top-k
    (1.0, 0, 0.9),      # nucleus over the whole vocabulary
    (0.8, 50, 0.95),    # both filters
    (1.0, 1, 1.0),      # top-1: the argmax, whatever the draw
    (1.0, V_QWEN, 0.5),  # k >= V is a no-op
])
def test_sampler_matches_oracle_on_the_vocabulary_of_the_decode_shape(t, k, p):
    rng = np.random.default_rng(20261202)
    B = 6
    logits = (rng.standard_normal((B, V_QWEN)) * 2.5).astype(np.float32)
    r = rng.random(B).astype(np.float32)
    check(logits, t, k, p, r, "vocab")


def test_sampler_ties_masks_and_edges():
    rng = np.random.default_rng(7)
    V = 3000
    # few distinct values: top-k thresholds fall on ties, which survive
    lg = np.round(rng.standard_normal((5, V)) * 2.0).astype(np.float32)
    r = rng.random(5).astype(np.float32)
    for t, k, p in ((1.0, 10, 1.0), (1.0, 700, 0.6), (0.5, 2, 0.99), (2.0, 0, 0.3)):
        check(lg, t, k, p, r, f"ties t={t} k={k} p={p}")
    # one dominant logit: every draw takes it
    peak = rng.standard_normal((3, V)).astype(np.float32)
    peak[:, 1234] = 80.0
    assert list(check(peak, 1.0, 0, 0.9, rng.random(3).astype(np.float32), "peak")) == [1234] * 3
    # every logit -inf: the softmax falls back to uniform, token floor(r * V)
    inf = np.full((3, V), -np.inf, dtype=np.float32)
    rr = np.array([0.0, 0.3337, 0.9999], dtype=np.float32)
    got = check(inf, 1.0, 0, 1.0, rr, "uniform fallback")
    assert list(got) == [int(np.floor(np.float64(x) * V)) for x in rr]
    # masked entries (-inf) are never drawn
    part = rng.standard_normal((4, V)).astype(np.float32)
    part[:, ::2] = -np.inf
    got = check(part, 1.0, 0, 1.0, rng.random(4).astype(np.float32), "masked")
    assert all(g % 2 == 1 for g in got)


def test_greedy_temperature_is_the_first_maximal_index():
    rng = np.random.default_rng(3)
    V = 5003
    lg = rng.standard_normal((4, V)).astype(np.float32)
    lg[1, [17, 4000]] = 9.0          # a tie: the first index wins
    lg[2, 77] = np.nan               # NaN counts as maximal (numpy argmax)
    lg[3, :] = -1.0                  # all equal: index 0
    for t in (0.0, -1.0):
        got = gpu_sample(lg, t, 0, 1.0, np.zeros(4, np.float32))
        assert list(got) == [int(np.argmax(lg[b])) for b in range(4)]
    assert list(got)[1:] == [17, 77, 0]


def test_sampler_is_deterministic_and_validates_arguments():
    rng = np.random.default_rng(11)
    lg = (rng.standard_normal((8, 20000)) * 3).astype(np.float32)
    r = rng.random(8).astype(np.float32)
    a = gpu_sample(lg, 0.9, 100, 0.8, r)
    b = gpu_sample(lg, 0.9, 100, 0.8, r)
    assert np.array_equal(a, b)
    P = C.c_void_p
    x = torch.zeros(4, 16, device="cuda")
    o = torch.zeros(4, dtype=torch.int32, device="cuda")
    lib = E.load()
    assert lib.ember_sample(None, 4, 16, 16, 1.0, 0, 1.0, None, P(o.data_ptr()), None) == 1
    assert lib.ember_sample(P(x.data_ptr()), 4, 16, 8, 1.0, 0, 1.0, P(x.data_ptr()), P(o.data_ptr()), None) == 1
    assert lib.ember_sample(P(x.data_ptr()), 4, 16, 16, 1.0, -1, 1.0, P(x.data_ptr()), P(o.data_ptr()), None) == 1
    # r may be NULL only when greedy
    assert lib.ember_sample(P(x.data_ptr()), 4, 16, 16, 1.0, 0, 1.0, None, P(o.data_ptr()), None) == 1
    assert lib.ember_sample(P(x.data_ptr()), 4, 16, 16, 0.0, 0, 1.0, None, P(o.data_ptr()), None) == 0
    torch.cuda.synchronize()


def test_greedy_sampler_on_decode_logits_equals_the_fused_argmax():
    """t = 0 through ember_sample on the logits of decode steps equals the
    argmax the LM head's fused epilogue writes in the same steps."""
    from gqa_transformer_decode_gb300 import runtime as R
    from gqa_transformer_decode_gb300 import synth
    shape = synth.ModelShape("s-samp", vocab=4000, hidden=256, layers=2, n_heads=8, n_kv_heads=2,
                             head_dim=64, ff=512, rope_theta=1e6, qkv_bias=1)
    m = R.Model(shape, synth.weights_bf16(shape), max_tokens=64)
    kv = m.kv_alloc(1, 64)
    s = torch.cuda.Stream()
    steps = 6
    lg = torch.empty((steps, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(steps, dtype=torch.int32, device="cuda")
    cur = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = torch.zeros(1, dtype=torch.int32, device="cuda")
    prompt = torch.as_tensor(synth.prompt_ids(shape, 20)).cuda()
    with torch.cuda.stream(s):
        m.prefill(kv, 0, prompt, 0, argmax=cur, stream=s)
        for i in range(steps):
            m.decode_step(kv, seqs, cur, None, logits=lg[i], argmax=am[i:i + 1], stream=s)
            cur.copy_(am[i:i + 1])
    assert m.sync_status(s) == 0
    got = gpu_sample(lg.cpu().numpy(), 0.0, 0, 1.0, np.zeros(steps, np.float32))
    assert np.array_equal(got, am.cpu().numpy())
