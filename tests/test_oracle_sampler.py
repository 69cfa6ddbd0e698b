"""Pins of the oracle's sampler ("ember internals" §sampler: temperature ->
top-k -> top-p -> softmax with the uniform fallback -> inverse CDF) against
what the page and the mathematics fix: temperature 0 is greedy; a single
survivor is drawn with certainty; known distributions are drawn at the right
boundaries; a stratified sweep of the draw reproduces the probabilities; the
filters keep ties with the threshold, follow the page's order, and reduce to
the unfiltered softmax when disabled; a fully masked row is uniform; the
probabilities are the f64 softmax of the f32 logits, summed in order."""
import numpy as np
import pytest

from oracle import sampler as S

F32 = np.float32


def log_probs(p):
    return np.log(np.asarray(p, dtype=np.float64)).astype(F32)


def test_temperature_zero_is_first_argmax_whatever_the_draw():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.standard_normal(257).astype(F32)
        x[rng.integers(0, 257)] = x.max()            # a tie at the top
        first = int(np.argmax(x))
        for r in (0.0, 0.3, 0.999):
            assert S.sample(x, 0.0, 5, 0.9, r) == first


def test_inverse_cdf_boundaries_of_a_known_distribution():
    """softmax(log p) = p: draws below 0.1 give 0, below 0.3 give 1, below 0.6
    give 2, the rest 3 (cumulative 0.1 / 0.3 / 0.6 / 1)."""
    x = log_probs([0.1, 0.2, 0.3, 0.4])
    for r, want in [(0.0, 0), (0.05, 0), (0.15, 1), (0.25, 1), (0.45, 2), (0.59, 2), (0.65, 3), (0.999, 3)]:
        assert S.sample(x, 1.0, 0, 1.0, r) == want, r


def test_temperature_divides_the_logits():
    """t * log p at temperature t gives back p; log p at temperature 1/t gives
    p^t renormalised."""
    p = np.array([0.1, 0.2, 0.3, 0.4])
    for t in (0.5, 2.0, 3.0):
        d = S.sample_distribution(t * log_probs(p), t, 0, 1.0)
        assert np.allclose(d, p, atol=2e-6)
        # temperature 1/t turns p into p^t / sum(p^t)
        assert np.allclose(S.sample_distribution(log_probs(p), 1.0 / t, 0, 1.0), p ** t / (p ** t).sum(),
                           atol=2e-6)
    # sharper / flatter: t < 1 raises the top probability, t > 1 lowers it
    x = log_probs(p)
    assert S.sample_distribution(x, 0.5, 0, 1.0)[3] > 0.4 > S.sample_distribution(x, 2.0, 0, 1.0)[3]
    assert np.allclose(S.sample_distribution(x, 0.5, 0, 1.0), p ** 2 / (p ** 2).sum(), atol=2e-6)


def test_stratified_draws_reproduce_the_probabilities():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(7).astype(F32) * 2
    p = np.exp(x.astype(np.float64) - x.max())
    p /= p.sum()
    N = 20000
    counts = np.zeros(7)
    for i in range(N):
        counts[S.sample(x, 1.0, 0, 1.0, (i + 0.5) / N)] += 1
    assert np.abs(counts / N - p).max() <= 1.0 / N + 1e-5


def test_top_k_keeps_ties_with_the_threshold():
    x = np.array([3, 1, 3, 1, 2], dtype=F32)
    d = S.sample_distribution(x, 1.0, 2, 1.0)          # threshold = 3: both 3s survive
    assert np.allclose(d, [0.5, 0, 0.5, 0, 0])
    assert S.sample(x, 1.0, 2, 1.0, 0.25) == 0 and S.sample(x, 1.0, 2, 1.0, 0.75) == 2
    d = S.sample_distribution(x, 1.0, 3, 1.0)          # threshold = 2
    assert (d > 0).tolist() == [True, False, True, False, True]


def test_top_k_one_is_the_argmax_and_k_out_of_range_is_a_no_op():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(100).astype(F32)
    for r in (0.0, 0.5, 0.99):
        assert S.sample(x, 1.0, 1, 1.0, r) == int(np.argmax(x))
    full = S.sample_distribution(x, 1.0, 0, 1.0)
    for k in (0, 100, 1000):
        assert np.array_equal(S.sample_distribution(x, 1.0, k, 1.0), full)


def test_top_p_keeps_the_shortest_prefix_that_exceeds_p():
    x = log_probs([0.5, 0.3, 0.15, 0.05])
    # 0.5 does not exceed 0.7, 0.8 does: keep {0, 1}, renormalised 0.625 / 0.375
    assert np.allclose(S.sample_distribution(x, 1.0, 0, 0.7), [0.625, 0.375, 0, 0], atol=1e-6)
    assert S.sample(x, 1.0, 0, 0.7, 0.6) == 0 and S.sample(x, 1.0, 0, 0.7, 0.65) == 1
    # exactly reaching p is not exceeding it (exact binary fractions)
    assert S.nucleus_cutoff(np.array([0.5, 0.25, 0.25], dtype=F32), 0.5) == F32(0.25)
    assert S.nucleus_cutoff(np.array([0.25, 0.5, 0.25], dtype=F32), 0.49) == F32(0.5)
    # p just below the top probability keeps the top token alone
    assert np.allclose(S.sample_distribution(x, 1.0, 0, 0.49), [1, 0, 0, 0])
    # p >= 1 and p <= 0 leave the distribution alone
    full = S.sample_distribution(x, 1.0, 0, 1.0)
    assert np.array_equal(S.sample_distribution(x, 1.0, 0, 0.0), full)
    assert np.allclose(full, [0.5, 0.3, 0.15, 0.05], atol=1e-6)


def test_top_k_then_top_p_in_the_pages_order():
    """top-k first: k = 3 keeps 0.35, 0.25, 0.15, renormalised to 0.467,
    0.333, 0.2; top-p 0.7 then keeps the first two (0.8 > 0.7): 0.583 /
    0.417.  In the other order top-p 0.7 would keep three (0.35, 0.6, 0.75)
    and top-k 3 nothing more: 0.467 / 0.333 / 0.2."""
    x = log_probs([0.35, 0.25, 0.15, 0.12, 0.08, 0.05])
    d = S.sample_distribution(x, 1.0, 3, 0.7)
    assert np.allclose(d, [0.35 / 0.6, 0.25 / 0.6, 0, 0, 0, 0], atol=1e-6)
    # ties with the k-th value survive top-k before top-p sees them
    y = log_probs([0.4, 0.2, 0.1, 0.1, 0.1, 0.1])
    assert (S.sample_distribution(y, 1.0, 3, 1.0) > 0).all()


def test_fully_masked_row_is_uniform():
    x = np.full(4, -np.inf, dtype=F32)
    d = S.softmax_f64(x)
    assert np.array_equal(d, np.full(4, 0.25))
    assert S.categorical(d, 0.0) == 0 and S.categorical(d, 0.5) == 2 and S.categorical(d, 0.999) == 3


def test_rounding_fallback_takes_the_last_maximal_index():
    d = np.array([0.25, 0.25, 0.25, 0.25], dtype=F32)
    assert S.categorical(d, 1.0) == 3           # r at the total: no running sum exceeds it
    d = np.array([0.4, 0.1, 0.4, 0.1], dtype=F32)
    assert S.categorical(d, 1.5) == 2


def test_running_sums_are_in_index_order_and_f64():
    """The page's loops add one term at a time: the sampler's running sums are
    that order, in f64 (numpy's own sum is pairwise and may differ in the last
    bit); the distribution sums to 1 within f64 rounding over a vocabulary-
    sized row, where an f32 running sum would drift by ~1e-4."""
    rng = np.random.default_rng(4)
    e = rng.random(100003)
    s = 0.0
    for v in e[:5000]:
        s = s + v
    assert np.add.accumulate(e[:5000])[-1] == s
    x = np.log(e).astype(F32)
    d = S.softmax_f64(x)
    assert d.dtype == np.float64 and abs(float(d.sum()) - 1.0) < 1e-12
    # the probabilities are the f64 softmax of the f32 logits
    ref = np.exp(x.astype(np.float64) - x.max())
    assert np.allclose(d, ref / ref.sum(), rtol=1e-13, atol=0)


def test_boundary_draws_in_f64_follow_the_exact_cdf():
    """Probabilities that are exact binary fractions: a draw exactly at a
    cumulative boundary goes to the next token (r < cum is strict), a draw one
    f32 step below it stays; the f64 sums are exact here, so no rounding
    enters the decision."""
    x = log_probs([0.25, 0.25, 0.5])
    d = S.sample_distribution(np.log(np.array([1, 1, 2], np.float64)).astype(F32), 1.0, 0, 1.0)
    assert np.allclose(d, [0.25, 0.25, 0.5], atol=1e-7)
    q = np.array([0.25, 0.25, 0.5])
    assert S.categorical(q, 0.25) == 1 and S.categorical(q, 0.5) == 2
    assert S.categorical(q, float(np.nextafter(F32(0.25), F32(0)))) == 0
    assert S.categorical(q, float(np.nextafter(F32(0.5), F32(0)))) == 1
    assert x.dtype == F32


def test_rows_use_their_own_draws():
    x = np.stack([log_probs([0.1, 0.2, 0.3, 0.4])] * 3)
    assert S.sample_rows(x, 1.0, 0, 1.0, np.array([0.05, 0.25, 0.95])).tolist() == [0, 1, 3]
