"""Token sampler of the oracle (numpy), following "ember internals" §sampler:
temperature -> top-k -> top-p (nucleus) -> softmax (uniform fallback for a
fully masked row) -> categorical sample by inverse CDF.

TEST INFRASTRUCTURE ONLY: tests/ are the only callers; nothing here imports
the CUDA library.  The uniform draw `r` in [0, 1) is an input (the page draws
it from its seeded generator); so are temperature t, k and p.

Precision.  The page's code works in f32 (Rust `f32` logits, `exp`, running
sums).  The temperature division (stage 1) and the top-k threshold (stage 2)
act on the f32 logits, as there: both are exact selections or IEEE-rounded
divisions that any implementation reproduces bit for bit.  The probabilities,
their sums and the comparisons against p and r (stages 3-5) are held in f64,
the reading this oracle takes for the whole forward pass: a sequential f32
running sum over a 150 K-entry vocabulary cannot be reproduced by a parallel
implementation, and any other f32 order moves draws near a CDF boundary to a
neighbouring token, whereas in f64 the order of summation changes the sums by
~1e-16 relative, so two implementations take the same integer decision unless
a draw falls within ~1e-12 of a boundary.  Running sums are still taken in
index order (stage 5) and in descending-probability order (stage 3), one
term at a time, as the page's loops do.

Readings (the page is a translation and leaves these open):
- temperature <= 0 is greedy: the page skips the scaling and takes the
  argmax; the argmax is the first maximal index, as in the rest of the path.
- top-k acts for 0 < k < V: the threshold is the k-th largest value after
  sorting in descending order, and only values strictly below it are
  masked, so ties with it survive (the page's `*l < threshold`).
- top-p acts for 0 < p < 1: a temporary softmax, sorted in descending order
  and summed until the running sum first exceeds p (strictly); the cutoff is
  the probability of the token that made it exceed (the smallest probability
  in the kept set), and probabilities strictly below it are masked.  When
  rounding keeps the sum from ever exceeding p, every token is kept.
- the rounding fallback of the inverse CDF returns the last maximal index of
  the distribution (the page's `max_by`, which keeps the last of equal
  maxima).
- t, p and r are f32 values (the page's types), widened exactly to f64
  where they meet the f64 probabilities.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64


def temperature_scale(logits: np.ndarray, t: float) -> np.ndarray:
    """Stage 1: divide every logit by t when t > 0 (IEEE f32 division)."""
    x = np.asarray(logits, dtype=F32).copy()
    if F32(t) > 0.0:
        x = (x / F32(t)).astype(F32)
    return x


def top_k_mask(logits: np.ndarray, k: int) -> np.ndarray:
    """Stage 2: mask every logit below the k-th largest (no-op for k <= 0 or k >= V)."""
    x = np.asarray(logits, dtype=F32).copy()
    V = x.shape[0]
    if k <= 0 or k >= V:
        return x
    ordered = np.sort(x)[::-1]          # descending values
    threshold = ordered[k - 1]
    x[x < threshold] = -np.inf
    return x


def softmax_f64(logits: np.ndarray) -> np.ndarray:
    """Stage 4: max-subtracted exponentials (f64) over their sum (f64, in
    index order); a row whose maximum is -inf becomes uniform."""
    x = np.asarray(logits, dtype=F32).astype(F64)
    V = x.shape[0]
    m = x.max()
    if m == -np.inf:
        return np.full(V, 1.0 / V, dtype=F64)
    e = np.exp(x - m)
    s = np.add.accumulate(e)[-1]          # in index order
    return e / s


def nucleus_cutoff(probs: np.ndarray, p: float) -> float:
    """The smallest probability of the shortest descending prefix whose running
    sum exceeds p (all tokens when rounding never lets it exceed)."""
    ordered = np.sort(np.asarray(probs, dtype=F64))[::-1]
    cum = np.add.accumulate(ordered)       # in descending order
    over = np.nonzero(cum > F64(F32(p)))[0]
    return ordered[over[0]] if over.size else ordered[-1]


def top_p_mask(logits: np.ndarray, p: float) -> np.ndarray:
    """Stage 3: mask the logits whose temporary softmax probability lies below
    the nucleus cutoff (no-op unless 0 < p < 1)."""
    x = np.asarray(logits, dtype=F32).copy()
    if not (0.0 < F32(p) < 1.0):
        return x
    soft = softmax_f64(x)
    cutoff = nucleus_cutoff(soft, p)
    x[soft < cutoff] = -np.inf
    return x


def categorical(dist: np.ndarray, r: float) -> int:
    """Stage 5: the first index whose running sum exceeds r; when rounding
    leaves r above the total, the last maximal index."""
    d = np.asarray(dist, dtype=F64)
    cum = np.add.accumulate(d)             # in index order
    hit = np.nonzero(F64(F32(r)) < cum)[0]
    if hit.size:
        return int(hit[0])
    return int(d.shape[0] - 1 - np.argmax(d[::-1]))


def sample_distribution(logits: np.ndarray, t: float, k: int, p: float) -> np.ndarray:
    """The distribution the categorical draw reads: stages 1-4."""
    x = temperature_scale(logits, t)
    x = top_k_mask(x, k)
    x = top_p_mask(x, p)
    return softmax_f64(x)


def sample(logits: np.ndarray, t: float, k: int, p: float, r: float) -> int:
    """One token from one row of logits; t <= 0 is greedy."""
    x = np.asarray(logits, dtype=F32)
    if F32(t) <= 0.0:
        return int(np.argmax(x))
    return categorical(sample_distribution(x, t, k, p), r)


def sample_rows(logits: np.ndarray, t: float, k: int, p: float, r: np.ndarray) -> np.ndarray:
    """sample() for each row of [B, V] logits with its own draw r[b]."""
    L = np.asarray(logits, dtype=F32)
    return np.array([sample(L[b], t, k, p, float(r[b])) for b in range(L.shape[0])], dtype=np.int64)
