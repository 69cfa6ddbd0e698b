"""Pins of the oracle's q8_0 weight format ("ember internals" §q8_0 block
quantization) and its f16 helpers.

- f16 rounding: every result equals numpy's float16 conversion (nearest even,
  subnormals, overflow) on 200 K values over 15 decades; decoding agrees with
  numpy on all 65 536 patterns.
- Decoding follows the pages' loop: hand-built 34-byte blocks (little-endian
  f16 scale, then 32 signed int8) give q * d exactly, -128 included.
- The encoder (reading: amax / 127 in f32, stored as f16; codes rounded to
  nearest-even in f32, clamped to +-127): the largest |x| of a block maps to
  +-127; negating a block negates its codes; scaling a block by a power of two
  scales d by it and keeps the codes; a zero block is all zeros; the round
  trip error is at most d/2 plus 127 |d - f16(d)| per element.
"""
import numpy as np

from oracle import oracle as O


def test_f16_round_and_decode_match_numpy():
    rng = np.random.default_rng(0)
    xs = (rng.standard_normal(200_000).astype(np.float32)
          * np.float32(10.0) ** rng.integers(-9, 6, 200_000).astype(np.float32))
    xs = np.concatenate([xs, np.array([1e-9, 2.98e-8, 2.99e-8, 65519, 65520, -0.0, 6.1e-5], np.float32)])
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([O.f16_round(v) for v in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = np.array([O.f16_decode(int(b)) for b in bits], dtype=np.float32)
    want = bits.view(np.float16).astype(np.float32)
    same = (dec == want) | (np.isnan(dec) & np.isnan(want))
    assert same.all()


def block(d_bits, q):
    b = np.zeros(34, dtype=np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2:] = np.asarray(q, dtype=np.int8).view(np.uint8)
    return b


def test_dequant_follows_the_pages_loop():
    q = np.array([-128, -127, -1, 0, 1, 2, 127] + list(range(-12, 13)), dtype=np.int8)
    assert q.size == 32
    blocks = np.stack([block(0x3800, q), block(0x0001, q), block(0xBC00, q)])   # 0.5, 2^-24, -1
    got = O.q8_0_dequant(blocks).reshape(3, 32)
    assert np.array_equal(got[0], q.astype(np.float32) * 0.5)
    assert np.array_equal(got[1], q.astype(np.float32) * np.float32(2.0 ** -24))
    assert np.array_equal(got[2], -q.astype(np.float32))


def test_quantize_properties():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(32 * 500) * 0.02).astype(np.float32)
    x[32 * 7: 32 * 8] = 0.0                                   # a zero block
    b = O.q8_0_quantize(x)
    q = b[:, 2:].view(np.int8).astype(np.int32)
    d16 = np.array([O.f16_decode(int(v)) for v in b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8)],
                   dtype=np.float64)
    xb = x.reshape(-1, 32).astype(np.float64)
    amax = np.abs(xb).max(1)
    d32 = (amax.astype(np.float32) / np.float32(127.0)).astype(np.float64)
    nz = amax > 0
    # the largest |x| of each block codes as +-127, every code within +-127
    assert np.all(np.abs(q).max(1)[nz] == 127) and np.abs(q).max() <= 127
    assert np.all(q[~nz] == 0) and np.all(d16[~nz] == 0)
    # round trip
    err = np.abs(xb - q * d16[:, None])
    bound = 0.5 * d32 + 127 * np.abs(d32 - d16) + 1e-12
    assert np.all(err <= bound[:, None])
    # sign and power-of-two scaling
    bn = O.q8_0_quantize(-x)
    assert np.array_equal(bn[:, 2:].view(np.int8), -b[:, 2:].view(np.int8))
    assert np.array_equal(bn[:, :2], b[:, :2])
    b4 = O.q8_0_quantize(x * np.float32(4.0))
    assert np.array_equal(b4[:, 2:], b[:, 2:])
    d4 = np.array([O.f16_decode(int(v)) for v in b4[:, 0].astype(np.uint16) | (b4[:, 1].astype(np.uint16) << 8)])
    assert np.array_equal(d4[nz], 4.0 * d16[nz])
    # decoding the blocks gives q * d
    assert np.array_equal(O.q8_0_dequant(b).astype(np.float64), (q * d16[:, None]).reshape(-1))
