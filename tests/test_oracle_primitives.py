"""Pins of the oracle's primitives against closed forms, invariants and
independent library routines (torch / numpy), never against the oracle itself.

Pages: ember scripts/reference_forward.py (rmsnorm, rope, softmax in forward,
bf16 decode in load_safetensors); LowLlamaBasic reference.py (llama3 RoPE
scaling in rotary_cos_sin); ember internals (softmax fallback, GQA mapping).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


# ---- bf16 decode / round ----------------------------------------------------

def test_bf16_decode_ieee_values():
    # IEEE-754 binary32 values whose low 16 bits are zero.
    cases = {0x3F80: 1.0, 0x4000: 2.0, 0xC040: -3.0, 0x3F00: 0.5, 0x0000: 0.0,
             0x7F80: math.inf, 0xFF80: -math.inf, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x3DCD: 0.10009765625}
    bits = np.array(list(cases), dtype=np.uint16)
    got = O.bf16_decode(bits)
    for b, g in zip(bits, got):
        assert g == np.float32(cases[int(b)]), hex(b)
    neg0 = O.bf16_decode(np.array([0x8000], dtype=np.uint16))[0]
    assert neg0 == 0 and math.copysign(1.0, neg0) < 0


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_decode(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(2000) * 1e37).astype(np.float32),
        np.array([3.3895314e38, 3.4e38, -3.4e38, 1.00390625, 1.01171875, -1.00390625],
                 dtype=np.float32),   # overflow to inf, and exact ties
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([O.bf16_round(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 is halfway between 1 (even) and 1 + 2^-7 (odd): goes to 1.
    assert O.bf16_round(1.0 + 2 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even).
    assert O.bf16_round(1.0 + 3 * 2 ** -8) == 0x3F82
    # just above the tie rounds up
    assert O.bf16_round(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81


# ---- RMSNorm -----------------------------------------------------------------

def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 64, 0.37, 1e-6
    w = np.linspace(0.5, 1.5, n).astype(np.float32)
    y = O.rmsnorm(np.full(n, c), w, eps)
    expect = c * w.astype(np.float64) / math.sqrt(c * c + eps)
    assert np.allclose(y, expect, rtol=1e-15, atol=0)


def test_rmsnorm_unit_weight_has_norm_sqrt_n():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(896) * 3.0
    y = O.rmsnorm(x, np.ones(896, np.float32), 0.0)
    assert abs(np.linalg.norm(y) - math.sqrt(896)) < 1e-12
    # no mean subtraction: a shifted input is not re-centred
    y2 = O.rmsnorm(x + 5.0, np.ones(896, np.float32), 0.0)
    assert abs(y2.mean()) > 0.5


def test_rmsnorm_matches_torch_rms_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(2048)
    w = (1 + 0.1 * rng.standard_normal(2048)).astype(np.float32)
    ref = F.rms_norm(torch.from_numpy(x), (2048,), torch.from_numpy(w).double(), eps=1e-6)
    assert np.allclose(O.rmsnorm(x, w, 1e-6), ref.numpy(), rtol=1e-13, atol=1e-14)


# ---- RoPE --------------------------------------------------------------------

def test_inv_freq_closed_form_plain():
    inv = O.rope_inv_freq(synth.QWEN25_05B)          # D = 64, theta = 1e6
    assert inv.shape == (32,)
    assert inv[0] == 1.0
    assert abs(inv[16] - 1e6 ** -0.5) < 1e-18        # i = D/4 -> theta^(-1/2)
    ratio = inv[1:] / inv[:-1]
    assert np.allclose(ratio, 1e6 ** (-2 / 64), rtol=1e-13)


def test_inv_freq_llama3_bands():
    """LowLlamaBasic rotary_cos_sin(): wavelengths below orig/high keep their
    frequency, above orig/low are divided by the factor, between them the
    scale moves smoothly (continuous at both band edges)."""
    m = synth.LLAMA32_1B
    plain = O.rope_inv_freq(synth.ModelShape("p", 1, 64, 1, 32, 8, 64, 64, rope_theta=5e5))
    scaled = O.rope_inv_freq(m)
    lam = 2 * math.pi / plain
    hi_band = lam < 8192 / 4.0
    lo_band = lam > 8192 / 1.0
    assert np.array_equal(np.nonzero(hi_band)[0], np.arange(0, 15))
    assert np.array_equal(np.nonzero(lo_band)[0], np.arange(18, 32))
    assert np.allclose(scaled[hi_band], plain[hi_band], rtol=1e-15)
    assert np.allclose(scaled[lo_band], plain[lo_band] / 32.0, rtol=1e-15)
    mid = ~(hi_band | lo_band)
    s = scaled[mid] / plain[mid]
    assert np.all((s > 1 / 32) & (s < 1)) and np.all(np.diff(s) < 0)
    # interpolation weight of the band between 2048 and 8192 tokens of wavelength
    z = (8192.0 / lam[mid] - 1.0) / 3.0
    # i = 15, 16, 17 at theta 5e5, D 64: wavelengths 2948.3, 4442.9, 6695.1 tokens,
    # worked by hand from 2*pi*5e5^(2i/64); weights z = (8192/wavelength - 1)/3.
    assert np.allclose(2 * math.pi / plain[mid], [2948.3, 4442.9, 6695.1], rtol=1e-4)
    assert np.allclose(z, [0.5928, 0.2813, 0.0745], atol=5e-4)
    assert np.allclose(s, 1 / 32 + z * (1 - 1 / 32), rtol=1e-13)


def test_rope_position_zero_is_identity_and_norm_preserved():
    rng = np.random.default_rng(3)
    inv = O.rope_inv_freq(synth.QWEN25_05B)
    v = rng.standard_normal(64)
    assert np.array_equal(O.rope_apply(v, inv, 0), v)
    for pos in (1, 17, 4095, 100000):
        r = O.rope_apply(v, inv, pos)
        assert abs(np.linalg.norm(r) - np.linalg.norm(v)) < 1e-12


def test_rope_is_complex_rotation_of_half_pairs():
    """Rotate-half pairs element i with element i + D/2: as a complex number
    z_i = v_i + j v_{i+D/2}, position p multiplies it by exp(j p f_i)."""
    rng = np.random.default_rng(4)
    inv = O.rope_inv_freq(synth.LLAMA32_1B)
    v = rng.standard_normal(64)
    for pos in (1, 5, 2047):
        r = O.rope_apply(v, inv, pos)
        z = (v[:32] + 1j * v[32:]) * np.exp(1j * pos * inv)
        assert np.allclose(r[:32], z.real, atol=1e-12)
        assert np.allclose(r[32:], z.imag, atol=1e-12)


def test_rope_composition_and_relative_position():
    rng = np.random.default_rng(5)
    inv = O.rope_inv_freq(synth.TINY)
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    a, b = 7, 12
    assert np.allclose(O.rope_apply(O.rope_apply(q, inv, a), inv, b), O.rope_apply(q, inv, a + b),
                       atol=1e-12)
    d1 = O.rope_apply(q, inv, 30) @ O.rope_apply(k, inv, 21)
    d2 = O.rope_apply(q, inv, 9) @ O.rope_apply(k, inv, 0)
    assert abs(d1 - d2) < 1e-12


def test_rope_f32_table_and_bf16_store():
    """The f32 table is cos/sin of the double angle rounded once; the f32 store
    path equals an f32 torch evaluation of the same rotation, rounded RNE."""
    m = synth.QWEN25_05B
    inv = O.rope_inv_freq(m)
    c, s = O.rope_table_f32(m, 100, 3)
    assert np.array_equal(c[1], np.cos(101 * inv).astype(np.float32))
    assert np.array_equal(s[2], np.sin(102 * inv).astype(np.float32))
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(2 * 64) * 2).astype(np.float32)
    bits = O.rope_store_bf16_f32(x, 2, 64, c[0], s[0])
    xt = torch.from_numpy(x).view(2, 2, 32)
    ct, st = torch.from_numpy(c[0]), torch.from_numpy(s[0])
    r0 = xt[:, 0] * ct - xt[:, 1] * st
    r1 = xt[:, 1] * ct + xt[:, 0] * st
    ref = torch.stack([r0, r1], 1).reshape(-1).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(bits, ref.numpy().view(np.uint16))


# ---- softmax / silu / argmax ---------------------------------------------------

def test_softmax_rows_sum_to_one_and_match_torch():
    rng = np.random.default_rng(8)
    for n in (1, 2, 7, 300):
        s = rng.standard_normal(n) * 10
        p = O.softmax(s)
        assert abs(p.sum() - 1) < 1e-12
        assert np.allclose(p, torch.softmax(torch.from_numpy(s), 0).numpy(), rtol=1e-12,
                           atol=1e-300)
        assert np.allclose(O.softmax(s + 1234.5), p, rtol=1e-9, atol=1e-300)


def test_softmax_fully_masked_row_is_uniform():
    """ember internals, edge cases: an all -inf row would give NaN; it takes
    the uniform distribution instead."""
    p = O.softmax(np.full(5, -np.inf))
    assert np.array_equal(p, np.full(5, 0.2))
    p = O.softmax(np.array([0.0, -np.inf, 1.0]))
    assert p[1] == 0.0 and abs(p.sum() - 1) < 1e-15


def test_silu_closed_forms_and_torch():
    assert O.silu(0.0) == 0.0
    for x in (0.3, 2.0, 7.5, 40.0):
        assert abs((O.silu(x) - O.silu(-x)) - x) < 1e-12     # x*sig(x) + x*sig(-x) - ... = x
    xs = np.linspace(-30, 30, 121)
    ref = F.silu(torch.from_numpy(xs)).numpy()
    assert np.allclose([O.silu(v) for v in xs], ref, rtol=1e-13, atol=1e-300)
    assert O.silu(-1000.0) == 0.0      # exp overflow gives -0, still finite


def test_argmax_first_max_and_nan():
    assert O.argmax(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert O.argmax(np.array([-np.inf, -np.inf])) == 0
    v = np.array([1.0, np.nan, 5.0, np.nan])
    assert O.argmax(v) == np.argmax(v) == 1
    rng = np.random.default_rng(9)
    for _ in range(20):
        v = rng.integers(0, 5, 1000).astype(np.float64)
        assert O.argmax(v) == int(np.argmax(v))


# ---- attention -------------------------------------------------------------------

def _sdpa(q, k, v, NH, NKV, D):
    qt = torch.from_numpy(q).view(1, NH, 1, D)
    kt = torch.from_numpy(k).view(1, NKV, -1, D)
    vt = torch.from_numpy(v).view(1, NKV, -1, D)
    return F.scaled_dot_product_attention(qt, kt, vt, enable_gqa=True).reshape(-1).numpy()


@pytest.mark.parametrize("NH,NKV,D,S", [(4, 2, 16, 9), (14, 2, 64, 33), (8, 8, 32, 5),
                                        (16, 8, 128, 17)])
def test_attention_matches_torch_sdpa_gqa(NH, NKV, D, S):
    rng = np.random.default_rng(NH * 100 + S)
    q = rng.standard_normal(NH * D)
    k = rng.standard_normal((NKV, S, D))
    v = rng.standard_normal((NKV, S, D))
    out = O.attention(q, k, v, NH, NKV, D)
    assert np.allclose(out, _sdpa(q, k, v, NH, NKV, D), rtol=1e-10, atol=1e-12)


def test_attention_gqa_equals_mha_on_repeated_heads():
    """GQA reads kv head h // (NH/NKV): identical to MHA whose kv heads are the
    GQA heads repeated with repeat_interleave (PII-Tracer forward())."""
    rng = np.random.default_rng(10)
    NH, NKV, D, S = 14, 2, 64, 20
    q = rng.standard_normal(NH * D)
    k = rng.standard_normal((NKV, S, D))
    v = rng.standard_normal((NKV, S, D))
    kr = np.repeat(k, NH // NKV, axis=0)
    vr = np.repeat(v, NH // NKV, axis=0)
    assert np.allclose(O.attention(q, k, v, NH, NKV, D), O.attention(q, kr, vr, NH, NH, D),
                       rtol=0, atol=0)
    # and a wrong mapping (h % NKV) would differ
    kw = np.tile(k, (NH // NKV, 1, 1))
    assert not np.allclose(O.attention(q, k, v, NH, NKV, D), O.attention(q, kw, vr, NH, NH, D))


def test_attention_identical_keys_average_values_and_prefix_only():
    rng = np.random.default_rng(11)
    NH, NKV, D, S = 4, 2, 16, 12
    q = rng.standard_normal(NH * D)
    k = np.broadcast_to(rng.standard_normal(D), (NKV, S, D)).copy()
    v = rng.standard_normal((NKV, S, D))
    out = O.attention(q, k, v, NH, NKV, D, n_keys=5).reshape(NH, D)
    for h in range(NH):
        assert np.allclose(out[h], v[h // 2, :5].mean(0), atol=1e-14)
