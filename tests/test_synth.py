"""Pins of the seeded input generator shared by the oracle and the CUDA tests
(it holds no step of the forward pass): SplitMix64 and FNV-1a against their
published outputs, the bf16 rounding against torch, and the weight / id
recipe's moments (matrices N(0, 0.02), norm weights 1 + N(0, 0.1), ids
uniform over the vocabulary)."""
import numpy as np
import torch

from gqa_transformer_decode_gb300 import synth


def test_splitmix64_first_outputs_of_seed_zero():
    """Steele, Lea and Flood's SplitMix64 from state 0: the widely published
    first three outputs."""
    w = synth._words(np.uint64(0), 0, 3)
    assert [int(v) for v in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # counter-based: any window of the stream equals the same slice of a longer draw
    k = synth._key(7, "x")
    assert np.array_equal(synth._words(k, 5, 10), synth._words(k, 0, 20)[5:15])


def test_fnv1a64_published_vectors():
    assert synth._fnv1a64("") == 0xCBF29CE484222325
    assert synth._fnv1a64("a") == 0xAF63DC4C8601EC8C
    assert synth._fnv1a64("foobar") == 0x85944171F73967E8


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 0.02,
                        rng.standard_normal(2000).astype(np.float32) * 1e3,
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, 1.00390625, 1.01171875],
                                 dtype=np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_normals_have_the_requested_moments():
    n = 1 << 20
    z = synth.normal(3, "moments", n)
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.std() - 1.0) < 5 / np.sqrt(2 * n)
    assert np.isfinite(z).all()
    # chunks are drawn in parallel: the result does not depend on the chunking
    assert np.array_equal(synth.normal(3, "moments", 1000), z[:1000])


def test_weight_recipe_and_ids():
    shape = synth.TINY
    w = synth.weights_f32(shape)
    big = np.concatenate([w["embed"].ravel(), w["layers.0.w_gate"].ravel()]).astype(np.float64)
    assert abs(big.std() - 0.02) < 0.02 * 0.02 and abs(big.mean()) < 1e-3
    norms = np.concatenate([w["final_norm"], w["layers.0.attn_norm"], w["layers.1.mlp_norm"]])
    assert abs(norms.mean() - 1.0) < 0.05 and abs(norms.std() - 0.1) < 0.03
    # bf16 weights are the RNE rounding of the f32 draws
    wb = synth.weights_bf16(shape)
    assert np.array_equal(wb["layers.0.wq"], synth.f32_to_bf16_bits(w["layers.0.wq"]))
    ids = synth.uniform_ids(5, "ids", 200000, 1000)
    assert ids.min() >= 0 and ids.max() < 1000
    counts = np.bincount(ids, minlength=1000)
    chi2 = ((counts - 200.0) ** 2 / 200.0).sum()
    assert chi2 < 1000 + 6 * np.sqrt(2 * 999)      # ~6 sigma of a chi-square with 999 dof
