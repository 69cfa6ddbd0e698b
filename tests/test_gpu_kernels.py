"""Kernel-level parity through the C ABI: the RoPE + bf16 cache store (bit
exact against the oracle's f32 evaluation) and the tcgen05 GEMM (against a
float64 matmul of the same bf16 inputs)."""
import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu


def _p(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def stream():
    return torch.cuda.Stream()


@pytest.mark.parametrize("shape,n_heads,n_tok,pos0", [
    (synth.TINY, 2, 5, 0), (synth.QWEN25_05B, 2, 7, 120), (synth.LLAMA32_1B, 8, 4, 2040),
    (synth.QWEN3_ENC, 8, 3, 500)])
def test_rope_store_is_bit_exact(shape, n_heads, n_tok, pos0, stream):
    """ember reference_forward.py rope(): identical f32 inputs and tables give
    identical bf16 cache bits."""
    D = shape.head_dim
    rng = np.random.default_rng(D + n_tok)
    x = (rng.standard_normal((n_tok, n_heads * D)) * 1.5).astype(np.float32)
    cos_t, sin_t = O.rope_table_f32(shape, pos0, n_tok)
    expect = np.stack([O.rope_store_bf16_f32(x[t], n_heads, D, cos_t[t], sin_t[t])
                       for t in range(n_tok)])
    xd = torch.from_numpy(x).cuda()
    cd, sd = torch.from_numpy(cos_t).cuda(), torch.from_numpy(sin_t).cuda()
    out = torch.empty((n_tok, n_heads * D), dtype=torch.int16, device="cuda")
    with torch.cuda.stream(stream):
        st = E.ember_rope_store(_p(xd), n_tok, n_heads, D, _p(cd), _p(sd), _p(out),
                                _p_stream(stream))
    E.check(st, "ember_rope_store")
    stream.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, expect)


def _p_stream(s):
    import ctypes
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(rng, shape, scale=1.0):
    return synth.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (1, 64, 64), (7, 1152, 896), (130, 256, 128),
                                   (300, 896, 4864), (257, 9728, 896), (64, 2048, 2048),
                                   (2048, 3072, 2048)])
def test_gemm_bf16_matches_float64_matmul(M, N, K, stream):
    rng = np.random.default_rng(M * 7 + N + K)
    a = _bf16(rng, (M, K))
    b = _bf16(rng, (N, K), 0.05)
    ad = torch.from_numpy(a.view(np.int16)).cuda()
    bd = torch.from_numpy(b.view(np.int16)).cuda()
    d = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = E.ember_gemm_bf16(_p(ad), _p(bd), _p(d), M, N, K, _p_stream(stream))
    E.check(st, "ember_gemm_bf16")
    stream.synchronize()
    af = O.bf16_decode(a).astype(np.float64)
    bf = O.bf16_decode(b).astype(np.float64)
    ref = af @ bf.T
    got = d.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    # f32 accumulation of K exact bf16 products: error well below 1e-5 * sqrt(K) * scale
    tol = 1e-5 * np.sqrt(K) * np.abs(af).max() * np.abs(bf).max() * 4
    err = np.abs(got - ref).max()
    assert err <= tol, (err, tol)
