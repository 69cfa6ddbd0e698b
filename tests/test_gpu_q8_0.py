"""q8_0 weights on the GPU ("ember internals" §q8_0 block quantization),
through the C ABI, against the oracle's encoder and decoder.

- The device quantizer (ember_q8_0_quantize) gives the oracle's codes and
  scales bit for bit: random blocks, ties at x / d = k + 1/2, zero and
  negative-zero blocks, scales in the f16 subnormal range and below it.
- The q8_0 GEMV (ember_gemv_q8_0) equals the f64 product of the decoded
  weights within the f32 accumulation bound (K + 16) 2^-24 sum |w x|, on
  ragged row counts.
- A weights_q8 model (prefill on the tensor-core GEMMs over the f16 copy of
  the decoded values, batch-1 and batch-3 decode on the q8_0 GEMVs, batch-12
  decode on the GEMMs) matches the oracle run on the decoded weights within
  the parity bar, and is nearer to it than to the unquantized model.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import runtime as R
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from parity_util import assert_close, assert_tokens, first_argmax, metrics

pytestmark = pytest.mark.gpu

P = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731


def bf16_bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def gpu_quantize(w_bits):
    w = torch.as_tensor(w_bits.view(np.int16)).cuda()
    n = w.numel()
    q = torch.full((n,), 99, dtype=torch.int8, device="cuda")
    d = torch.full((n // 32,), 0x7E00, dtype=torch.int16, device="cuda")
    s = torch.cuda.current_stream()
    assert E.ember_q8_0_quantize(P(w), n, P(q), P(d), C.c_void_p(s.cuda_stream)) == 0, E.last_error()
    s.synchronize()
    return q.cpu().numpy(), d.cpu().numpy().view(np.uint16)


def oracle_blocks(w_bits):
    b = O.q8_0_quantize(O.bf16_decode(w_bits))
    return b[:, 2:].reshape(-1).view(np.int8), (b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8))


def test_device_quantizer_is_bit_exact_with_the_oracle():
    rng = np.random.default_rng(20261202)
    parts = [rng.standard_normal(32 * 4000) * 0.02,                     # weight-like
             rng.standard_normal(32 * 64) * 3e4,                        # d near the top of f16
             rng.standard_normal(32 * 64) * 1e-5,                       # d in the f16 subnormals
             rng.standard_normal(32 * 64) * 1e-9,                       # d rounds to 0 in f16
             np.zeros(32 * 3)]
    tie = np.zeros(32)                                                  # amax 127 -> d = 1: x/d = k + 1/2
    tie[0] = 127.0
    tie[1:9] = [2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 126.5, -1.5]
    negz = np.full(32, -0.0)
    mixed = rng.standard_normal(32 * 64) * np.repeat(10.0 ** rng.integers(-6, 4, 64), 32)
    x = np.concatenate(parts + [tie, negz, mixed]).astype(np.float32)
    w = bf16_bits(x)
    q, d = gpu_quantize(w)
    oq, od = oracle_blocks(w)
    assert np.array_equal(d, od), np.nonzero(d != od)[0][:10]
    assert np.array_equal(q, oq), np.nonzero(q != oq)[0][:10]
    # the tie block: d = 1.0 exactly, halves to even
    tb = (x.size - 32 * 64 - 64) // 32
    assert od[tb] == 0x3C00 and list(oq[tb * 32: tb * 32 + 9]) == [127, 2, 4, -2, -4, 0, 0, 126, -2]


@pytest.mark.parametrize("N,K,nb", [(1, 32, 1), (37, 96, 3), (1000, 896, 8), (4864, 896, 1),
                                    (896, 4864, 2), (151, 4096, 5)])
def test_q8_0_gemv_equals_the_decoded_product(N, K, nb):
    rng = np.random.default_rng(N * 131 + K)
    w = bf16_bits(rng.standard_normal((N, K)) * 0.03)
    x = rng.standard_normal((nb, K)).astype(np.float32)
    q, d = gpu_quantize(w.reshape(-1))
    blocks = np.empty((q.size // 32, 34), dtype=np.uint8)
    blocks[:, 0], blocks[:, 1] = d & 0xFF, d >> 8
    blocks[:, 2:] = q.reshape(-1, 32).view(np.uint8)
    wd = O.q8_0_dequant(blocks).reshape(N, K).astype(np.float64)
    ref = x.astype(np.float64) @ wd.T
    # decoded weights are exact in f32; K products and sums, each rounded once
    bound = (K + 16) * 2.0 ** -24 * (np.abs(x).astype(np.float64) @ np.abs(wd).T) + 1e-30
    qd = torch.as_tensor(q).cuda()
    dd = torch.as_tensor(d.view(np.int16)).cuda()
    xd = torch.as_tensor(x).cuda()
    y = torch.full((nb, N), np.nan, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    assert E.ember_gemv_q8_0(P(qd), P(dd), N, K, P(xd), nb, P(y), C.c_void_p(s.cuda_stream)) == 0, E.last_error()
    s.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def test_q8_0_entry_points_validate_arguments():
    lib = E.load()
    t = torch.zeros(64, dtype=torch.int16, device="cuda")
    assert lib.ember_q8_0_quantize(P(t), 48, P(t), P(t), None) == 1       # n % 32
    assert lib.ember_q8_0_quantize(None, 32, P(t), P(t), None) == 1
    assert lib.ember_gemv_q8_0(P(t), P(t), 4, 40, P(t), 1, P(t), None) == 1   # K % 32
    assert lib.ember_gemv_q8_0(P(t), P(t), 4, 32, P(t), 9, P(t), None) == 1   # nb > 8
    torch.cuda.synchronize()


Q8_QWEN2 = synth.ModelShape("q8-qwen2", vocab=2000, hidden=448, layers=2, n_heads=7,
                            n_kv_heads=1, head_dim=64, ff=640, rope_theta=1e6, qkv_bias=1)
Q8_D128 = synth.ModelShape("q8-d128", vocab=900, hidden=256, layers=2, n_heads=4, n_kv_heads=2,
                           head_dim=128, ff=384, rope_theta=1e6, qk_norm=1)


_models = {}


def q8_models(shape):
    if shape.name not in _models:
        w = synth.weights_bf16(shape)
        _models[shape.name] = (O.OracleModel(shape, O.q8_0_layer_weights(w, shape.layers)), O.OracleModel(shape, w),
                               R.Model(shape, w, max_tokens=512, weights_q8=1))
    return _models[shape.name]


def i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("shape,n_prompt,n_steps", [(Q8_QWEN2, 150, 8), (Q8_D128, 77, 6)])
def test_q8_0_model_prefill_and_batch1_decode_match_the_oracle(shape, n_prompt, n_steps):
    oq, ob, gm = q8_models(shape)
    prompt = synth.prompt_ids(shape, n_prompt)
    toks, olg, _ = oq.greedy(prompt, n_steps)
    kv = gm.kv_alloc(1, n_prompt + n_steps + 8)
    s = torch.cuda.Stream()
    lg = torch.empty((n_steps + 1, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(n_steps + 1, dtype=torch.int32, device="cuda")
    hid = torch.empty((n_prompt, shape.hidden), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        gm.prefill(kv, 0, i32(prompt), 0, logits=lg[0], argmax=am[0:1], hidden=hid, stream=s)
        for i in range(1, n_steps + 1):
            gm.decode_step(kv, i32([0]), i32([toks[i - 1]]), i32([n_prompt + i - 1]), logits=lg[i],
                           argmax=am[i:i + 1], stream=s)
    assert gm.sync_status(s) == 0
    glg, gam = lg.cpu().numpy(), am.cpu().numpy()
    h_full, _, _ = oq.forward_full(prompt, logits=False)
    assert_close(h_full, hid.cpu().numpy(), "q8_0 prefill hidden")
    assert_close(olg, glg, "q8_0 logits")
    assert_tokens(olg, toks, gam, "q8_0 greedy tokens")
    for i in range(n_steps + 1):
        assert gam[i] == first_argmax(glg[i])
    # the quantization is really applied: the unquantized model is farther away
    _, blg, _ = ob.forward_full(np.concatenate([prompt, toks[:-1]]))
    blg = blg[n_prompt - 1:]
    assert metrics(olg, glg)["mean_abs"] < 0.5 * metrics(blg, glg)["mean_abs"]


@pytest.mark.parametrize("B", [3, 12])
def test_q8_0_model_batched_decode(B):
    """B <= 8 runs the q8_0 GEMVs, larger batches the tensor-core GEMMs over
    the f16 copy of the decoded weights."""
    shape = Q8_QWEN2
    oq, _, gm = q8_models(shape)
    lens = [4 + 5 * b for b in range(B)]
    kv = gm.kv_alloc(B, 80)
    prompts = [synth.prompt_ids(shape, L, seq=b) for b, L in enumerate(lens)]
    nxt = [synth.uniform_ids(9, f"q8next.{b}", 3, shape.vocab) for b in range(B)]
    s = torch.cuda.Stream()
    lg = torch.empty((3, B, shape.vocab), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        for b in range(B):
            gm.prefill(kv, b, i32(prompts[b]), 0, stream=s)
        for t in range(3):
            gm.decode_step(kv, i32(list(range(B))), i32([nxt[b][t] for b in range(B)]),
                           i32([lens[b] + t for b in range(B)]), logits=lg[t], stream=s)
    assert gm.sync_status(s) == 0
    glg = lg.cpu().numpy()
    for b in range(B):
        _, olg, _ = oq.forward_full(np.concatenate([prompts[b], nxt[b]]))
        assert_close(olg[lens[b]:lens[b] + 3], glg[:, b], f"q8_0 seq {b}")


def test_q8_0_config_is_validated():
    w = synth.weights_bf16(synth.TINY)          # hidden 64, ff and heads fine ...
    odd = synth.ModelShape("q8-odd", vocab=256, hidden=112, layers=1, n_heads=7, n_kv_heads=1,
                           head_dim=16, ff=160, rope_theta=1e6)
    with pytest.raises(E.EmberError) as ei:
        R.Model(odd, synth.weights_bf16(odd), max_tokens=64, weights_q8=1)
    assert ei.value.status == 8   # UNSUPPORTED: hidden 112 is not a multiple of 32
    with pytest.raises(E.EmberError) as ei:
        R.Model(synth.TINY, w, max_tokens=64, weights_q8=2)
    assert ei.value.status == 1
    big = dict(w)
    a = O.bf16_decode(big["layers.0.w_up"]).copy()
    a[3, 5] = 2.0e7                              # |w| / 127 beyond the f16 range
    big["layers.0.w_up"] = bf16_bits(a)
    with pytest.raises(E.EmberError) as ei:
        R.Model(synth.TINY, big, max_tokens=64, weights_q8=1)
    assert ei.value.status == 8
