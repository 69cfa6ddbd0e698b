"""The f16 tensor-core operands against bf16 checkpoints.

1. Weights beyond the f16 range (|w| > 65504): the layer matrix is stored as
   f16(W * 2^-e) and every product with it multiplied by 2^e, an exact
   rescaling.  Weights of 1e5 and -2e5 (with the norm weights of their
   columns small enough that the activations stay in range) must give the
   oracle's results on the prefill (tensor-core GEMMs), the fused batch-1
   decode and the batched decode (split GEMV).
2. Activations beyond the f16 range: a layer whose SwiGLU output exceeds
   65504 where it is rounded to f16 for the down projection (the prefill
   GEMM path) raises EMBER_ERR_RANGE, which ember_sync_status returns."""
import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import runtime as R
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from parity_util import assert_close, assert_tokens

pytestmark = pytest.mark.gpu

SHAPE = synth.ModelShape("r-qwen2", vocab=2000, hidden=448, layers=2, n_heads=7, n_kv_heads=1,
                         head_dim=64, ff=640, rope_theta=1e6, qkv_bias=1)
RANGE = 9


def bf16(x):
    return synth.f32_to_bf16_bits(np.float32(x)).reshape(())


def large_weight_model():
    """Entries of 1e5 .. 2e5 in four layer matrices, each meeting an input
    that the model keeps small (a norm weight or a projection row scaled
    down), so that every product stays O(1-10) and the f16 activations in
    range: the test is about the weights' storage, not the activations."""
    w = {k: v.copy() for k, v in synth.weights_bf16(SHAPE).items()}
    dec = O.bf16_decode
    # up_proj row 3, column 11: 1e5 against an input column normed by 1e-4
    w["layers.0.w_up"][3, 11] = bf16(1e5)
    w["layers.0.mlp_norm"][11] = bf16(1e-4)
    # q_proj row 5, column 20: -2e5 against an input column normed by 2e-5
    w["layers.1.wq"][5, 20] = bf16(-2e5)
    w["layers.1.attn_norm"][20] = bf16(2e-5)
    # down_proj column 7 of 7e4 against feature 7, whose up row is scaled by 1e-3
    w["layers.1.w_down"][100, 7] = bf16(7e4)
    w["layers.1.w_up"][7] = synth.f32_to_bf16_bits(dec(w["layers.1.w_up"][7]) * np.float32(1e-3))
    # o_proj column 30 of -7e4 against value dim 30 (kv head 0), its v row scaled by 1e-4
    w["layers.0.wo"][9, 30] = bf16(-7e4)
    w["layers.0.wv"][30] = synth.f32_to_bf16_bits(dec(w["layers.0.wv"][30]) * np.float32(1e-4))
    assert max(np.abs(dec(w[k])).max() for k in w if k.startswith("layers.")) > 65504
    return w


def test_weights_beyond_the_f16_range_match_the_oracle():
    w = large_weight_model()
    om = O.OracleModel(SHAPE, w)
    gm = R.Model(SHAPE, w, max_tokens=256)
    s = torch.cuda.Stream()
    n = 150
    prompt = synth.prompt_ids(SHAPE, n)
    toks, olg, _ = om.greedy(prompt, 4, kv_bf16=True)
    h_full, _, _ = om.forward_full(prompt, logits=False)
    kv = gm.kv_alloc(3, n + 8)
    lg = torch.empty((5, SHAPE.vocab), device="cuda")
    hid = torch.empty((n, SHAPE.hidden), device="cuda")
    am = torch.empty(5, dtype=torch.int32, device="cuda")
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = torch.zeros(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        gm.prefill(kv, 0, torch.as_tensor(prompt).cuda(), 0, logits=lg[0], argmax=am[0:1], hidden=hid,
                   stream=s)
        for i in range(4):      # fused batch-1 decode, the oracle's tokens fed
            ids.copy_(torch.tensor([int(toks[i])], dtype=torch.int32))
            gm.decode_step(kv, seqs, ids, None, logits=lg[i + 1], argmax=am[i + 1:i + 2], stream=s)
    assert gm.sync_status(s) == 0
    assert_close(h_full, hid.cpu().numpy(), "prefill hidden, large weights")
    assert_close(olg, lg.cpu().numpy(), "logits, large weights")
    assert_tokens(olg, toks, am.cpu().numpy(), "tokens, large weights")
    # batched decode (split GEMV) over three copies of the sequence
    for b in (1, 2):
        with torch.cuda.stream(s):
            gm.prefill(kv, b, torch.as_tensor(prompt).cuda(), 0, stream=s)
    blg = torch.empty((3, SHAPE.vocab), device="cuda")
    with torch.cuda.stream(s):
        kv.set_cursor(0, n, stream=s)
        gm.decode_step(kv, torch.arange(3, dtype=torch.int32, device="cuda"),
                       torch.full((3,), int(toks[0]), dtype=torch.int32, device="cuda"), None,
                       logits=blg, stream=s)
    assert gm.sync_status(s) == 0
    for b in range(3):
        assert_close(olg[1][None], blg[b].cpu().numpy()[None], f"batched step, sequence {b}")


def test_activation_beyond_the_f16_range_raises_a_status():
    w = {k: v.copy() for k, v in synth.weights_bf16(SHAPE).items()}
    # normed inputs of ~5000 into gate/up: SwiGLU outputs far above 65504
    w["layers.0.mlp_norm"][:] = bf16(5000.0)
    gm = R.Model(SHAPE, w, max_tokens=256)
    s = torch.cuda.Stream()
    kv = gm.kv_alloc(1, 160)
    with torch.cuda.stream(s):
        gm.prefill(kv, 0, torch.as_tensor(synth.prompt_ids(SHAPE, 150)).cuda(), 0, stream=s)
    assert gm.sync_status(s) == RANGE
    assert gm.sync_status(s) == 0
