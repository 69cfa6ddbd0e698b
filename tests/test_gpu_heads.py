"""The activation probe (ember_prefill_activations, "ember internals"
forward_with_activations) and the mean-pooled sensitivity head
(ember_mean_pooled_head, PII-Tracer-vLLM forward()) against the oracle, on
the tensor-core prefill path (head_dim 64 / 128) and the SIMT one (head_dim
16), through the C ABI.  Tolerance as for every hidden state: max-abs 2e-2
and cosine >= 0.9999 per row."""
import ctypes as C

import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import runtime as R
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from parity_util import assert_close

pytestmark = pytest.mark.gpu

PROBE_SHAPES = [
    synth.ModelShape("p-qwen2", vocab=2000, hidden=448, layers=3, n_heads=7, n_kv_heads=1,
                     head_dim=64, ff=640, rope_theta=1e6, qkv_bias=1),
    synth.ModelShape("p-llama", vocab=1500, hidden=256, layers=2, n_heads=8, n_kv_heads=2,
                     head_dim=64, ff=512, rope_theta=5e5, rope_llama3=1, rs_factor=32.0,
                     rs_low=1.0, rs_high=4.0, rs_orig_max_pos=256),
    synth.ModelShape("p-small", vocab=300, hidden=112, layers=3, n_heads=14, n_kv_heads=2,
                     head_dim=16, ff=160, rope_theta=1e6, qkv_bias=1),
]


@pytest.mark.parametrize("shape", PROBE_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("n", [1, 37, 150])
def test_probe_matches_oracle_after_every_block(shape, n):
    w = synth.weights_bf16(shape)
    om = O.OracleModel(shape, w)
    gm = R.Model(shape, w, max_tokens=256)
    prompt = synth.prompt_ids(shape, n)
    acts_ref, lg_ref = om.forward_activations(prompt)
    kv = gm.kv_alloc(1, n + 4)
    s = torch.cuda.Stream()
    acts = torch.full((shape.layers, shape.hidden), float("nan"), device="cuda")
    lg = torch.empty(shape.vocab, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        gm.prefill_activations(kv, 0, torch.as_tensor(prompt).cuda(), 0, acts, logits=lg, argmax=am,
                               stream=s)
    assert gm.sync_status(s) == 0
    assert_close(acts_ref, acts.cpu().numpy(), f"{shape.name} residual after each block")
    assert_close(lg_ref[None], lg.cpu().numpy()[None], f"{shape.name} last logits")
    # the cache advanced like a prefill: a decode step continues from position n
    with torch.cuda.stream(s):
        gm.decode_step(kv, torch.zeros(1, dtype=torch.int32, device="cuda"), am, None, argmax=am,
                       stream=s)
    assert gm.sync_status(s) == 0


def test_probe_rejects_null_acts():
    lib = E.load()
    assert lib.ember_prefill_activations(None, None, 0, None, 1, 0, None, None, None, None) == 1


ENC = synth.ModelShape("h-enc", vocab=600, hidden=256, layers=2, n_heads=4, n_kv_heads=2,
                       head_dim=128, ff=384, rope_theta=1e6, qk_norm=1, causal=0, n_labels=16)


@pytest.mark.parametrize("B,T,n_out", [(1, 5, 1), (3, 40, 1), (2, 130, 3)])
def test_mean_pooled_head_matches_oracle(B, T, n_out):
    w = synth.weights_bf16(ENC)
    om = O.OracleModel(ENC, w)
    gm = R.Model(ENC, w, max_tokens=512, max_positions=256)
    hw = synth.f32_to_bf16_bits(synth.normal(20261202, "sensitivity_head.weight", n_out * ENC.hidden,
                                             std=0.02).astype(np.float32)).reshape(n_out, ENC.hidden)
    hb = synth.f32_to_bf16_bits(synth.normal(20261202, "sensitivity_head.bias", n_out,
                                             std=0.02).astype(np.float32))
    ids = np.stack([synth.prompt_ids(ENC, T, seq=b) for b in range(B)])
    s = torch.cuda.Stream()
    hid = torch.empty((B * T, ENC.hidden), device="cuda")
    out = torch.empty((B, n_out), device="cuda")
    W = torch.from_numpy(hw.view(np.int16).copy()).cuda()
    Bi = torch.from_numpy(hb.view(np.int16).copy()).cuda()
    P = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
    with torch.cuda.stream(s):
        gm.encode(torch.as_tensor(ids.reshape(-1)).cuda(), B, T, hidden=hid, stream=s)
        assert E.ember_mean_pooled_head(P(hid), B, T, ENC.hidden, P(W), P(Bi), n_out, P(out),
                                        C.c_void_p(s.cuda_stream)) == 0
    assert gm.sync_status(s) == 0
    got = out.cpu().numpy()
    Wf, bf = O.bf16_decode(hw), O.bf16_decode(hb)
    for b in range(B):
        h, _, _ = om.forward_full(ids[b], logits=False)
        ref = O.mean_pooled_head(h, Wf, bf)
        # every element of the mean within the hidden-state tolerance (2e-2)
        # bounds output j by 2e-2 * ||w_j||_1
        tol = 2e-2 * np.abs(Wf.astype(np.float64)).sum(1)
        assert np.all(np.abs(ref - got[b]) <= tol), (b, ref, got[b], tol)
        assert_close(h, hid.cpu().numpy()[b * T:(b + 1) * T], f"encoder hidden seq {b}")
    # no bias
    with torch.cuda.stream(s):
        assert E.ember_mean_pooled_head(P(hid), B, T, ENC.hidden, P(W), None, n_out, P(out),
                                        C.c_void_p(s.cuda_stream)) == 0
    s.synchronize()
    assert np.allclose(out.cpu().numpy(), got - bf[None], atol=1e-5)
