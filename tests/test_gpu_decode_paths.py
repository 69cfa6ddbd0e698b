"""Parity of the alternative batch-1 decode path, run in a child process so
its switch is read at model creation: the chained per-projection kernels
(EMBER_NO_FUSED=1, the path batch 2..8 takes) give the same greedy
continuation and logits as the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, %(root)r); sys.path.insert(0, %(tests)r)
from gqa_transformer_decode_gb300 import runtime as R, synth
from oracle import oracle as O
from parity_util import assert_close, assert_tokens, first_argmax
shapes = [synth.TINY,
          synth.ModelShape("s-qwen2", vocab=300, hidden=112, layers=3, n_heads=14, n_kv_heads=2,
                           head_dim=16, ff=160, rope_theta=1e6, qkv_bias=1),
          synth.ModelShape("s-llama", vocab=1000, hidden=256, layers=2, n_heads=8, n_kv_heads=2,
                           head_dim=32, ff=512, rope_theta=5e5, rope_llama3=1, rs_factor=32.0,
                           rs_low=1.0, rs_high=4.0, rs_orig_max_pos=64),
          synth.ModelShape("s-qk", vocab=400, hidden=256, layers=2, n_heads=4, n_kv_heads=2,
                           head_dim=128, ff=384, rope_theta=1e6, qk_norm=1),
          synth.ModelShape("s-d64", vocab=700, hidden=192, layers=2, n_heads=6, n_kv_heads=2,
                           head_dim=64, ff=256, rope_theta=1e6, qkv_bias=1)]
from gqa_transformer_decode_gb300 import ember as E
s = torch.cuda.Stream()
for shape in shapes:
    w = synth.weights_bf16(shape)
    om = O.OracleModel(shape, w)
    prompt = synth.prompt_ids(shape, 37)
    toks, olg, _ = om.greedy(prompt, 300 if shape.name == "s-llama" else 12)
    n = len(toks) - 1
    m = R.Model(shape, w, max_tokens=64)
    kv = m.kv_alloc(1, 37 + n + 1)
    lg = torch.empty((n + 1, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        m.prefill(kv, 0, torch.as_tensor(prompt).cuda(), 0, logits=lg[0], argmax=am[0:1], stream=s)
        seqs = torch.zeros(1, dtype=torch.int32, device="cuda")
        for i in range(1, n + 1):
            if i == n:
                s.synchronize()
                l0 = E.ember_kernel_launches()
            m.decode_step(kv, seqs, torch.tensor([toks[i - 1]], dtype=torch.int32, device="cuda"),
                          None, logits=lg[i], argmax=am[i:i + 1], stream=s)
    assert m.sync_status(s) == 0
    # which path ran: embed + 5 per layer + head + finish
    launches = E.ember_kernel_launches() - l0
    assert launches == 5 * shape.layers + 3, (shape.name, launches)
    glg, gam = lg.cpu().numpy(), am.cpu().numpy()
    assert_close(olg, glg, shape.name + " logits")
    assert_tokens(olg, toks, gam, shape.name + " tokens")
    assert all(gam[i] == first_argmax(glg[i]) for i in range(n + 1))
print("decode path ok")
"""


def test_chained_decode_path_matches_oracle():
    env = dict(os.environ, EMBER_NO_FUSED="1")
    code = CHILD % {"root": ROOT, "tests": os.path.join(ROOT, "tests")}
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "decode path ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
