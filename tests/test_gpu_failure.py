"""Failure detection on the device without a GPU fault: a bounded wait that
runs out returns an error status the host reads, and the context stays
usable.  ember_test_bounded_wait runs the library's two wait helpers (the
TMA / tensor-core kernels' mbarrier wait and the fused decode's cluster-scope
wait) on an mbarrier that nothing completes, with a budget of ~0.1 ms."""
import ctypes as C

import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import runtime as R
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from parity_util import assert_tokens

pytestmark = pytest.mark.gpu

TIMEOUT = 5


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_times_out_into_the_status_word(which):
    shape = synth.TINY
    w = synth.weights_bf16(shape)
    m = R.Model(shape, w, max_tokens=64)
    s = torch.cuda.Stream()
    sp = C.c_void_p(s.cuda_stream)
    assert m.sync_status(s) == 0
    assert E.load().ember_test_bounded_wait(m.handle, which, 200000, sp) == 0
    assert m.sync_status(s) == TIMEOUT          # the wait gave up and said so
    assert m.sync_status(s) == 0                # read and cleared
    # the context is intact: a prefill and greedy steps still match the oracle
    prompt = synth.prompt_ids(shape, 8)
    toks, olg, _ = O.OracleModel(shape, w).greedy(prompt, 4)
    kv = m.kv_alloc(1, 16)
    am = torch.zeros(5, dtype=torch.int32, device="cuda")
    cur = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = torch.zeros(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        m.prefill(kv, 0, torch.as_tensor(prompt).cuda(), 0, argmax=cur, stream=s)
        am[0:1].copy_(cur)
        for i in range(1, 5):
            m.decode_step(kv, seqs, cur, None, argmax=cur, stream=s)
            am[i:i + 1].copy_(cur)
    assert m.sync_status(s) == 0
    assert_tokens(olg, toks, am.cpu().numpy(), "greedy after a timeout")


def test_bounded_wait_argument_checks():
    lib = E.load()
    assert lib.ember_test_bounded_wait(None, 0, 1000, None) == 1
