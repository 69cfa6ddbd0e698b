"""Parity at the full model sizes of the benchmark workloads, in the launch
configuration bench.py times (CUDA graphs; the fused batch-1 decode; the
batched tensor-core path): against the f64 oracle where it finishes in
seconds, on sampled outputs where the whole run would not, and through
properties that hold at any size (a prefix's rows do not depend on later
tokens; a batched step equals the batch-1 step of the same cache; a prompt
split into chunks equals the prompt in one piece).  The method keeps its KV
cache in bf16, so the oracle rounds K and V to bf16 (RNE) at write time."""
import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import runtime as R
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from parity_util import assert_close, assert_tokens, first_argmax, oracle_step_on_gpu_cache

pytestmark = pytest.mark.gpu

_weights = {}


def weights(name):
    if name not in _weights:
        _weights[name] = synth.weights_bf16(synth.WORKLOADS[name].model)
    return _weights[name]


def i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


@pytest.fixture(scope="module")
def stream():
    return torch.cuda.Stream()


def greedy_gpu(model, kv, prompt, forced, stream, seq=0):
    """Prefill, then one decode step per forced token through the graph path
    (positions from the device cursor, ids from one fixed buffer)."""
    n = len(forced)
    lg = torch.empty((n + 1, model.V), dtype=torch.float32, device="cuda")
    am = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    hid = torch.empty((len(prompt), model.H), dtype=torch.float32, device="cuda")
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = i32([seq])
    with torch.cuda.stream(stream):
        kv.set_cursor(seq, 0, stream=stream)
        model.prefill(kv, seq, i32(prompt), 0, logits=lg[0], argmax=am[0:1], hidden=hid,
                      stream=stream)
        for i in range(n):
            ids.copy_(i32([forced[i]]), non_blocking=True)
            model.decode_step(kv, seqs, ids, None, logits=lg[i + 1], argmax=am[i + 1:i + 2],
                              stream=stream)
    assert model.sync_status(stream) == 0
    return lg.cpu().numpy(), am.cpu().numpy(), hid.cpu().numpy()


def test_qwen25_05b_prefill_and_decode(stream):
    """Qwen2.5-0.5B shape, batch 1: the benchmark's 128-token prompt and 32
    greedy steps (fused decode path) against the oracle."""
    name = "qwen2.5-0.5b"
    shape = synth.WORKLOADS[name].model
    w = weights(name)
    prompt = synth.prompt_ids(shape, 128)
    toks, olg, _ = O.OracleModel(shape, w).greedy(prompt, 32, kv_bf16=True)
    m = R.Model(shape, w, max_tokens=128)
    kv = m.kv_alloc(1, 128 + 40)
    glg, gam, _ = greedy_gpu(m, kv, prompt, toks[:-1], stream)
    assert_close(olg, glg, "logits")
    assert_tokens(olg, toks, gam, "greedy tokens")
    assert all(gam[i] == first_argmax(glg[i]) for i in range(len(gam)))


def test_qwen25_05b_q8_0_weights(stream):
    """Qwen2.5-0.5B shape with q8_0 layer weights (the bench's q8_0 line):
    the 128-token prompt (tensor-core GEMMs on the f16 copy of the decoded
    values) and 16 greedy steps (q8_0 GEMVs) against the oracle run on the
    decoded weights."""
    name = "qwen2.5-0.5b"
    shape = synth.WORKLOADS[name].model
    w = weights(name)
    prompt = synth.prompt_ids(shape, 128)
    om = O.OracleModel(shape, O.q8_0_layer_weights(w, shape.layers))
    toks, olg, _ = om.greedy(prompt, 16, kv_bf16=True)
    m = R.Model(shape, w, max_tokens=128, weights_q8=1)
    kv = m.kv_alloc(1, 128 + 24)
    glg, gam, _ = greedy_gpu(m, kv, prompt, toks[:-1], stream)
    assert_close(olg, glg, "q8_0 logits")
    assert_tokens(olg, toks, gam, "q8_0 greedy tokens")
    assert all(gam[i] == first_argmax(glg[i]) for i in range(len(gam)))


def test_llama32_1b_prefix_and_full_prompt(stream):
    """Llama-3.2-1B shape: a 128-token prefix and 4 steps against the oracle;
    the benchmark's 2048-token prefill then reproduces the prefix's hidden
    states (causality), equals the same prompt prefilled in two chunks, and
    greedy-decodes like the chunked cache."""
    name = "llama-3.2-1b"
    shape = synth.WORKLOADS[name].model
    w = weights(name)
    full = synth.prompt_ids(shape, 2048)
    prefix = full[:128]
    toks, olg, _ = O.OracleModel(shape, w).greedy(prefix, 4, kv_bf16=True)
    m = R.Model(shape, w, max_tokens=2048)
    kv = m.kv_alloc(2, 2048 + 8)
    glg, gam, ghd = greedy_gpu(m, kv, prefix, toks[:-1], stream)
    assert_close(olg, glg, "prefix logits")
    assert_tokens(olg, toks, gam, "prefix greedy tokens")

    # the full prompt in one piece (slot 0) and in two chunks (slot 1)
    H, V = shape.hidden, shape.vocab
    hid = torch.empty((2048, H), dtype=torch.float32, device="cuda")
    lg = torch.empty((2, V), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        kv.set_cursor(0, 0, stream=stream)
        m.prefill(kv, 0, i32(full), 0, logits=lg[0], hidden=hid, stream=stream)
        kv.set_cursor(1, 0, stream=stream)
        m.prefill(kv, 1, i32(full[:1000]), 0, stream=stream)
        m.prefill(kv, 1, i32(full[1000:]), 1000, logits=lg[1], stream=stream)
    assert m.sync_status(stream) == 0
    assert_close(ghd, hid[:128].cpu().numpy(), "prefix rows of the 2048-token prefill")
    lgn = lg.cpu().numpy()
    assert_close(lgn[0:1], lgn[1:2], "2048-token prefill vs two chunks")
    # sampled rows of the 2048-token prefill against the oracle: row t from the
    # GPU's cache rows [0, t) and token t (conditional parity), the last row's
    # logits too, and the K / V rows the prefill wrote at position t
    om = O.OracleModel(shape, w)
    K, Vc = kv.tensors()
    hidn = hid.cpu().numpy()
    for t in (500, 1300, 2047):
        oh, olg_t, ok, ov = oracle_step_on_gpu_cache(om, kv, 0, t, int(full[t]))
        assert_close(oh[None], hidn[t:t + 1], f"prefill row {t} hidden")
        if t == 2047:
            assert_close(olg_t[None], lgn[0:1], "prefill last-position logits")
        gk = O.bf16_decode(K[0][:, :, t].cpu().numpy().view(np.uint16))
        gv = O.bf16_decode(Vc[0][:, :, t].cpu().numpy().view(np.uint16))
        assert_close(ok.reshape(-1, 64), gk.reshape(-1, 64), f"prefill K row {t}")
        assert_close(ov.reshape(-1, 64), gv.reshape(-1, 64), f"prefill V row {t}")
    # four decode steps of both caches in one batch, both fed slot 0's argmax
    # (teacher forcing keeps the histories equal): the rows must agree
    ids = i32([first_argmax(lgn[0])] * 2)
    seqs2 = i32([0, 1])
    step_lg = torch.empty((4, 2, V), dtype=torch.float32, device="cuda")
    am = torch.zeros(2, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for i in range(4):
            m.decode_step(kv, seqs2, ids, None, logits=step_lg[i], argmax=am, stream=stream)
            ids.copy_(am[0:1].expand(2))
    assert m.sync_status(stream) == 0
    sl = step_lg.cpu().numpy()
    assert_close(sl[:, 0], sl[:, 1], "decode after the full vs the chunked prompt")


def test_batch64_decode_sampled_sequences(stream):
    """Qwen2.5-0.5B shape, 64 sequences: ragged short prompts with two
    sampled sequences against the oracle; then the benchmark's 4096-token
    caches, where a batched step's logits for sampled sequences equal the
    batch-1 (fused) step on the same cache."""
    name = "qwen2.5-0.5b"
    shape = synth.WORKLOADS[name].model
    w = weights(name)
    B = 64
    m = R.Model(shape, w, max_tokens=4096)
    V = shape.vocab

    # ragged short prompts, oracle on sequences 5 and 50
    lens = [24 + (7 * b) % 41 for b in range(B)]
    kv = m.kv_alloc(B, 80)
    prompts = [synth.prompt_ids(shape, lens[b], seq=b) for b in range(B)]
    cur = torch.zeros(B, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            m.prefill(kv, b, i32(prompts[b]), 0, argmax=cur[b:b + 1], stream=stream)
    lg = torch.empty((2, B, V), dtype=torch.float32, device="cuda")
    seqs = torch.arange(B, dtype=torch.int32, device="cuda")
    toks = [cur.clone()]
    with torch.cuda.stream(stream):
        for i in range(2):
            m.decode_step(kv, seqs, cur, None, logits=lg[i], argmax=cur, stream=stream)
            toks.append(cur.clone())
    assert m.sync_status(stream) == 0
    glg = lg.cpu().numpy()
    gt = np.stack([t.cpu().numpy() for t in toks])   # [3][B]: prefill argmax, step 1, step 2
    om = O.OracleModel(shape, w)
    for b in (5, 50):
        otoks, olg, _ = om.greedy(prompts[b], 2, forced=gt[:2, b], kv_bf16=True)
        assert_close(olg[1:], glg[:, b], f"seq {b} batched decode logits")
        assert_tokens(olg[1:], otoks[1:], gt[1:, b], f"seq {b} batched greedy")
    del kv

    # the benchmark's 4096-token caches: batched step vs the batch-1 step
    P = 4096
    kv = m.kv_alloc(B, P + 2)
    with torch.cuda.stream(stream):
        for b in range(B):
            m.prefill(kv, b, i32(synth.prompt_ids(shape, P, seq=b)), 0, argmax=cur[b:b + 1],
                      stream=stream)
    ids0 = cur.clone()
    lgb = torch.empty((B, V), dtype=torch.float32, device="cuda")
    amb = torch.empty(B, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        m.decode_step(kv, seqs, ids0, None, logits=lgb, argmax=amb, stream=stream)
    assert m.sync_status(stream) == 0
    # every sequence's 4096-key step against one oracle step from the GPU's own
    # cache rows (conditional parity of the decode step; a prefill of 64 x 4096
    # tokens is out of the oracle's reach)
    glb, gab, idn = lgb.cpu().numpy(), amb.cpu().numpy(), ids0.cpu().numpy()
    checked = 0
    for b in range(B):
        _, olg_b, _, _ = oracle_step_on_gpu_cache(om, kv, b, P, int(idn[b]))
        assert_close(olg_b[None], glb[b:b + 1], f"seq {b}: 4096-key step vs oracle")
        checked += assert_tokens(olg_b[None], [first_argmax(olg_b)], gab[b:b + 1], f"seq {b} token")
    assert checked > B // 2
    for b in (0, 37, 63):
        lg1 = torch.empty((1, V), dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            kv.set_cursor(b, P, stream=stream)   # the same position again
            m.decode_step(kv, i32([b]), ids0[b:b + 1].clone(), None, logits=lg1, stream=stream)
        assert m.sync_status(stream) == 0
        assert_close(lgb[b:b + 1].cpu().numpy(), lg1.cpu().numpy(),
                     f"seq {b}: batched vs batch-1 step at 4096 keys")


def test_encoder_8x512_sampled_sequence(stream):
    """Qwen3 encoder shape, 8 x 512: the label logits and final hidden states
    of a sampled sequence against the oracle (sequences are independent)."""
    name = "qwen3-encoder"
    wl = synth.WORKLOADS[name]
    shape = wl.model
    w = weights(name)
    B, T = wl.batch, wl.prompt
    m = R.Model(shape, w, max_tokens=B * T, max_positions=T)
    ids = np.concatenate([synth.prompt_ids(shape, T, seq=b) for b in range(B)])
    out = torch.empty((B * T, shape.n_labels), dtype=torch.float32, device="cuda")
    hid = torch.empty((B * T, shape.hidden), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        m.encode(i32(ids), B, T, out=out, hidden=hid, stream=stream)
    assert m.sync_status(stream) == 0
    b = 5
    ohd, _, ocl = O.OracleModel(shape, w).forward_full(ids[b * T:(b + 1) * T], logits=False, cls=True)
    assert_close(ocl, out[b * T:(b + 1) * T].cpu().numpy(), "label logits")
    assert_close(ohd, hid[b * T:(b + 1) * T].cpu().numpy(), "final hidden states")


@pytest.mark.slow
def test_batch64_full_run_of_one_sequence_against_oracle(stream):
    """Qwen2.5-0.5B shape, 64 sequences of 4096-token caches: the oracle's
    whole run of one sequence (its 4096-token prefill and 64 greedy steps,
    bf16 cache) against that sequence inside the batched GPU run, with the
    oracle's tokens fed to it (teacher forcing) so every step stays
    comparable; the other 63 sequences decode their own argmax beside it."""
    name = "qwen2.5-0.5b"
    shape = synth.WORKLOADS[name].model
    w = weights(name)
    B, P, S, s = 64, 4096, 64, 21
    m = R.Model(shape, w, max_tokens=4096)
    V = shape.vocab
    prompt_s = synth.prompt_ids(shape, P, seq=s)
    otoks, olg, _ = O.OracleModel(shape, w).greedy(prompt_s, S, kv_bf16=True, hidden=False)
    kv = m.kv_alloc(B, P + S + 1)
    cur = torch.zeros(B, dtype=torch.int32, device="cuda")
    plg = torch.empty(V, dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            m.prefill(kv, b, i32(synth.prompt_ids(shape, P, seq=b)), 0, argmax=cur[b:b + 1],
                      logits=plg if b == s else None, stream=stream)
    seqs = torch.arange(B, dtype=torch.int32, device="cuda")
    lg = torch.empty((S, V), dtype=torch.float32, device="cuda")
    am = torch.empty((S, B), dtype=torch.int32, device="cuda")
    full = torch.empty((B, V), dtype=torch.float32, device="cuda")
    forced = i32(otoks[:S])
    with torch.cuda.stream(stream):
        for i in range(S):
            cur[s:s + 1].copy_(forced[i:i + 1])
            m.decode_step(kv, seqs, cur, None, logits=full, argmax=cur, stream=stream)
            lg[i].copy_(full[s])
            am[i].copy_(cur)
    assert m.sync_status(stream) == 0
    glg = np.concatenate([plg.cpu().numpy()[None], lg.cpu().numpy()])
    gam = np.concatenate([[first_argmax(glg[0])], am.cpu().numpy()[:, s]])
    assert_close(olg, glg, f"seq {s}: prefill + {S} batched steps vs the oracle's run")
    assert assert_tokens(olg, otoks, gam, f"seq {s} greedy tokens") > S // 2
