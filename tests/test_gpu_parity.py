"""Whole-forward parity of the CUDA library against the CPU oracle, through the
C ABI, on seeded synthetic weights: prefill + greedy decode, token-by-token
decode, chunked prefill, batched decode on both decode paths, the bf16 KV
cache contents, device-side argument errors and the encoder."""
import numpy as np
import pytest
import torch

from gqa_transformer_decode_gb300 import runtime as R
from gqa_transformer_decode_gb300 import synth
from oracle import oracle as O

from parity_util import assert_close, assert_tokens, first_argmax, oracle_step_on_gpu_cache

pytestmark = pytest.mark.gpu

SMALL_QWEN2 = synth.ModelShape("s-qwen2", vocab=300, hidden=112, layers=3, n_heads=14,
                               n_kv_heads=2, head_dim=16, ff=160, rope_theta=1e6, qkv_bias=1)
SMALL_LLAMA = synth.ModelShape("s-llama", vocab=1000, hidden=256, layers=2, n_heads=8,
                               n_kv_heads=2, head_dim=32, ff=512, rope_theta=5e5,
                               rope_llama3=1, rs_factor=32.0, rs_low=1.0, rs_high=4.0,
                               rs_orig_max_pos=64)
SMALL_ENC = synth.ModelShape("s-enc", vocab=500, hidden=256, layers=2, n_heads=4, n_kv_heads=2,
                             head_dim=128, ff=384, rope_theta=1e6, qk_norm=1, causal=0,
                             n_labels=16)

_cache = {}


def model_pair(shape, max_tokens=512):
    key = (shape.name, max_tokens)
    if key not in _cache:
        w = synth.weights_bf16(shape)
        _cache[key] = (w, O.OracleModel(shape, w), R.Model(shape, w, max_tokens=max_tokens))
    return _cache[key]


@pytest.fixture(scope="module")
def stream():
    return torch.cuda.Stream()


def i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def run_greedy_gpu(model, kv, prompt, n_steps, forced, stream, seq=0, pos0=0):
    """Prefill, then n_steps decode steps fed the given tokens (teacher forcing
    with the oracle's tokens keeps later steps comparable)."""
    V, H, n = model.V, model.H, len(prompt)
    logits = torch.empty((n_steps + 1, V), dtype=torch.float32, device="cuda")
    hidden = torch.empty((n, H), dtype=torch.float32, device="cuda")
    amax = torch.empty(n_steps + 1, dtype=torch.int32, device="cuda")
    ids = i32(prompt)
    with torch.cuda.stream(stream):
        model.prefill(kv, seq, ids, pos0, logits=logits[0], argmax=amax[0:1], hidden=hidden,
                      stream=stream)
        seqs = i32([seq])
        for i in range(1, n_steps + 1):
            tok = i32([forced[i - 1]])
            pos = i32([pos0 + n + i - 1])
            model.decode_step(kv, seqs, tok, pos, logits=logits[i], argmax=amax[i:i + 1],
                              stream=stream)
    st = model.sync_status(stream)
    assert st == 0, st
    return logits.cpu().numpy(), amax.cpu().numpy(), hidden.cpu().numpy()


@pytest.mark.parametrize("shape,n_prompt,n_steps", [(synth.TINY, 8, 16), (SMALL_QWEN2, 37, 12),
                                                    (SMALL_LLAMA, 150, 10)])
def test_prefill_and_greedy_decode_match_oracle(shape, n_prompt, n_steps, stream):
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, n_prompt)
    toks, olg, ohd = om.greedy(prompt, n_steps)
    kv = gm.kv_alloc(2, n_prompt + n_steps + 8)
    glg, gam, ghd = run_greedy_gpu(gm, kv, prompt, n_steps, toks[:-1], stream)
    h_full, _, _ = om.forward_full(np.concatenate([prompt, toks[:-1]]), logits=False)
    assert_close(h_full[:n_prompt], ghd, "prefill hidden")
    assert_close(olg, glg, "logits")
    assert_tokens(olg, toks, gam, "greedy tokens")
    for i in range(n_steps + 1):   # argmax is the first maximum of the GPU's own logits
        assert gam[i] == first_argmax(glg[i])


def test_token_by_token_decode_equals_oracle(stream):
    """ember reference_forward.py main(): the prompt fed one token at a time."""
    shape = SMALL_QWEN2
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, 9)
    _, olg, _ = om.forward_full(prompt)
    kv = gm.kv_alloc(1, 16)
    lg = torch.empty((9, shape.vocab), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        for t in range(9):
            gm.decode_step(kv, i32([0]), i32([prompt[t]]), i32([t]), logits=lg[t], stream=stream)
    assert gm.sync_status(stream) == 0
    assert_close(olg, lg.cpu().numpy(), "token-by-token logits")


def test_chunked_prefill_equals_single_prefill(stream):
    shape = SMALL_LLAMA
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, 200)
    _, olg, _ = om.forward_full(prompt)
    kv = gm.kv_alloc(1, 256)
    lg = torch.empty((2, shape.vocab), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        gm.prefill(kv, 0, i32(prompt[:130]), 0, logits=lg[0], stream=stream)
        gm.prefill(kv, 0, i32(prompt[130:]), 130, logits=lg[1], stream=stream)
    assert gm.sync_status(stream) == 0
    assert_close(olg[[129, 199]], lg.cpu().numpy(), "chunked prefill logits")


def test_kv_cache_rows_match_oracle(stream):
    shape = SMALL_QWEN2
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, 20)
    oc = om.new_cache(24)
    om.forward_cached(oc, prompt)
    kv = gm.kv_alloc(2, 24)
    with torch.cuda.stream(stream):
        gm.prefill(kv, 1, i32(prompt), 0, stream=stream)
    assert gm.sync_status(stream) == 0
    K, V = kv.tensors()
    gk = O.bf16_decode(K[1].cpu().numpy().view(np.uint16))[:, :, :20]
    gv = O.bf16_decode(V[1].cpu().numpy().view(np.uint16))[:, :, :20]
    ok, ov = oc.arrays()
    assert_close(ok[:, :, :20].reshape(-1, shape.head_dim), gk.reshape(-1, shape.head_dim), "K")
    assert_close(ov[:, :, :20].reshape(-1, shape.head_dim), gv.reshape(-1, shape.head_dim), "V")
    # nothing written past the prompt, nothing in the other sequence
    assert not K[0].any() and not K[1][:, :, 20:].any()


@pytest.mark.parametrize("B", [3, 8, 13])
def test_batched_decode_matches_oracle_per_sequence(B, stream):
    """B sequences with different prompt lengths decoded together (B <= 8 on
    the GEMV path, larger on the tensor-core path)."""
    shape = SMALL_QWEN2
    w, om, gm = model_pair(shape)
    lens = [5 + 3 * b for b in range(B)]
    kv = gm.kv_alloc(B, 64)
    prompts = [synth.prompt_ids(shape, L, seq=b) for b, L in enumerate(lens)]
    nxt = [synth.uniform_ids(7, f"next.{b}", 3, shape.vocab) for b in range(B)]
    lg = torch.empty((3, B, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty((3, B), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            gm.prefill(kv, b, i32(prompts[b]), 0, stream=stream)
        seqs = i32(list(range(B)))
        for s in range(3):
            gm.decode_step(kv, seqs, i32([nxt[b][s] for b in range(B)]),
                           i32([lens[b] + s for b in range(B)]), logits=lg[s], argmax=am[s],
                           stream=stream)
    assert gm.sync_status(stream) == 0
    glg = lg.cpu().numpy()
    gam = am.cpu().numpy()
    for b in range(B):
        _, olg, _ = om.forward_full(np.concatenate([prompts[b], nxt[b]]))
        assert_close(olg[lens[b]:lens[b] + 3], glg[:, b], f"seq {b}")
        for s in range(3):
            assert gam[s, b] == first_argmax(glg[s, b])


def test_device_status_errors(stream):
    shape = synth.TINY
    w, om, gm = model_pair(shape)
    kv = gm.kv_alloc(2, 16)
    with torch.cuda.stream(stream):
        gm.prefill(kv, 0, i32([1, 2, 3]), 0, stream=stream)
    assert gm.sync_status(stream) == 0
    with torch.cuda.stream(stream):   # position 5 != cursor 3
        gm.decode_step(kv, i32([0]), i32([4]), i32([5]), stream=stream)
    assert gm.sync_status(stream) == 3
    with torch.cuda.stream(stream):   # token outside the vocabulary
        gm.decode_step(kv, i32([1]), i32([shape.vocab + 5]), i32([0]), stream=stream)
    assert gm.sync_status(stream) == 4
    with torch.cuda.stream(stream):   # seq out of range
        gm.decode_step(kv, i32([7]), i32([1]), i32([0]), stream=stream)
    assert gm.sync_status(stream) == 1
    with torch.cuda.stream(stream):   # prefill at the wrong start position
        gm.prefill(kv, 1, i32([1, 2]), 4, stream=stream)
    assert gm.sync_status(stream) == 3
    with pytest.raises(R.E.EmberError) as ei:
        gm.prefill(kv, 0, i32(list(range(20))), 0, stream=stream)
    assert ei.value.status == 2   # capacity: 20 > max_len 16


@pytest.mark.parametrize("B,T", [(1, 7), (3, 40), (2, 130)])
def test_encoder_matches_oracle(B, T, stream):
    """PII-Tracer forward(): bidirectional, q/k norm, positions restart per
    sequence, 16-label head with bias."""
    shape = SMALL_ENC
    w, om, gm = model_pair(shape)
    ids = np.stack([synth.prompt_ids(shape, T, seq=b) for b in range(B)])
    out = torch.empty((B * T, shape.n_labels), dtype=torch.float32, device="cuda")
    hid = torch.empty((B * T, shape.hidden), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        gm.encode(i32(ids.reshape(-1)), B, T, out=out, hidden=hid, stream=stream)
    assert gm.sync_status(stream) == 0
    go, gh = out.cpu().numpy(), hid.cpu().numpy()
    for b in range(B):
        h, _, cls = om.forward_full(ids[b], logits=False, cls=True)
        assert_close(h, gh[b * T:(b + 1) * T], f"encoder hidden seq {b}")
        assert_close(cls, go[b * T:(b + 1) * T], f"encoder labels seq {b}")


SMALL_ENC_TIED = synth.ModelShape("s-enc-tied", vocab=700, hidden=256, layers=2, n_heads=4,
                                  n_kv_heads=2, head_dim=128, ff=384, rope_theta=1e6, qk_norm=1,
                                  causal=0, n_labels=0)


@pytest.mark.parametrize("B,T", [(3, 9), (2, 70), (1, 200)])
def test_encoder_with_the_tied_vocabulary_head(B, T, stream):
    """n_labels = 0: ember_encode writes the tied-head logits E . h at every
    position ([B*T, vocab]); B*T <= 128 runs the one-row-tile GEMM, more rows
    the persistent one."""
    shape = SMALL_ENC_TIED
    w, om, gm = model_pair(shape)
    ids = np.stack([synth.prompt_ids(shape, T, seq=b) for b in range(B)])
    out = torch.empty((B * T, shape.vocab), dtype=torch.float32, device="cuda")
    hid = torch.empty((B * T, shape.hidden), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        gm.encode(i32(ids.reshape(-1)), B, T, out=out, hidden=hid, stream=stream)
    assert gm.sync_status(stream) == 0
    go, gh = out.cpu().numpy(), hid.cpu().numpy()
    for b in range(B):
        h, lg, _ = om.forward_full(ids[b], logits=True)
        assert_close(h, gh[b * T:(b + 1) * T], f"encoder hidden seq {b}")
        assert_close(lg, go[b * T:(b + 1) * T], f"tied-head logits seq {b}")


def test_graph_replayed_greedy_loop_with_cursor_positions(stream):
    """positions = NULL (each token at its sequence's cursor) and argmax fed
    back as the next ids: one CUDA graph replayed every step; then the cursor
    is rewound and the same continuation is produced again."""
    shape = SMALL_QWEN2
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, 11)
    toks, olg, _ = om.greedy(prompt, 8)
    kv = gm.kv_alloc(1, 32)
    cur = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = i32([0])
    lg = torch.empty((9, shape.vocab), dtype=torch.float32, device="cuda")
    got = []
    for rep in range(2):
        out = torch.empty(9, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            kv.set_cursor(0, 0, stream=stream)
            gm.prefill(kv, 0, i32(prompt), 0, argmax=cur, logits=lg[0], stream=stream)
            out[0:1].copy_(cur)
            for i in range(1, 9):
                gm.decode_step(kv, seqs, cur, None, argmax=cur, stream=stream)
                out[i:i + 1].copy_(cur)
        assert gm.sync_status(stream) == 0
        got.append(out.cpu().numpy())
    assert np.array_equal(got[0], got[1])
    assert_tokens(olg, toks, got[0], "graph greedy")


# head_dim 64 / 128 decoders: prompts run through the tensor-core attention
MID_QWEN2 = synth.ModelShape("m-qwen2", vocab=2000, hidden=448, layers=2, n_heads=7,
                             n_kv_heads=1, head_dim=64, ff=640, rope_theta=1e6, qkv_bias=1)
MID_LLAMA = synth.ModelShape("m-llama", vocab=1500, hidden=256, layers=2, n_heads=8,
                             n_kv_heads=2, head_dim=64, ff=512, rope_theta=5e5, rope_llama3=1,
                             rs_factor=32.0, rs_low=1.0, rs_high=4.0, rs_orig_max_pos=256)
MID_D128 = synth.ModelShape("m-d128", vocab=900, hidden=256, layers=2, n_heads=4, n_kv_heads=2,
                            head_dim=128, ff=384, rope_theta=1e6, qk_norm=1)


@pytest.mark.parametrize("shape,n_prompt", [(MID_QWEN2, 1), (MID_QWEN2, 150), (MID_LLAMA, 128),
                                            (MID_LLAMA, 300), (MID_D128, 77), (MID_D128, 257)])
def test_tensor_core_prefill_matches_oracle(shape, n_prompt, stream):
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, n_prompt)
    toks, olg, _ = om.greedy(prompt, 3)
    kv = gm.kv_alloc(1, n_prompt + 8)
    glg, gam, ghd = run_greedy_gpu(gm, kv, prompt, 3, toks[:-1], stream)
    h_full, _, _ = om.forward_full(prompt, logits=False)
    assert_close(h_full, ghd, "prefill hidden")
    assert_close(olg, glg, "logits")
    assert_tokens(olg, toks, gam, "greedy tokens")


def test_tensor_core_chunked_prefill(stream):
    """Second chunk starts at position 200 (not a key-tile boundary)."""
    shape = MID_LLAMA
    w, om, gm = model_pair(shape)
    prompt = synth.prompt_ids(shape, 420)
    _, olg, _ = om.forward_full(prompt)
    kv = gm.kv_alloc(2, 448)
    lg = torch.empty((3, shape.vocab), dtype=torch.float32, device="cuda")
    hid = torch.empty((220, shape.hidden), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        gm.prefill(kv, 1, i32(prompt[:200]), 0, logits=lg[0], stream=stream)
        gm.prefill(kv, 1, i32(prompt[200:]), 200, logits=lg[1], hidden=hid, stream=stream)
    assert gm.sync_status(stream) == 0
    assert_close(olg[[199, 419]], lg[:2].cpu().numpy(), "chunked prefill logits")
    h_full, _, _ = om.forward_full(prompt, logits=False)
    assert_close(h_full[200:], hid.cpu().numpy(), "second chunk hidden")


@pytest.mark.parametrize("shape,n_prompt,n_steps,seq", [(MID_QWEN2, 1, 20, 0),
                                                        (MID_QWEN2, 124, 8, 0),
                                                        (MID_QWEN2, 380, 8, 1),
                                                        (MID_LLAMA, 2100, 6, 1),
                                                        (MID_D128, 300, 8, 1)])
def test_fused_batch1_decode_matches_oracle(shape, n_prompt, n_steps, seq, stream):
    """Batch-1 decode on the two-kernels-per-layer path (head_dim 64 / 128): one
    key; contexts crossing 128 keys (one CTA, second tile double-buffered) and
    384 keys (one CTA -> keys spread over the cluster); a context of more than
    16 tiles of 128 keys (every CTA of a cluster loops over two tiles); three
    tiles in one CTA and q/k norm with head_dim 128; second cache slot."""
    w, om, gm = model_pair(shape, max_tokens=max(512, n_prompt + 16))
    prompt = synth.prompt_ids(shape, n_prompt)
    toks, olg, _ = om.greedy(prompt, n_steps)
    kv = gm.kv_alloc(2, n_prompt + n_steps + 8)
    glg, gam, _ = run_greedy_gpu(gm, kv, prompt, n_steps, toks[:-1], stream, seq=seq)
    assert_close(olg, glg, "logits")
    assert_tokens(olg, toks, gam, "greedy tokens")
    for i in range(n_steps + 1):
        assert gam[i] == first_argmax(glg[i])
    # the step ran as embed + two kernels per layer + LM head + finish
    from gqa_transformer_decode_gb300 import ember as E
    pos = n_prompt + n_steps
    l0 = E.ember_kernel_launches()
    with torch.cuda.stream(stream):
        gm.decode_step(kv, i32([seq]), i32([toks[-1]]), i32([pos]), stream=stream)
    assert gm.sync_status(stream) == 0
    assert E.ember_kernel_launches() - l0 == 2 * shape.layers + 3


@pytest.mark.parametrize("shape,n_prompt,cl", [(MID_LLAMA, 2100, 12), (MID_QWEN2, 500, 9),
                                             (MID_D128, 700, 11)])
def test_fused_batch1_decode_with_smaller_clusters(shape, n_prompt, cl, stream, monkeypatch):
    """Batch-1 decode on clusters of fewer than 16 CTAs (the plan's choice
    when 16-CTA clusters for every kv head do not fit on the chip at once),
    over contexts past the single-CTA range so that every CTA of the cluster
    takes keys, receives every q/k/v row and merges a slice of the heads."""
    from gqa_transformer_decode_gb300 import ember as E
    monkeypatch.setenv("EMBER_FUSED_CLUSTER", str(cl))
    w = synth.weights_bf16(shape)
    gm = R.Model(shape, w, max_tokens=max(512, n_prompt + 16))
    monkeypatch.delenv("EMBER_FUSED_CLUSTER")
    om = model_pair(shape)[1]
    n_steps = 4
    prompt = synth.prompt_ids(shape, n_prompt)
    toks, olg, _ = om.greedy(prompt, n_steps)
    kv = gm.kv_alloc(1, n_prompt + n_steps + 8)
    glg, gam, _ = run_greedy_gpu(gm, kv, prompt, n_steps, toks[:-1], stream)
    assert_close(olg, glg, "logits")
    assert_tokens(olg, toks, gam, "greedy tokens")
    l0 = E.ember_kernel_launches()   # still the fused path: embed, 2 per layer, head, finish
    with torch.cuda.stream(stream):
        gm.decode_step(kv, i32([0]), i32([toks[-1]]), i32([n_prompt + n_steps]), stream=stream)
    assert gm.sync_status(stream) == 0
    assert E.ember_kernel_launches() - l0 == 2 * shape.layers + 3
    gm.close()


def test_traced_decode_step_matches_the_step_and_names_its_launches(stream):
    """ember_decode_step_traced computes the same step (logits, argmax, cache
    cursor) as ember_decode_step and reports every launch in order: embed, an
    attention and an MLP kernel per layer, the LM head and finish, each with
    a positive device time."""
    shape = MID_QWEN2
    w, om, gm = model_pair(shape, max_tokens=64)
    prompt = synth.prompt_ids(shape, 40)
    kv = gm.kv_alloc(2, 64)
    V = shape.vocab
    lg = torch.empty((2, V), dtype=torch.float32, device="cuda")
    am = torch.zeros(2, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for seq in (0, 1):
            gm.prefill(kv, seq, i32(prompt), 0, argmax=am[seq:seq + 1], stream=stream)
        gm.decode_step(kv, i32([0]), am[0:1].clone(), None, logits=lg[0], stream=stream)
    trace = gm.decode_step_traced(kv, i32([1]), am[1:2].clone(), None, logits=lg[1],
                                  argmax=am[1:2], stream=stream)
    assert gm.sync_status(stream) == 0
    g = lg.cpu().numpy()
    assert_close(g[0:1], g[1:2], "traced vs graph-replayed step")   # split-K sums: order may differ
    assert int(am[1].item()) == first_argmax(g[1])
    names = [n.split("<")[0] for n, _ in trace]
    L = shape.layers
    assert names == ["k_embed"] + ["k_fused_attn", "k_fused_mlp"] * L + ["k_gemv", "k_finish"], names
    assert all(us > 0 for _, us in trace)
    # the cursor advanced: the next normal step of slot 1 is accepted at position 41
    with torch.cuda.stream(stream):
        gm.decode_step(kv, i32([1]), am[1:2].clone(), i32([41]), stream=stream)
    assert gm.sync_status(stream) == 0


@pytest.mark.parametrize("shape", [SMALL_QWEN2, MID_QWEN2])
def test_decode_graph_follows_a_new_cache_with_the_same_buffers(shape, stream):
    """A decode graph is bound to the KV cache it was captured against: the same
    seqs / ids / argmax tensors used with a second cache (after the first one
    is freed) must read and write the second cache."""
    w, om, gm = model_pair(shape)
    seqs, cur = i32([0]), i32([0])
    got = []
    for k, n_prompt in enumerate((11, 23)):
        prompt = synth.prompt_ids(shape, n_prompt, seq=k)
        kv = gm.kv_alloc(1, 64 + 40 * k)   # another row stride: a stale graph misreads it
        out = torch.empty(5, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            gm.prefill(kv, 0, i32(prompt), 0, argmax=cur, stream=stream)
            out[0:1].copy_(cur)
            for i in range(1, 5):
                gm.decode_step(kv, seqs, cur, None, argmax=cur, stream=stream)
                out[i:i + 1].copy_(cur)
        assert gm.sync_status(stream) == 0
        toks, olg, _ = om.greedy(prompt, 4)
        assert_tokens(olg, toks, out.cpu().numpy(), f"cache {k} greedy")
        kv.close()


@pytest.mark.parametrize("shape", [MID_QWEN2, MID_LLAMA, MID_D128])
def test_batched_tensor_core_decode_attention_at_multi_split_contexts(shape, stream):
    """Batch 3 (head_dim 64 / 128: k_attn_decode_mma) at ragged contexts of 130,
    700 and 2100 keys -- 3, 11 and 32 key splits whose partials the last CTA of
    each (token, kv head) merges -- for G = 7, 4 and 2, two steps, against the
    oracle's whole run (bf16 cache on both sides)."""
    w, om, gm = model_pair(shape, max_tokens=2112)
    lens = [130, 700, 2100]
    B, n_steps = 3, 2
    kv = gm.kv_alloc(B, 2100 + 8)
    prompts = [synth.prompt_ids(shape, n, seq=b) for b, n in enumerate(lens)]
    nxt = [synth.uniform_ids(11, f"mma.{b}", n_steps, shape.vocab) for b in range(B)]
    lg = torch.empty((n_steps, B, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty((n_steps, B), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            gm.prefill(kv, b, i32(prompts[b]), 0, stream=stream)
        seqs = i32(list(range(B)))
        for s in range(n_steps):
            gm.decode_step(kv, seqs, i32([nxt[b][s] for b in range(B)]),
                           i32([lens[b] + s for b in range(B)]), logits=lg[s], argmax=am[s],
                           stream=stream)
    assert gm.sync_status(stream) == 0
    glg, gam = lg.cpu().numpy(), am.cpu().numpy()
    for b in range(B):
        # greedy with the forced tokens: logits of the prompt's last position,
        # then of each forced step
        _, olg, _ = om.greedy(prompts[b], n_steps, forced=nxt[b], kv_bf16=True)
        assert_close(olg[1:], glg[:, b], f"{shape.name} seq {b} ({lens[b]} keys)")
        for s in range(n_steps):
            assert gam[s, b] == first_argmax(glg[s, b])


@pytest.mark.parametrize("shape", [MID_LLAMA, MID_D128])
def test_batch64_decode_ring_wraps_against_oracle_on_the_gpu_cache(shape, stream):
    """64 sequences with ragged contexts up to 3100 keys: two key splits per
    (token, kv head), so one CTA streams up to 13 tiles of 128 keys through its
    2-3 stage copy ring (the ring wraps several times); the projections run on
    the tensor-core GEMMs (batch > 8).  Every sequence's step is checked
    against one oracle step started from the GPU's own cache rows."""
    w, om, gm = model_pair(shape, max_tokens=3200)
    B = 64
    lens = [200 + (97 * b) % 2900 for b in range(B)]
    assert max(lens) > 3000
    kv = gm.kv_alloc(B, 3200)
    nxt = synth.uniform_ids(13, "ring", B, shape.vocab)
    lg = torch.empty((B, shape.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for b in range(B):
            gm.prefill(kv, b, i32(synth.prompt_ids(shape, lens[b], seq=b)), 0, stream=stream)
        gm.decode_step(kv, torch.arange(B, dtype=torch.int32, device="cuda"), i32(nxt), None,
                       logits=lg, argmax=am, stream=stream)
    assert gm.sync_status(stream) == 0
    glg, gam = lg.cpu().numpy(), am.cpu().numpy()
    K, V = kv.tensors()
    for b in range(B):
        _, olg, ok, ov = oracle_step_on_gpu_cache(om, kv, b, lens[b], nxt[b])
        assert_close(olg[None], glg[b:b + 1], f"{shape.name} seq {b} ({lens[b]} keys)")
        assert gam[b] == first_argmax(glg[b])
        if b % 16 == 0:   # the new K / V row the step wrote, against the oracle's
            gk = O.bf16_decode(K[b][:, :, lens[b]].cpu().numpy().view(np.uint16))
            gv = O.bf16_decode(V[b][:, :, lens[b]].cpu().numpy().view(np.uint16))
            assert_close(ok.reshape(-1, shape.head_dim), gk.reshape(-1, shape.head_dim), "K row")
            assert_close(ov.reshape(-1, shape.head_dim), gv.reshape(-1, shape.head_dim), "V row")
