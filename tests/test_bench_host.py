"""Host-side pieces of the measurement (no GPU): the traced decode step's
argument checks, the kernel-name reading of its trace, and the algorithmic
byte model bench.py divides by -- the per-kernel-family bytes of a decode
step must add up to the step's own algorithmic bytes (every bf16 weight
once plus the K/V rows), so the dominant kernel's roofline and the step's
HBM fraction count the same traffic."""
import ctypes as C
import importlib.util
import os
import types

import pytest

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traced_step_rejects_null_arguments_on_the_host():
    lib = E.load()
    n = C.c_int32(-1)
    st = lib.ember_decode_step_traced(None, None, 1, None, None, None, None, None, None,
                                      None, None, 0, C.byref(n))
    assert st == 1 and "NULL" in E.last_error(), (st, E.last_error())
    # trace buffers are required once cap > 0
    st = lib.ember_decode_step_traced(None, None, 1, None, None, None, None, None, None,
                                      None, None, 4, C.byref(n))
    assert st == 1


@pytest.mark.parametrize("mangled,name", [
    ("_ZN5ember12k_fused_attnILi64ELi4EEEv14CUtensorMap_stS1_NS_13FusedAttnArgsE", "k_fused_attn<64,4>"),
    ("_ZN5ember11k_fused_mlpILi8ELi4EEEvNS_12FusedMlpArgsE", "k_fused_mlp<8,4>"),
    ("_ZN5ember6k_gemvILi16ELi1ELb0ELb1EEEvNS_8GemvArgsE", "k_gemv<16,1,0,1>"),
    ("_ZN5ember7k_embedENS_9EmbedArgsE", "k_embed"),
    ("?", "?"),
])
def test_kernel_names_of_a_trace(mangled, name):
    assert E.kernel_name(mangled) == name


@pytest.mark.parametrize("key,B,fams", [
    ("qwen2.5-0.5b", 1, ("k_fused_attn", "k_fused_mlp", "k_gemv")),
    ("llama-3.2-1b", 1, ("k_fused_attn", "k_fused_mlp", "k_gemv")),
    ("qwen2.5-0.5b", 64, ("k_gemm_tcp", "k_attn_decode_mma")),
    ("qwen2.5-0.5b-q8_0", 1, ("k_gemv", "k_attn_decode_mma")),
])
def test_kernel_family_bytes_add_up_to_the_step(key, B, fams):
    bench = _bench()
    wl = synth.WORKLOADS[key]
    shape = wl.model
    ctx = 4097 if B > 1 else 200
    fam = bench.decode_family_bytes(shape, B, ctx, bool(wl.weights_q8))
    total = sum(fam[f] for f in fams)
    job = types.SimpleNamespace(wl=types.SimpleNamespace(model=shape, weights_q8=wl.weights_q8), B=B)
    step = bench.DecodeJob.bytes_per_decode_step(job, ctx - 1)   # ctx_mid + 1 keys
    # the families add the f32 residual stream and count biases as f32; the
    # step model counts the norm vectors: both differences are < 0.5 %
    assert abs(total - step) / step < 5e-3, (total, step)
    # the fused path's MLP block is exactly the three projection matrices
    if "k_fused_mlp" in fams:
        assert fam["k_fused_mlp"] == shape.layers * (3 * shape.ff * shape.hidden * 2 + 5 * shape.hidden * 4)
