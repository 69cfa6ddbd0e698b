"""The C ABI library builds, loads and exports every symbol include/ember.h
declares; host-side argument checks run without a GPU (no compute calls)."""
import ctypes as C
import json
import os
import re

import pytest

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "ember.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ember_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = E.load()
    names = declared_symbols()
    assert len(names) >= 14, names
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_kv_bytes_matches_the_pages_worked_example():
    """ember internals, "kv cache" layout: GPT-2 small at 2048 context, factors
    12 layers x 12 heads x 2048 x 64 x 4 bytes x 2 (K and V).  The printed
    total (~72 MB) is one tensor's share; the factor product is the size of
    both.  The library stores bf16, so its figure is half the f32 one."""
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_size_gpt2_small.json")))
    cfg = E.ember_config(vocab=50257, hidden=768, layers=g["layers"], n_heads=g["heads"],
                         n_kv_heads=g["heads"], head_dim=g["head_dim"], ff=3072)
    f32_bytes = E.ember_kv_bytes(cfg, 1, g["max_seq_len"]) * g["dtype_bytes"] // 2
    assert f32_bytes == g["bytes_f32_product_of_factors"]
    assert abs(f32_bytes / 2 / 2 ** 20 - g["stated_total_mb"]) < 0.5


def _create(shape, weights_q8=0, **over):
    d = {**shape.asdict(), **over}
    cfg = E.make_config(d, weights_q8=weights_q8)
    w = E.ember_weights()
    out = C.c_void_p()
    st = E.load().ember_model_create(C.byref(cfg), C.byref(w), C.byref(out))
    return st, E.last_error()


@pytest.mark.parametrize("over,msg", [
    (dict(n_kv_heads=3), "GQA"),          # Falcon-H1 Config::validate: heads % kv_heads
    (dict(head_dim=15), "GQA"),           # odd head_dim
    (dict(hidden=0), "zero dimension"),
    (dict(vocab=0), "zero dimension"),
    (dict(rope_theta=0.0), "rope_theta"),
])
def test_invalid_configs_are_rejected_on_the_host(over, msg):
    st, err = _create(synth.TINY, **over)
    assert st == 1 and msg in err, (st, err)


def test_missing_weights_are_reported():
    st, err = _create(synth.TINY)
    assert st == 1 and "missing weight" in err


def test_unsupported_shapes_say_so():
    st, err = _create(synth.TINY, head_dim=24, n_heads=4, n_kv_heads=2)
    assert st == 8 and "head_dim" in err


@pytest.mark.parametrize("q8,over,status,msg", [
    (2, dict(), 1, "weights_q8 must be 0 or 1"),
    # q8_0 blocks of 32 along every layer matrix's input dimension
    (1, dict(hidden=112, n_heads=7, n_kv_heads=1, head_dim=16, ff=160), 8, "multiples of 32"),
    (0, dict(n_heads=34, n_kv_heads=2), 8, "GQA group > 16"),
    (0, dict(hidden=8200), 8, "hidden > 8192"),
    (0, dict(hidden=100), 8, "multiples of 8"),
])
def test_limits_and_the_q8_0_flag_are_checked_before_any_device_work(q8, over, status, msg):
    st, err = _create(synth.TINY, weights_q8=q8, **over)
    assert st == status and msg in err, (st, err)


def _zero_args(f):
    """NULL for every pointer, 0 for every number, following the binding's
    argument types."""
    out = []
    for t in f.argtypes:
        if t in (C.c_float, C.c_double):
            out.append(t(0.0))
        elif t in (C.c_int32, C.c_int64, C.c_uint32, C.c_uint64, C.c_size_t):
            out.append(t(0))
        else:
            out.append(None)
    return out


def test_every_status_entry_rejects_null_arguments_before_device_work():
    """Each ember_status entry point answers INVALID_ARG (with a message) when
    its handles / buffers are NULL, without reaching the CUDA runtime."""
    lib = E.load()
    status_entries = [n for n in declared_symbols()
                      if getattr(lib, n).restype is C.c_int and getattr(lib, n).argtypes]
    assert len(status_entries) >= 15, status_entries
    for n in status_entries:
        f = getattr(lib, n)
        st = f(*_zero_args(f))
        assert st == 1, (n, st, E.last_error())
        assert E.last_error(), n
    # the void destructors accept NULL; the size query answers 0
    lib.ember_model_destroy(None)
    lib.ember_kv_free(None)
    assert lib.ember_kv_bytes(None, 1, 1) == 0
