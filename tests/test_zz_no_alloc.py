"""The allocation-free greedy LM head (ember_gemv_argmax_noalloc) against the
allocating entry point it varies (ember_gemv_bf16, whose logits give the
expected argmax) and against an f64 numpy product of the same bf16 weights and
f32 inputs, on two calls in a row so that the scratch clearing between calls
is exercised, and once more with a CUDA error left pending on the calling
thread.  Collected last; passes alone and after the other tests."""
import ctypes
import os

import numpy as np
import pytest

from gqa_transformer_decode_gb300 import ember as E
from gqa_transformer_decode_gb300 import synth
from parity_util import GAP, MAX_ABS


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_rows_beyond_the_fixed_scratch_are_rejected_on_the_host():
    """nb > EMBER_NOALLOC_MAX_ROWS fails before any device work; the pointers
    are never touched."""
    fake = ctypes.c_void_p(256)
    st = E.ember_gemv_argmax_noalloc(fake, 64, 64, fake, 9, None, fake, None)
    assert st == 2, E.STATUS_NAMES.get(st)
    assert "EMBER_NOALLOC_MAX_ROWS = 8" in E.last_error()


def _cudart():
    """The CUDA runtime this process already loaded (the library links it shared)."""
    for line in open(f"/proc/{os.getpid()}/maps"):
        path = line.split()[-1]
        if "libcudart.so" in path:
            return ctypes.CDLL(path)
    return None


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(N, K, nb, seed):
    rng = np.random.default_rng(seed)
    w = synth.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.05).astype(np.float32))
    x = rng.standard_normal((nb, K)).astype(np.float32)
    if nb > 1:
        # an exact tie at the top of row 1 (two identical weight rows along x[1]):
        # the first of the two indices must win
        w[N // 3] = synth.f32_to_bf16_bits((x[1] * 0.15).astype(np.float32))
        w[N - 1] = w[N // 3]
    return w, x


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,nb", [(151936, 896, 1), (32000, 2048, 1), (5003, 2048, 5),
                                    (1001, 64, 8), (130, 16384, 3)])
def test_noalloc_argmax_matches_the_allocating_gemv(N, K, nb):
    import torch
    w, x = _case(N, K, nb, N + K + nb)
    wd = torch.from_numpy(w.view(np.int16)).cuda()
    xd = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    sp = ctypes.c_void_p(s.cuda_stream)

    y_ref = torch.full((nb, N), float("nan"), dtype=torch.float32, device="cuda")
    E.check(E.ember_gemv_bf16(_p(wd), N, K, _p(xd), nb, _p(y_ref), sp), "ember_gemv_bf16")
    s.synchronize()
    ref = y_ref.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(ref))
    first = ref.argmax(axis=1)                      # numpy: first index of the max
    top2 = np.sort(ref, axis=1)[:, -2:]
    gap = top2[:, 1] - top2[:, 0]

    # an independent product: f64 numpy over the same bf16 weights and f32 x
    y64 = x.astype(np.float64) @ _bf16_to_f64(w).T
    assert np.abs(ref - y64).max() <= MAX_ABS
    first64 = y64.argmax(axis=1)
    s64 = np.sort(y64, axis=1)[:, -2:]
    gap64 = s64[:, 1] - s64[:, 0]
    rt = _cudart()

    for call in range(3):
        y = torch.full((nb, N), float("nan"), dtype=torch.float32, device="cuda") \
            if call == 0 else None
        am = torch.full((nb,), -1, dtype=torch.int32, device="cuda")
        pending = call == 2 and rt is not None
        if pending:   # an error the caller left on this thread (invalid device ordinal)
            rt.cudaSetDevice.argtypes = [ctypes.c_int]
            assert rt.cudaSetDevice(1 << 20) != 0
            assert rt.cudaPeekAtLastError() != 0
        st = E.ember_gemv_argmax_noalloc(_p(wd), N, K, _p(xd), nb, _p(y), _p(am), sp)
        if pending:   # still the caller's to collect, and the call did not fail on it
            assert rt.cudaPeekAtLastError() != 0
            rt.cudaGetLastError()
        E.check(st, f"ember_gemv_argmax_noalloc call {call}")
        s.synchronize()
        got = am.cpu().numpy()
        assert np.all((got >= 0) & (got < N)), (call, got)
        for b in range(nb):
            if gap[b] > GAP:
                assert got[b] == first[b], (call, b, got[b], first[b], gap[b])
            else:
                assert ref[b, got[b]] >= ref[b].max() - MAX_ABS, (call, b)
            if gap64[b] > GAP:
                assert got[b] == first64[b], (call, b, got[b], first64[b], gap64[b])
        if nb > 1:
            assert ref[1, N // 3] == ref[1, N - 1] == ref[1].max()
            assert got[1] == N // 3, (call, got[1])
        if y is not None:
            yg = y.cpu().numpy().astype(np.float64)
            assert np.abs(yg - ref).max() <= MAX_ABS, call
            assert np.abs(yg - y64).max() <= MAX_ABS, call
