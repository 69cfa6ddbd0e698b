#!/usr/bin/env python
"""Benchmark of the decoder forward on one GB300 (or N replicas).

Headline workload (one "step" = one whole generation job on the
Qwen2.5-0.5B-shaped decoder, random bf16 weights, batch 1): prefill of a
128-token uniform prompt, then 128 greedy decode steps, each fed the previous
argmax, through the C ABI (ember_prefill, ember_decode_step).  Weights (988 MB)
exceed the 129 MB L2, so no L2 flush is needed between steps.

The default run then measures the other three workloads of the metric, each
on a short timed region of its own, and reports them under "workloads": the
Llama-3.2-1B shape (2048-token prefill + 256 greedy steps, batch 1), the
Qwen2.5-0.5B shape at batch 64 over 4096-token caches (64 greedy steps), and
the Qwen3-style encoder (8 x 512 tokens).  Every record carries its value,
the roofline of its dominant kernel (or of the job where the work is a chain
of tensor-core GEMMs), the clocks seen while it ran and the CPU oracle timed
on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ember|reference]
                    [--workload qwen2.5-0.5b|llama-3.2-1b|qwen2.5-0.5b-b64|qwen3-encoder]
                    [--headline-only] [--no-cpu-baseline]

Timing: CUDA events on the launching stream around every job; a record's
time per job is the median over its timed jobs.  Prints one JSON line (rank
0).  --gpus N > 1 without a launcher re-runs this script under
torch.distributed.run with N processes (one replica per GPU).  --impl
reference times the CPU oracle on the host cores instead (bounded sample,
extrapolated to the same job), since the pages hold no runnable reference
implementation.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from gqa_transformer_decode_gb300 import synth  # noqa: E402

METRIC = "decode tok/s @B=1,64 + prefill tok/s (0.5B/1B shapes); HBM GB/s vs peak"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained",
                                                                         d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- distributed --
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------- GPU workloads --
class DecodeJob:
    """B sequences: prefill `prompt` tokens each, then `steps` greedy decode
    steps of the whole batch with argmax fed back as the next ids."""

    def __init__(self, wl: synth.Workload, weights, stream):
        import torch
        from gqa_transformer_decode_gb300 import runtime as R
        self.torch = torch
        self.wl = wl
        m = wl.model
        self.B, self.P, self.S = wl.batch, wl.prompt, wl.steps
        self.stream = stream
        self.model = R.Model(m, weights, max_tokens=max(self.P, 64), weights_q8=wl.weights_q8)
        self.kv = self.model.kv_alloc(self.B, self.P + self.S + 1)
        self.prompts = [torch.as_tensor(synth.prompt_ids(m, self.P, seq=b)).cuda()
                        for b in range(self.B)]
        self.seqs = torch.arange(self.B, dtype=torch.int32, device="cuda")
        self.cur = torch.zeros(self.B, dtype=torch.int32, device="cuda")
        self.prefill_in_job = self.B == 1
        if not self.prefill_in_job:   # batched decode: prompts prefilled once, outside timing
            with torch.cuda.stream(stream):
                for b in range(self.B):
                    self.model.prefill(self.kv, b, self.prompts[b], 0, argmax=self.cur[b:b + 1],
                                       stream=stream)
            assert self.model.sync_status(stream) == 0
            self.cur0 = self.cur.clone()

    def run(self, ev=None, host_ids=None, host_out=None):
        """One job; ev = (start, after_prefill, end) CUDA events."""
        torch, s, m, kv = self.torch, self.stream, self.model, self.kv
        with torch.cuda.stream(s):
            if ev:
                ev[0].record(s)
            # NVTX ranges name the phases for profilers (ncu --nvtx-include prefill/ | decode/)
            if self.prefill_in_job:
                kv.set_cursor(0, 0, stream=s)
                ids = self.prompts[0]
                if host_ids is not None:
                    ids = self._dev_ids
                    ids.copy_(host_ids, non_blocking=True)
                torch.cuda.nvtx.range_push("prefill")
                m.prefill(kv, 0, ids, 0, argmax=self.cur[0:1], stream=s)
                torch.cuda.nvtx.range_pop()
            else:   # every job restarts from the same prefilled caches and first tokens
                for b in range(self.B):
                    kv.set_cursor(b, self.P, stream=s)
                self.cur.copy_(self.cur0)
            if ev:
                ev[1].record(s)
            torch.cuda.nvtx.range_push("decode")
            for _ in range(self.S):
                m.decode_step(kv, self.seqs, self.cur, None, argmax=self.cur, stream=s)
            torch.cuda.nvtx.range_pop()
            if host_out is not None:
                host_out.copy_(self.cur, non_blocking=True)
            if ev:
                ev[2].record(s)

    def prepare_e2e(self):
        torch = self.torch
        self._dev_ids = torch.empty(self.P, dtype=torch.int32, device="cuda")
        host_ids = self.prompts[0].cpu().pin_memory()
        host_out = torch.empty(self.B, dtype=torch.int32).pin_memory()
        return host_ids, host_out

    def tokens_per_job(self):
        return self.B * self.S

    def bytes_per_decode_step(self, ctx_mid):
        """Algorithmic HBM bytes of one decode step: every bf16 weight once
        (layers + tied head) plus the KV rows read and the new rows written."""
        m = self.wl.model
        weights = 2 * m.params() - 2 * m.hidden   # bf16; final norm not re-read per token
        if self.wl.weights_q8:   # layer matrices as 34-byte blocks of 32 weights
            weights -= int((2 - 34 / 32) * m.layers * layer_matrix_params(m))
        kv_tok = m.layers * 2 * m.n_kv_heads * m.head_dim * 2
        return weights + self.B * kv_tok * (ctx_mid + 1)

    def prefill_flops(self):
        """Prefill FLOPs of the prompt: 2 * tokens * linear parameters of the
        layers, causal attention 2 * 2 * T^2 / 2 * D per head and layer, and
        the LM head at the last position."""
        m = self.wl.model
        H, D, F, T = m.hidden, m.head_dim, m.ff, self.P
        q, kv = m.n_heads * D, m.n_kv_heads * D
        lin = 2 * T * m.layers * ((q + 2 * kv) * H + q * H + 3 * F * H)
        att = 2 * T * T * D * m.n_heads * m.layers
        return lin + att + 2 * m.vocab * H


class EncodeJob:
    """B sequences of T tokens through the bidirectional encoder and the label
    head (ember_encode)."""

    def __init__(self, wl: synth.Workload, weights, stream):
        import torch
        from gqa_transformer_decode_gb300 import runtime as R
        self.torch = torch
        self.wl = wl
        m = wl.model
        self.B, self.T = wl.batch, wl.prompt
        self.stream = stream
        self.model = R.Model(m, weights, max_tokens=self.B * self.T, max_positions=self.T)
        ids = np.concatenate([synth.prompt_ids(m, self.T, seq=b) for b in range(self.B)])
        self.ids = torch.as_tensor(ids).cuda()
        self.out = torch.empty((self.B * self.T, m.n_labels), dtype=torch.float32, device="cuda")
        self.prefill_in_job = True

    def run(self, ev=None, host_ids=None, host_out=None):
        torch, s = self.torch, self.stream
        with torch.cuda.stream(s):
            if ev:
                ev[0].record(s)
            ids = self.ids
            if host_ids is not None:
                ids = self._dev_ids
                ids.copy_(host_ids, non_blocking=True)
            if ev:
                ev[1].record(s)
            torch.cuda.nvtx.range_push("encode")
            self.model.encode(ids, self.B, self.T, out=self.out, stream=s)
            torch.cuda.nvtx.range_pop()
            if host_out is not None:
                host_out.copy_(self.out, non_blocking=True)
            if ev:
                ev[2].record(s)

    def prepare_e2e(self):
        torch = self.torch
        self._dev_ids = torch.empty_like(self.ids)
        return self.ids.cpu().pin_memory(), torch.empty(tuple(self.out.shape)).pin_memory()

    def tokens_per_job(self):
        return self.B * self.T

    def flops_per_job(self):
        m = self.wl.model
        H, D, F = m.hidden, m.head_dim, m.ff
        q, kv = m.n_heads * D, m.n_kv_heads * D
        lin = 2 * self.B * self.T * m.layers * ((q + 2 * kv) * H + q * H + 3 * F * H)
        att = 4 * self.B * self.T * self.T * D * m.n_heads * m.layers
        return lin + att


def _family(name: str) -> str:
    return name.split("<")[0]


def layer_matrix_params(shape) -> int:
    H, D, F = shape.hidden, shape.head_dim, shape.ff
    return (shape.n_heads + 2 * shape.n_kv_heads) * D * H + H * shape.n_heads * D + 3 * F * H


def decode_family_bytes(shape, B: int, ctx: int, q8: bool = False) -> dict:
    """Algorithmic HBM bytes per decode step of each kernel family (weights
    in bf16, or the layer matrices as q8_0 at 34 bytes per 32 weights, once;
    K/V rows of ctx keys per sequence and kv head, bf16; the f32 residual
    stream: read x and z, write x, zero z, accumulate z)."""
    H, D, F, V, L = shape.hidden, shape.head_dim, shape.ff, shape.vocab, shape.layers
    NH, NKV = shape.n_heads, shape.n_kv_heads
    wb = 34 / 32 if q8 else 2
    qkv = int((NH + 2 * NKV) * D * H * wb) + (NH + 2 * NKV) * D * 4 * shape.qkv_bias
    o = int(H * NH * D * wb)
    mlp = int(3 * F * H * wb)
    kv_read = B * NKV * D * 2 * 2 * ctx
    kv_write = B * NKV * D * 2 * 2
    resid = 5 * B * H * 4
    head = V * H * 2
    if q8:   # every decode batch of a q8_0 model runs the split GEMVs
        return {"k_gemv": L * (qkv + o + mlp) + head,
                "k_attn_decode_mma": L * (kv_read + kv_write),
                "k_attn_decode": L * (kv_read + kv_write)}
    return {
        # batch-1 fused path: the attention block carries its projections
        "k_fused_attn": L * (qkv + o + kv_read + kv_write + resid),
        "k_fused_mlp": L * (mlp + resid),
        "k_fused_mlp_res": L * (mlp + resid),
        "k_gemv": head,
        # batched path: projections and head on the tensor-core GEMM, attention
        # reads the cache
        "k_gemm_tcp": L * (qkv + o + mlp) + head,
        "k_gemm_tc": L * (qkv + o + mlp) + head,
        "k_attn_decode_mma": L * (kv_read + kv_write),
        "k_attn_decode": L * (kv_read + kv_write),
    }


# dram__bytes_read.sum + dram__bytes_write.sum per launch of a kernel, from an
# ncu capture of this build's kernel (the same source) on the same workload;
# a kernel without an entry reports null.
NCU_TRAFFIC = {}
# The same counters summed over the launches of one decode step (workload ->
# bytes), from an ncu capture of this build's kernels (dram__bytes_read.sum +
# dram__bytes_write.sum of every launch in the "decode/" range, one step of
# 51 launches); a workload without a capture of the current kernels reports null.
# (The last batch-1 captures predate the f16 cluster broadcast of the fused
# attention's merged heads, so no workload has one.)
NCU_STEP_TRAFFIC = {}


def decode_roofline(job, hbm_peak):
    """The dominant kernel of a decode step: one step run through
    ember_decode_step_traced (eager, one kernel at a time, CUDA events around
    every launch on the launching stream), kernels grouped by family; the
    family with the most device time gets achieved = its algorithmic bytes
    per launch / its mean launch time."""
    m, kv, s = job.model, job.kv, job.stream
    ctx = job.P + job.S + 1          # keys a sequence holds after the traced step
    trace = m.decode_step_traced(kv, job.seqs, job.cur, None, argmax=job.cur, stream=s)
    fam = {}
    for name, us in trace:
        f = fam.setdefault(_family(name), {"us": 0.0, "n": 0, "name": name})
        f["us"] += us
        f["n"] += 1
    total = sum(f["us"] for f in fam.values())
    top = max(fam, key=lambda k: fam[k]["us"])
    nbytes = decode_family_bytes(job.wl.model, job.B, ctx, bool(job.wl.weights_q8)).get(top)
    t = fam[top]
    avg_us = t["us"] / t["n"]
    out = {"kernel": t["name"], "bound": "hbm", "unit": "GB/s", "peak": hbm_peak,
           "launches_per_step": t["n"], "avg_launch_us": round(avg_us, 2),
           "share_of_step": round(t["us"] / total, 4),
           "timing": "one decode step via ember_decode_step_traced: launches serialised (a one-off graph), "
                     "CUDA events on the launching stream",
           "traffic": NCU_TRAFFIC.get((job.wl.key, t["name"])),
           "step_launches": {k: {"n": v["n"], "us": round(v["us"], 1)} for k, v in
                             sorted(fam.items(), key=lambda kv_: -kv_[1]["us"])}}
    if nbytes is None:
        out.update({"achieved": None, "frac": None, "bytes_per_launch": None})
    else:
        per = nbytes / t["n"]
        gbs = per / (avg_us * 1e-6) / 1e9
        out.update({"achieved": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
                    "bytes_per_launch": int(per)})
    return out


def decode_step_kernels(job) -> str:
    L = job.wl.model.layers
    if job.wl.weights_q8:
        return (f"{L} x (k_gemv q8_0 qkv / o_proj / gate-up / down, k_attn_decode*) + k_gemv LM head, "
                "argmax fused")
    if job.B == 1:
        return f"{L} x (k_fused_attn, k_fused_mlp*) + k_gemv LM head, argmax fused"
    return f"{L} x (k_gemm_tc projections, k_attn_decode_mma, k_rmsnorm) + k_gemm_tc LM head"


def gemv_roofline(stream, hbm_peak, n_launch=30):
    """Live CUDA-event timing of the split GEMV (the decode projections'
    kernel) on the LM-head shape of the workload, alone, inputs > L2."""
    import ctypes
    import torch
    from gqa_transformer_decode_gb300 import ember as E
    N, K = synth.QWEN25_05B.vocab, synth.QWEN25_05B.hidden
    W = (torch.randn(N, K, device="cuda") * 0.02).to(torch.bfloat16).view(torch.int16)
    x = torch.randn(K, device="cuda")
    y = torch.empty(N, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    sp = ctypes.c_void_p(stream.cuda_stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_launch)]
    with torch.cuda.stream(stream):
        for _ in range(5):
            E.check(E.ember_gemv_bf16(P(W), N, K, P(x), 1, P(y), sp), "gemv")
        for a, b in evs:
            a.record(stream)
            E.check(E.ember_gemv_bf16(P(W), N, K, P(x), 1, P(y), sp), "gemv")
            b.record(stream)
    stream.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    nbytes = N * K * 2 + K * 4 + N * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "k_gemv (split GEMV, LM-head shape 151936x896, nb=1, alone)",
            "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(gbs / hbm_peak, 4), "traffic": None, "bytes_per_launch": nbytes,
            "avg_launch_us": round(ms * 1e3, 2)}


def time_jobs(job, n_jobs, world, local):
    """n_jobs jobs with CUDA events around each on the launching stream, the
    clocks sampled meanwhile; -> (job_ms, prefill_ms, decode_ms, wall_s,
    clocks, kernel launches)."""
    import torch
    from gqa_transformer_decode_gb300 import ember as E
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(n_jobs)]
    barrier(world)
    torch.cuda.synchronize()
    launches0 = E.ember_kernel_launches()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(n_jobs):
            job.run(ev=evs[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    launches = E.ember_kernel_launches() - launches0
    barrier(world)
    return ([a.elapsed_time(c) for a, b, c in evs], [a.elapsed_time(b) for a, b, c in evs],
            [b.elapsed_time(c) for a, b, c in evs], wall, clk.summary(), launches)


def measure(wl, weights, args, stream, n_jobs, world, local, pk, headline):
    """One workload's record: warm-up, n_jobs timed jobs (median), rooflines,
    end to end (headline only), CPU oracle baseline (rank 0, N = 1)."""
    import torch
    hbm_peak, bf16_peak, bf16_sus, peak_src = pk
    encoder = wl.model.causal == 0
    job = EncodeJob(wl, weights, stream) if encoder else DecodeJob(wl, weights, stream)
    for _ in range(args.warmup):   # graph capture happens on the first decode call
        job.run()
    assert job.model.sync_status(stream) == 0
    job_ms, pre_ms, dec_ms, wall, clocks, launches = time_jobs(job, n_jobs, world, local)
    st = job.model.sync_status(stream)
    assert st == 0, f"device status {st}"
    med_job_s = max_over_ranks(statistics.median(job_ms) / 1e3, world)
    value = job.tokens_per_job() * world / med_job_s
    rec = {"workload": wl.key, "value": round(value, 2), "unit": "tok/s",
           "jobs_timed": n_jobs, "ms_per_step": round(med_job_s * 1e3, 3)}
    if encoder:
        enc_s = statistics.median(dec_ms) * 1e-3
        tf = job.flops_per_job() / enc_s / 1e12
        rec["encode_tflops"] = round(tf, 1)
        # the whole encode job is a chain of tensor-core GEMMs and attention
        rec["roofline"] = {"kernel": "encode job (all launches)", "bound": "tensor",
                           "unit": "TFLOP/s", "achieved": round(tf, 1), "peak": bf16_peak,
                           "frac": round(tf / bf16_peak, 4), "traffic": None,
                           "flops_per_job": job.flops_per_job(),
                           "timing": "median of CUDA events around each timed job"}
    else:
        step_s = statistics.median(dec_ms) * 1e-3 / wl.steps
        ctx_mid = wl.prompt + wl.steps // 2
        step_bytes = job.bytes_per_decode_step(ctx_mid)
        step_gbs = step_bytes / step_s / 1e9
        rec["decode_tok_s"] = round(wl.batch / step_s, 2)
        rec["decode_step_us"] = round(step_s * 1e6, 2)
        rec["step_hbm"] = {"bytes_per_step": step_bytes, "achieved": round(step_gbs, 1),
                           "peak": hbm_peak, "unit": "GB/s", "frac": round(step_gbs / hbm_peak, 4),
                           "peak_source": peak_src}
        if job.prefill_in_job:
            pre_s = statistics.median(pre_ms) * 1e-3
            rec["prefill_tok_s"] = round(wl.prompt / pre_s, 1)
            ptf = job.prefill_flops() / pre_s / 1e12
            rec["prefill_roofline"] = {"kernel": f"{wl.prompt}-token prefill (all launches)",
                                       "bound": "tensor", "unit": "TFLOP/s",
                                       "achieved": round(ptf, 1), "peak": bf16_peak,
                                       "frac": round(ptf / bf16_peak, 4),
                                       "flops": job.prefill_flops(), "traffic": None}
        # The unit the step launches is one CUDA graph: the layers' kernels are
        # chained with programmatic launch, each prefetching its weights while
        # its predecessor computes, so a kernel's own serialised time is not
        # its cost in the step.  The roofline is that of the graph launch; the
        # per-kernel breakdown of a serialised step follows it.
        rec["roofline"] = {"kernel": "decode step: one CUDA graph launch (%s)" % decode_step_kernels(job),
                           "bound": "hbm", "unit": "GB/s", "achieved": round(step_gbs, 1),
                           "peak": hbm_peak, "frac": round(step_gbs / hbm_peak, 4),
                           "bytes_per_launch": step_bytes, "avg_launch_us": round(step_s * 1e6, 2),
                           "traffic": NCU_STEP_TRAFFIC.get(wl.key),
                           "timing": "median over the timed jobs of CUDA events on the launching stream "
                                     "around the decode steps, divided by the steps"}
        rec["kernel_breakdown"] = decode_roofline(job, hbm_peak)
        assert job.model.sync_status(stream) == 0
    rec["clocks"] = clocks
    rec["gpu_launches"] = launches
    rec["wall_s"] = round(wall, 3)
    if headline and job.prefill_in_job:
        # end to end through the C ABI with host buffers (prompt in, last tokens out)
        host_ids, host_out = job.prepare_e2e()
        e2e_ms = []
        for i in range(max(1, min(n_jobs, 5))):
            barrier(world)
            torch.cuda.synchronize()
            t = time.perf_counter()
            job.run(host_ids=host_ids, host_out=host_out)
            stream.synchronize()
            _ = host_out.numpy().copy()
            e2e_ms.append((time.perf_counter() - t) * 1e3)
        e2e_s = max_over_ranks(statistics.median(e2e_ms) / 1e3, world)
        rec["e2e"] = {"value": round(job.tokens_per_job() * world / e2e_s, 2), "unit": "tok/s",
                      "h2d_bytes_per_step": int(host_ids.numel() * 4),
                      "d2h_bytes_per_step": int(host_out.numel() * 4)}
    rank = dist_env()[0]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(wl, weights, job)
    return rec, job


SUB_WORKLOADS = ("llama-3.2-1b", "qwen2.5-0.5b-b64", "qwen3-encoder", "qwen2.5-0.5b-q8_0")
SUB_JOBS = {"llama-3.2-1b": 3, "qwen2.5-0.5b-b64": 5, "qwen3-encoder": 10, "qwen2.5-0.5b-q8_0": 5}


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if local >= torch.cuda.device_count():
        raise SystemExit(f"rank {rank}: no GPU {local} (this node has {torch.cuda.device_count()})")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    wl = synth.WORKLOADS[args.workload]
    if args.decode_steps is not None:
        import dataclasses
        wl = dataclasses.replace(wl, steps=args.decode_steps)
    pk = peaks()
    hbm_peak, bf16_peak, bf16_sus, peak_src = pk
    stream = torch.cuda.Stream()
    weights = synth.weights_bf16(wl.model)
    rec, job = measure(wl, weights, args, stream, args.steps, world, local, pk, headline=True)
    del job, weights
    gemv_alone = gemv_roofline(stream, hbm_peak)
    out = {
        "metric": METRIC, "value": rec["value"], "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16*f16+f32 (bf16 weights and KV cache; f16 tensor-core operands, f32 accumulation)",
        "data": "synthetic (seeded random bf16 weights N(0,0.02), norms 1+N(0,0.1); uniform ids)",
        "config": {"workload": wl.key, "model_shape": wl.model.name, "batch": wl.batch,
                   "prompt": wl.prompt, "decode_steps": wl.steps,
                   "step": ("one job: prefill + greedy decode" if wl.batch == 1 or
                            wl.model.causal == 0 else "one job: greedy decode of the prefilled batch"),
                   "value": "tokens per job / median job time (prefill included when in the job)",
                   "l2": "weights 2x-20x larger than the 129 MB L2; no flush",
                   "parallelism": f"replicas x{world}"},
    }
    for k in ("decode_tok_s", "decode_step_us", "prefill_tok_s", "encode_tflops", "step_hbm",
              "prefill_roofline", "roofline", "kernel_breakdown", "e2e", "gpu_launches", "clocks", "wall_s",
              "cpu_baseline"):
        if k in rec:
            out[k] = rec[k]
    out["lm_head_gemv_alone"] = gemv_alone
    if not args.headline_only and args.workload == "qwen2.5-0.5b" and args.decode_steps is None:
        out["workloads"] = {}
        for key in SUB_WORKLOADS:
            swl = synth.WORKLOADS[key]
            w = synth.weights_bf16(swl.model)
            sub, job = measure(swl, w, args, stream, SUB_JOBS[key], world, local, pk,
                               headline=False)
            del job, w
            torch.cuda.empty_cache()
            out["workloads"][key] = sub
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ CPU oracle --
PREFILL_SAMPLE = 128     # oracle prefill tokens timed per sample (per-token rate)
ENC_SAMPLE = 256         # encoder tokens of one sequence timed per sample


def oracle_sample(wl: synth.Workload, weights, job=None, steps: int = 4):
    """The oracle on the host cores on a bounded sample of one workload; the
    oracle's model construction (bf16 -> f32 decode of the weights) is not
    timed.  Returns (job seconds extrapolated to the whole workload job,
    threads, what the sample was)."""
    from oracle import oracle as O
    m = wl.model
    if wl.weights_q8:   # the values a q8_0 model computes with (not timed)
        weights = O.q8_0_layer_weights(weights, m.layers)
    om = O.OracleModel(m, weights)
    if m.causal == 0:   # encoder: one sequence's first ENC_SAMPLE tokens
        T = min(wl.prompt, ENC_SAMPLE)
        ids = synth.prompt_ids(m, T)
        t = time.perf_counter()
        om.forward_full(ids, logits=False, cls=True)
        per_tok = (time.perf_counter() - t) / T
        return (per_tok * wl.batch * wl.prompt, O.num_threads(),
                f"one sequence's first {T} of {wl.prompt} tokens, per token, extrapolated to "
                f"{wl.batch} x {wl.prompt} (attention over fewer keys: an upper bound on the rate)")
    if wl.batch > 1 and job is not None:
        # one decode step of sequence 0 started from the GPU's cache of
        # wl.prompt rows (decoded exactly), extrapolated to batch x steps
        K, V = job.kv.tensors()
        cache = om.new_cache(wl.prompt + 1, kv_bf16=True)
        cache.load(K[0][:, :, :wl.prompt].cpu().numpy(), V[0][:, :, :wl.prompt].cpu().numpy(),
                   wl.prompt)
        tok = np.array([int(job.cur0[0].item())], dtype=np.int32)
        t = time.perf_counter()
        om.forward_cached(cache, tok)
        per = time.perf_counter() - t
        return (per * wl.batch * wl.steps, O.num_threads(),
                f"one decode step of one sequence at {wl.prompt} keys (from the GPU's cache), "
                f"extrapolated to {wl.batch} sequences x {wl.steps} steps")
    n = min(wl.prompt, PREFILL_SAMPLE)
    prompt = synth.prompt_ids(m, wl.prompt)[:n]
    cache = om.new_cache(n + steps + 1, kv_bf16=True)
    t = time.perf_counter()
    rc, _, lg = om.forward_cached(cache, prompt)
    pre = time.perf_counter() - t
    tok = np.array([O.argmax(lg)], dtype=np.int32)
    t = time.perf_counter()
    for _ in range(steps):
        rc, _, lg = om.forward_cached(cache, tok)
        tok = np.array([O.argmax(lg)], dtype=np.int32)
    per = (time.perf_counter() - t) / max(1, steps)
    job_s = pre / n * wl.prompt + wl.steps * per
    return (job_s, O.num_threads(),
            f"prefill of the first {n} prompt tokens (per token, x{wl.prompt}) + {steps} decode "
            f"steps of one sequence, extrapolated to the {wl.steps}-step job")


def cpu_baseline(wl, weights, job=None):
    job_s, thr, what = oracle_sample(wl, weights, job)
    tokens = wl.batch * (wl.prompt if wl.model.causal == 0 else wl.steps)
    return {"value": round(tokens / job_s, 4), "unit": "tok/s", "cores": thr, "kind": "oracle",
            "sample": what, "job_s": round(job_s, 3)}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    weights = synth.weights_bf16(wl.model)
    if wl.batch > 1:
        raise SystemExit("--impl reference times batch-1 and encoder workloads "
                         "(batch 64 starts from a GPU-prefilled cache)")
    vals, thr, what = [], 0, ""
    for i in range(args.warmup + args.steps):
        job_s, thr, what = oracle_sample(wl, weights, steps=2)
        if i >= args.warmup:
            vals.append(job_s)
    job_s = statistics.median(vals)
    tokens = wl.batch * (wl.prompt if wl.model.causal == 0 else wl.steps)
    value = tokens / job_s
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(job_s * 1e3, 1), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.key, "model_shape": wl.model.name, "batch": wl.batch,
                      "prompt": wl.prompt, "decode_steps": wl.steps},
           "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": thr,
                            "kind": "oracle", "sample": "each step: " + what},
           "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def spawn_replicas(n: int) -> int:
    """Re-run this script under torch.distributed.run with n processes."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__),
           *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ember", choices=["ember", "reference"])
    ap.add_argument("--workload", default="qwen2.5-0.5b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the headline workload (no 'workloads' records)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="override the workload's decode steps per job (short profiling runs)")
    ap.add_argument("--gemv-only", action="store_true",
                    help="only the standalone GEMV roofline launches (for counter captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_replicas(args.gpus))
    if args.impl == "reference":
        run_reference(args)
    elif args.gemv_only:
        import torch
        hbm_peak = peaks()[0]
        print(json.dumps(gemv_roofline(torch.cuda.Stream(), hbm_peak, n_launch=args.steps)))
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
