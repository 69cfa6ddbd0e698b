// common.cuh -- device helpers shared by the ember kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ember.h"

namespace ember {

constexpr unsigned FULL_MASK = 0xffffffffu;

// ---- status word ---------------------------------------------------------------
// First error wins; the host reads and clears it in ember_sync_status().
__device__ __forceinline__ void raise_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---- bf16 <-> f32 ------------------------------------------------------------------
// A bf16 value is the high half of an f32 (ember reference_forward.py,
// load_safetensors): widening is a 16-bit shift.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// f32 -> bf16, round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
}

__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
    f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
    f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

// f16 side: the layer weights and the activations fed to the tensor-core
// GEMMs are IEEE half (11 significant bits; the bf16 weights convert exactly
// above 6.1e-5 in magnitude, below it to the f16 subnormal grid, <= 3e-8 off).
__device__ __forceinline__ uint16_t f32_to_f16(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// 2^e as an f32 (e in [-126, 127]): a layer matrix whose bf16 values exceed
// the f16 range is stored as f16(W * 2^-e) and its products multiplied back
// by 2^e, an exact rescaling (e = 0 for every matrix within range).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Activations rounded to f16 must lie within its range: `bad` records a value
// beyond +-65504 (or NaN) so the kernel can raise EMBER_ERR_RANGE.
constexpr float F16_MAX = 65504.f;
__device__ __forceinline__ bool f16_out_of_range(float v) { return !(fabsf(v) <= F16_MAX); }
__device__ __forceinline__ uint32_t pack_f16x2_chk(float lo, float hi, bool& bad) {
    bad |= f16_out_of_range(lo) | f16_out_of_range(hi);
    return pack_f16x2(lo, hi);
}
__device__ __forceinline__ uint16_t f32_to_f16_chk(float f, bool& bad) {
    bad |= f16_out_of_range(f);
    return f32_to_f16(f);
}
__device__ __forceinline__ void unpack8_f16(const uint4& w, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
// bf16 or f16 weights (F16 is a compile-time choice of the caller)
template <bool F16>
__device__ __forceinline__ void unpack8w(const uint4& w, float* f) {
    if (F16) unpack8_f16(w, f);
    else unpack8(w, f);
}

// Streaming 128-bit load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 2^x by the hardware approximation (relative error ~2^-22; ftz)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- reductions --------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, o));
    return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024); `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
    if (warp == 0) t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
    __syncthreads();
    float r = red[0];
    __syncthreads();
    return r;
}

// ---- greedy argmax key -----------------------------------------------------------------
// A 64-bit key whose unsigned maximum is the first index of the largest value:
// high word = the value mapped to an order-preserving unsigned (NaN above
// everything, -0 == +0), low word = ~index so equal values prefer the lowest
// index (np.argmax semantics, ember reference_forward.py main()).
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
    uint32_t u = __float_as_uint(v);
    if (v != v) {
        u = 0xffffffffu;
    } else {
        if (u == 0x80000000u) u = 0u;
        u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - idx);
}
__device__ __forceinline__ int32_t argmax_key_index(unsigned long long k) {
    return (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
}

// ---- RoPE (rotate-half) ---------------------------------------------------------------
// Pair i rotates (x_i, x_{i+D/2}) by the angle of row `pos` of the f32 tables
// (ember reference_forward.py rope(); PII-Tracer apply_rope()).  Every product
// and sum is rounded separately (no FMA contraction), so the result is the
// exact f32 evaluation of  x0*c - x1*s  and  x1*c + x0*s.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& r0,
                                          float& r1) {
    r0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    r1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
}

// ---- programmatic dependent launch -------------------------------------------------------
// pdl_trigger: allow the next kernel in the stream to start its prologue;
// pdl_wait: block until the previous kernel has completed and its writes are
// visible.  Both are no-ops when the kernel was launched without the
// programmatic-serialization attribute.  Every read of data produced by an
// earlier kernel comes after pdl_wait().
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- device side of the model ------------------------------------------------------------
enum EpiMode : int {
    EPI_STORE = 0,   // out_f32[m][n] = acc (+ bias[n])
    EPI_RESID = 1,   // out_f32[m][n] += acc            (residual add)
    EPI_SWIGLU = 2,  // rows 2i / 2i+1 = gate_i / up_i -> act[m][i] = silu(gate)*up
    EPI_ARGMAX = 3,  // logits (optional store) + greedy argmax key
};

}  // namespace ember
