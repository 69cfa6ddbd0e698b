// sampler.cu -- the token sampler after the LM head ("ember internals",
// sampler): temperature -> top-k -> top-p (nucleus) -> softmax (uniform for
// a row whose every logit is -inf) -> inverse-CDF draw, one CTA of 1024
// threads per row of logits.
//
// Every selection is exact: the top-k threshold and the nucleus cutoff are
// found by radix selection on the logits' f32 values (an order-preserving
// 32-bit key, 8 bits per pass), and a token survives a stage when its key
// is not below the threshold's -- the pages' "mask what lies below", ties
// kept.  The probability masses that decide the nucleus and the draw are
// exp(x - max) in f32 quantised to 2^-40 and summed as 64-bit integers, so
// the sums are exact and independent of the order the threads add them in:
// the kernel is deterministic, and it departs from exact arithmetic only by
// the f32 exponential and the 2^-41 rounding of each term.
#include "common.cuh"
#include "kernels.h"

#include <climits>

namespace ember {

namespace {

constexpr int SP_THREADS = 1024;
constexpr int SP_PER = 8;                       // contiguous elements per thread in the index-order scan
constexpr int SP_TILE = SP_THREADS * SP_PER;
constexpr float SP_QSCALE = 1099511627776.0f;   // 2^40

// order-preserving map of f32 onto u32: a > b <=> key(a) > key(b) (NaN aside)
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct SampleRow {
    const float* L;
    float t;
    bool scale;
    __device__ __forceinline__ float x(int i) const {   // stage 1: logit / t (IEEE division)
        const float v = __ldg(L + i);
        return scale ? v / t : v;
    }
};

template <typename T>
__device__ __forceinline__ T warp_max_t(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const T w = __shfl_xor_sync(FULL_MASK, v, o);
        v = w > v ? w : v;
    }
    return v;
}

template <typename T>
__device__ __forceinline__ T warp_sum_t(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
    return v;
}

// block-wide max / sum over 1024 threads through s[32]
template <typename T>
__device__ __forceinline__ T block_max_t(T v, T* s) {
    v = warp_max_t(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
    __syncthreads();
    T r = s[0];
    for (int w = 1; w < SP_THREADS / 32; ++w) r = s[w] > r ? s[w] : r;
    return r;
}
template <typename T>
__device__ __forceinline__ T block_sum_t(T v, T* s) {
    v = warp_sum_t(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
    __syncthreads();
    T r = 0;
    for (int w = 0; w < SP_THREADS / 32; ++w) r += s[w];
    return r;
}

// the quantised mass of a survivor: exp(x - m) (uniform when m = -inf) in 2^-40 units
__device__ __forceinline__ unsigned long long qmass(float x, float m) {
    if (m == -INFINITY) return 1ull;
    return __float2ull_rn(expf(x - m) * SP_QSCALE);
}

__global__ void __launch_bounds__(SP_THREADS, 1) k_sample(SampleArgs a) {
    __shared__ unsigned s_cnt[256];
    __shared__ unsigned long long s_mass[256];
    __shared__ unsigned long long s_u64[32];
    __shared__ float s_f32[32];
    __shared__ unsigned s_sel[2];
    __shared__ unsigned long long s_sel64[1];
    const int tid = threadIdx.x;
    const int V = a.V;
    const SampleRow row{a.logits + (size_t)blockIdx.x * a.ldl, a.t, a.t > 0.f};

    // ---- greedy (t <= 0): the first maximal logit, NaN counting as maximal ----
    if (!(a.t > 0.f)) {
        unsigned long long best = 0;
        for (int i = tid; i < V; i += SP_THREADS) {
            const float v = __ldg(row.L + i);
            const uint32_t k = v != v ? 0xFFFFFFFFu : fkey(v);
            const unsigned long long c = ((unsigned long long)k << 32) | (0xFFFFFFFFu - (uint32_t)i);
            best = c > best ? c : best;
        }
        best = block_max_t(best, s_u64);
        if (tid == 0) a.out[blockIdx.x] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFu));
        return;
    }

    // ---- the maximum of x (survives every stage) ----
    float m = -INFINITY;
    for (int i = tid; i < V; i += SP_THREADS) m = fmaxf(m, row.x(i));
    m = block_max_t(m, s_f32);

    // radix selection over the keys of the survivors (key >= lo_key): the
    // largest key c whose "weight" at and above c, plus `above`, first
    // reaches `need` (counts for top-k, masses for top-p)
    auto select = [&](uint32_t lo_key, bool by_mass, unsigned long long need) -> uint32_t {
        uint32_t prefix = 0, pmask = 0;
        unsigned long long above = 0;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int j = tid; j < 256; j += SP_THREADS) {
                s_cnt[j] = 0;
                s_mass[j] = 0;
            }
            __syncthreads();
            for (int i = tid; i < V; i += SP_THREADS) {
                const float x = row.x(i);
                const uint32_t u = fkey(x);
                if (u >= lo_key && (u & pmask) == prefix) {
                    const int bin = (u >> shift) & 255;
                    if (by_mass) atomicAdd(&s_mass[bin], qmass(x, m));
                    else atomicAdd(&s_cnt[bin], 1u);
                }
            }
            __syncthreads();
            if (tid == 0) {
                int bin = 255;
                for (; bin > 0; --bin) {
                    const unsigned long long w = by_mass ? s_mass[bin] : s_cnt[bin];
                    if (above + w >= need) break;
                    above += w;
                }
                s_sel[0] = (unsigned)bin;
                s_sel64[0] = above;
            }
            __syncthreads();
            prefix |= s_sel[0] << shift;
            pmask |= 255u << shift;
            above = s_sel64[0];
            __syncthreads();
        }
        return prefix;
    };

    // ---- stage 2, top-k: the k-th largest x; keys below it are masked ----
    uint32_t lo_key = 0;
    if (a.k > 0 && a.k < V) lo_key = select(0u, false, (unsigned long long)a.k);

    // ---- stage 3, top-p: the largest x whose survivors at and above it
    // carry more than p of the mass (sum of soft > p <=> Q > floor(p * Q1)) ----
    if (a.p > 0.f && a.p < 1.f) {
        unsigned long long q = 0;
        for (int i = tid; i < V; i += SP_THREADS) {
            const float x = row.x(i);
            if (fkey(x) >= lo_key) q += qmass(x, m);
        }
        const unsigned long long Q1 = block_sum_t(q, s_u64);
        const unsigned long long P = (unsigned long long)floor((double)a.p * (double)Q1);
        lo_key = select(lo_key, true, P + 1);
    }

    // ---- stages 4-5: softmax over the survivors and the inverse-CDF draw:
    // the first index whose running mass exceeds r * Q2 ----
    unsigned long long q = 0;
    for (int i = tid; i < V; i += SP_THREADS) {
        const float x = row.x(i);
        if (fkey(x) >= lo_key) q += qmass(x, m);
    }
    const unsigned long long Q2 = block_sum_t(q, s_u64);
    const unsigned long long R = (unsigned long long)floor((double)a.r[blockIdx.x] * (double)Q2);
    __shared__ int s_hit;
    __shared__ unsigned long long s_scan[32];
    if (tid == 0) s_hit = INT_MAX;
    unsigned long long base = 0;
    const int lane = tid & 31, warp = tid >> 5;
    for (int t0 = 0; t0 < V; t0 += SP_TILE) {
        const int i0 = t0 + tid * SP_PER;
        unsigned long long w[SP_PER];
        unsigned long long own = 0;
#pragma unroll
        for (int e = 0; e < SP_PER; ++e) {
            w[e] = 0;
            if (i0 + e < V) {
                const float x = row.x(i0 + e);
                if (fkey(x) >= lo_key) w[e] = qmass(x, m);
            }
            own += w[e];
        }
        // exclusive prefix of the thread totals over the block (warp scan, then the warps)
        unsigned long long incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();
        if (lane == 31) s_scan[warp] = incl;
        __syncthreads();
        unsigned long long wbase = 0, tile = 0;
        for (int v = 0; v < SP_THREADS / 32; ++v) {
            if (v < warp) wbase += s_scan[v];
            tile += s_scan[v];
        }
        unsigned long long run = base + wbase + incl - own;
#pragma unroll
        for (int e = 0; e < SP_PER; ++e) {
            run += w[e];
            if (run > R && w[e] > 0) {
                atomicMin(&s_hit, i0 + e);
                break;
            }
        }
        __syncthreads();
        if (s_hit != INT_MAX) break;
        base += tile;
    }
    if (tid == 0) {
        int tok = s_hit;
        if (tok == INT_MAX) tok = -1;   // r * Q2 at or above the total: fallback below
        s_sel[0] = (unsigned)tok;
    }
    __syncthreads();
    if ((int)s_sel[0] >= 0) {
        if (tid == 0) a.out[blockIdx.x] = (int32_t)s_sel[0];
        return;
    }
    // rounding fallback: the last maximal probability, i.e. the last index holding the maximum
    int last = -1;
    for (int i = tid; i < V; i += SP_THREADS)
        if (row.x(i) == m) last = i;
    last = block_max_t(last, reinterpret_cast<int*>(s_f32));
    if (tid == 0) a.out[blockIdx.x] = last;
}

}  // namespace

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s) {
    return launch_k(k_sample, dim3(a.B), dim3(SP_THREADS), 0, s, a);
}

}  // namespace ember
