// decode_attn_mma.cu -- split-KV decode attention on the warp tensor cores
// (head_dim 64 / 128, up to 16 query heads per kv head).
//
// One CTA = (token b, kv head g, key split); 4 warps.  The G query heads of
// the group are the 16-row A operand (rows >= G are zero): per 64-key tile,
// warp w takes keys 16w..16w+15 and computes S = Q K^T with mma.m16n8k16
// (f16 operands, f32 accumulators; K fragments by ldmatrix from a swizzled
// shared tile), keeps an online softmax per row in the base-2 domain, packs P
// to f16 in registers as the A operand of O += P V (V fragments by
// ldmatrix.trans).  The four warps' states are merged in shared memory; the
// split partials are merged by the last CTA of the (token, kv head) as in
// the SIMT kernel.  K/V tiles are loaded one tile ahead into registers and
// converted from the bf16 cache to f16 when stored.  The prologue (optional
// q/k RMSNorm, RoPE, the new K/V row written as bf16 by the split holding the
// position) is that of grouped-query attention in the Llama / Qwen2 decoder.
#include "common.cuh"
#include "kernels.h"

namespace ember {

namespace {

constexpr int AM_THREADS = 128;
constexpr int AM_TK = 64;               // keys per tile, 16 per warp
constexpr int AM_MIN_CHUNK = 64;        // keys per split at least
constexpr int AM_MAX_SPLITS = 32;       // partial buffer layout (same as the SIMT kernel)

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// c += a (16x16, f16) * b (16x8, f16), f32 accumulators
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] f16 tile whose
// chunks are XOR-swizzled by (r & 7): ldmatrix reads 8 rows at one logical
// chunk without bank conflicts.
template <int D>
__device__ __forceinline__ int tile_off(int r, int c) {
    return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

// 8 bf16 (one uint4) -> 8 f16 (one uint4)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& u) {
    uint4 o;
    o.x = pack_f16x2(bf16_lo(u.x), bf16_hi(u.x));
    o.y = pack_f16x2(bf16_lo(u.y), bf16_hi(u.y));
    o.z = pack_f16x2(bf16_lo(u.z), bf16_hi(u.z));
    o.w = pack_f16x2(bf16_lo(u.w), bf16_hi(u.w));
    return o;
}

template <int D>
struct AmSmem {
    static constexpr int TILE = AM_TK * D * 2;          // one f16 K (or V) tile
    static constexpr int Q = 0;                          // [16][D] f16, swizzled
    static constexpr int K0 = 16 * D * 2;                // 2 stages of K then V
    static constexpr int V0 = K0 + 2 * TILE;
    static constexpr int END = V0 + 2 * TILE;
    // after the key loop the K/V area holds the warps' states [4][16][D + 2] f32
    static_assert(4 * 16 * (D + 2) * 4 <= 4 * TILE, "merge scratch");
    static constexpr int TOTAL = END + 1024;
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(AM_THREADS) k_attn_decode_mma(AttnDecodeArgs a) {
    constexpr int H2 = D / 2, C8 = D / 8, NT = D / 8, KS = D / 16;
    constexpr int PER = AM_TK * C8 / AM_THREADS;     // 16-byte K (and V) chunks per thread and tile
    using L = AmSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ float s_q[16][D];
    __shared__ float s_kv[2][D];
    __shared__ int s_last;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = a.NH / a.NKV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_trigger();
    pdl_wait();
    if (!__ldcg(a.tok_ok + b)) return;   // the embed kernel flagged this token
    const int pos = __ldcg(a.positions + b);
    const int seq = a.seqs[b];
    const int n_keys = pos + 1;
    int per = (n_keys + gridDim.x - 1) / gridDim.x;
    per = per < AM_MIN_CHUNK ? AM_MIN_CHUNK : per;
    const int S = (n_keys + per - 1) / per;          // active splits
    if (split >= S) return;
    const int lo = split * per;
    const int hi = min(n_keys, lo + per);
    const float* qkv = a.qkv + (size_t)b * a.ld_qkv;
    const float* cs = a.cos_t + (size_t)pos * H2;
    const float* sn = a.sin_t + (size_t)pos * H2;
    const size_t head_off = (((size_t)seq * a.L + a.layer) * a.NKV + g) * (size_t)a.max_len * D;
    uint16_t* kc = a.kc + head_off;
    uint16_t* vc = a.vc + head_off;
    const float qscale = 1.4426950408889634f * rsqrtf((float)D);   // scores in base 2

    // ---- q of the G heads (rows >= G zero), the new k / v; q/k norm; RoPE ----
    for (int e = tid; e < 16 * D; e += AM_THREADS) {
        const int h = e / D;
        s_q[h][e % D] = h < G ? __ldcg(qkv + (size_t)g * G * D + e) : 0.f;
    }
    for (int e = tid; e < 2 * D; e += AM_THREADS) {
        const int which = e / D, d = e % D;   // 0: k, 1: v
        s_kv[which][d] = __ldcg(qkv + (size_t)a.NH * D + (size_t)which * a.NKV * D + (size_t)g * D + d);
    }
    __syncthreads();
    if (a.q_norm) {
        for (int h = warp; h < G + 1; h += AM_THREADS / 32) {
            float* v = h < G ? s_q[h] : s_kv[0];
            const float* w = h < G ? a.q_norm : a.k_norm;
            float ss = 0.f;
            for (int d = lane; d < D; d += 32) ss += v[d] * v[d];
            ss = warp_sum(ss);
            const float ri = rsqrtf(ss / (float)D + a.eps);
            __syncwarp();
            for (int d = lane; d < D; d += 32) v[d] = v[d] * ri * w[d];
        }
        __syncthreads();
    }
    for (int e = tid; e < (G + 1) * H2; e += AM_THREADS) {
        const int h = e / H2, i = e % H2;
        float* v = h < G ? s_q[h] : s_kv[0];
        float r0, r1;
        rope_pair(v[i], v[i + H2], cs[i], sn[i], r0, r1);
        if (h < G) {
            v[i] = r0 * qscale;
            v[i + H2] = r1 * qscale;
        } else {
            v[i] = r0;
            v[i + H2] = r1;
        }
    }
    __syncthreads();
    if (pos >= lo && pos < hi) {   // the split holding pos writes the new K/V row (bf16)
        for (int d = tid; d < D; d += AM_THREADS) {
            kc[(size_t)pos * D + d] = f32_to_bf16(s_kv[0][d]);
            vc[(size_t)pos * D + d] = f32_to_bf16(s_kv[1][d]);
        }
    }
    for (int e = tid; e < 16 * C8; e += AM_THREADS) {   // q as the f16 A tile
        const int r = e / C8, c = e % C8;
        const float* q = &s_q[r][c * 8];
        *reinterpret_cast<uint4*>(sm + L::Q + tile_off<D>(r, c)) =
            make_uint4(pack_f16x2(q[0], q[1]), pack_f16x2(q[2], q[3]), pack_f16x2(q[4], q[5]),
                       pack_f16x2(q[6], q[7]));
    }
    __syncthreads();   // also orders the K/V row write before the tile loads below
    uint32_t qa[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        const int mi = lane >> 3;
        const int r = (mi & 1) * 8 + (lane & 7), c = 2 * kk + (mi >> 1);
        ldsm4(sa(sm + L::Q + tile_off<D>(r, c)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    // ---- keys [lo, hi) in tiles of 64, one tile ahead in registers ----
    uint4 kr[PER], vr[PER];
    auto load_tile = [&](int t0) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = tid + u * AM_THREADS;
            const int j = e / C8, c = e % C8;
            if (t0 + j < hi) {
                kr[u] = __ldcg(reinterpret_cast<const uint4*>(kc + (size_t)(t0 + j) * D + c * 8));
                vr[u] = __ldcg(reinterpret_cast<const uint4*>(vc + (size_t)(t0 + j) * D + c * 8));
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    auto store_tile = [&](int st) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = tid + u * AM_THREADS;
            const int j = e / C8, c = e % C8;
            *reinterpret_cast<uint4*>(sm + L::K0 + st * L::TILE + tile_off<D>(j, c)) = bf16x8_to_f16x8(kr[u]);
            *reinterpret_cast<uint4*>(sm + L::V0 + st * L::TILE + tile_off<D>(j, c)) = bf16x8_to_f16x8(vr[u]);
        }
    };
    float o[NT][4];
#pragma unroll
    for (int dn = 0; dn < NT; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows lane/4 and lane/4 + 8
    const int g4 = lane >> 2, q4 = lane & 3;
    int stg = 0;
    if (lo < hi) load_tile(lo);
    for (int t0 = lo; t0 < hi; t0 += AM_TK, stg ^= 1) {
        store_tile(stg);
        __syncthreads();
        if (t0 + AM_TK < hi) load_tile(t0 + AM_TK);
        const int kw = t0 + warp * 16;   // this warp's first key (valid when < hi)
        if (kw < hi) {
            const uint8_t* kt = sm + L::K0 + stg * L::TILE;
            const uint8_t* vt = sm + L::V0 + stg * L::TILE;
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {   // S = Q K^T over the warp's 16 keys
                const int mi = lane >> 3;
                const int row = warp * 16 + (mi >> 1) * 8 + (lane & 7), c = 2 * kk + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm4(sa(kt + tile_off<D>(row, c)), b0, b1, b2, b3);
                mma16816(s[0], qa[kk], b0, b1);
                mma16816(s[1], qa[kk], b2, b3);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int key = kw + nt * 8 + 2 * q4 + (i & 1);
                    if (key >= hi) s[nt][i] = -INFINITY;
                    if (i < 2) mx0 = fmaxf(mx0, s[nt][i]);
                    else mx1 = fmaxf(mx1, s[nt][i]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: key kw is valid
            const float sc0 = exp2f(m0 - mn0), sc1 = exp2f(m1 - mn1);   // 0 while m = -inf
            float p[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) p[nt][i] = exp2f(s[nt][i] - (i < 2 ? mn0 : mn1));
            l0 = l0 * sc0 + ((p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
            l1 = l1 * sc1 + ((p[0][2] + p[0][3]) + (p[1][2] + p[1][3]));
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int dn = 0; dn < NT; ++dn) {
                o[dn][0] *= sc0; o[dn][1] *= sc0;
                o[dn][2] *= sc1; o[dn][3] *= sc1;
            }
            const uint32_t pa[4] = {pack_f16x2(p[0][0], p[0][1]), pack_f16x2(p[0][2], p[0][3]),
                                    pack_f16x2(p[1][0], p[1][1]), pack_f16x2(p[1][2], p[1][3])};
#pragma unroll
            for (int dn = 0; dn < NT; dn += 2) {   // O += P V
                const int mi = lane >> 3;
                const int row = warp * 16 + (mi & 1) * 8 + (lane & 7), c = dn + (mi >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm4t(sa(vt + tile_off<D>(row, c)), r0, r1, r2, r3);
                mma16816(o[dn], pa, r0, r1);
                mma16816(o[dn + 1], pa, r2, r3);
            }
        }
        __syncthreads();
    }

    // ---- merge the four warps: [4][16][D + 2] f32 = (m, l, O) per warp and row ----
    l0 += __shfl_xor_sync(FULL_MASK, l0, 1);
    l0 += __shfl_xor_sync(FULL_MASK, l0, 2);
    l1 += __shfl_xor_sync(FULL_MASK, l1, 1);
    l1 += __shfl_xor_sync(FULL_MASK, l1, 2);
    float* ws = reinterpret_cast<float*>(sm + L::K0);   // the K/V tiles are no longer read
    {
        float* w0 = ws + ((size_t)warp * 16 + g4) * (D + 2);
        float* w1 = ws + ((size_t)warp * 16 + g4 + 8) * (D + 2);
        if (q4 == 0) {
            w0[0] = m0; w0[1] = l0;
            w1[0] = m1; w1[1] = l1;
        }
#pragma unroll
        for (int dn = 0; dn < NT; ++dn) {
            const int d = dn * 8 + 2 * q4;
            w0[2 + d] = o[dn][0]; w0[3 + d] = o[dn][1];
            w1[2 + d] = o[dn][2]; w1[3 + d] = o[dn][3];
        }
    }
    __syncthreads();
    const size_t out0 = (size_t)b * a.NH * D + (size_t)(g * G) * D;
    float* part = a.part + ((((size_t)b * a.NKV + g) * AM_MAX_SPLITS + split) * G) * (D + 2);
    for (int e = tid; e < G * (D + 2); e += AM_THREADS) {
        const int h = e / (D + 2), k = e % (D + 2);   // k: 0 = m, 1 = l, 2.. = O
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float* st = ws + ((size_t)w * 16 + h) * (D + 2);
            if (st[1] > 0.f) M = fmaxf(M, st[0]);
        }
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float* st = ws + ((size_t)w * 16 + h) * (D + 2);
            if (st[1] > 0.f) v = fmaf(k == 0 ? 0.f : st[k], exp2f(st[0] - M), v);
        }
        if (k == 0) v = M;
        if (S == 1) {   // a single split is already the answer
            if (k >= 2) {
                float Ls = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float* st = ws + ((size_t)w * 16 + h) * (D + 2);
                    if (st[1] > 0.f) Ls = fmaf(st[1], exp2f(st[0] - M), Ls);
                }
                const float out = Ls > 0.f ? v / Ls : 0.f;
                if (a.att_b) a.att_b[out0 + (size_t)h * D + k - 2] = f32_to_f16(out);
                else a.att[out0 + (size_t)h * D + k - 2] = out;
            }
        } else {
            part[e] = v;
        }
    }
    if (S == 1) return;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned done = atomicAdd(&a.counters[b * a.NKV + g], 1u);
        s_last = (done == (unsigned)(S - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last split: merge the S partials ----
    const float* pb = a.part + (((size_t)b * a.NKV + g) * AM_MAX_SPLITS) * G * (D + 2);
    float* s_pm = ws;                                  // [S][G] maxima -> weights
    float* s_pl = ws + AM_MAX_SPLITS * 16;             // [S][G] sums
    float* s_inv = ws + 2 * AM_MAX_SPLITS * 16;        // [G]
    for (int e = tid; e < S * G; e += AM_THREADS) {
        const float* ps = pb + (size_t)e * (D + 2);
        s_pm[e] = __ldcg(ps);
        s_pl[e] = __ldcg(ps + 1);
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < S; ++s2)
            if (s_pl[s2 * G + tid] > 0.f) M = fmaxf(M, s_pm[s2 * G + tid]);
        float Ls = 0.f;
        for (int s2 = 0; s2 < S; ++s2) {
            const float l = s_pl[s2 * G + tid];
            const float f = l > 0.f ? exp2f(s_pm[s2 * G + tid] - M) : 0.f;
            s_pm[s2 * G + tid] = f;
            Ls += l * f;
        }
        s_inv[tid] = Ls > 0.f ? 1.f / Ls : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += AM_THREADS) {
        const int h = e / D, d = e % D;
        float O = 0.f;
#pragma unroll 4
        for (int s2 = 0; s2 < S; ++s2)
            O = fmaf(__ldcg(pb + ((size_t)s2 * G + h) * (D + 2) + 2 + d), s_pm[s2 * G + h], O);
        O *= s_inv[h];
        if (a.att_b) a.att_b[out0 + e] = f32_to_f16(O);
        else a.att[out0 + e] = O;
    }
    if (tid == 0) a.counters[b * a.NKV + g] = 0u;
}

bool attn_decode_mma_supported(int D, int G) { return (D == 64 || D == 128) && G >= 1 && G <= 16; }

void launch_attn_decode_mma(const AttnDecodeArgs& a, cudaStream_t s) {
    dim3 grid(a.splits < AM_MAX_SPLITS ? a.splits : AM_MAX_SPLITS, a.NKV, a.nb);
    if (a.D == 64) {
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(k_attn_decode_mma<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AmSmem<64>::TOTAL);
            attr = true;
        }
        launch_k(k_attn_decode_mma<64>, grid, dim3(AM_THREADS), AmSmem<64>::TOTAL, s, a);
    } else {
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(k_attn_decode_mma<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AmSmem<128>::TOTAL);
            attr = true;
        }
        launch_k(k_attn_decode_mma<128>, grid, dim3(AM_THREADS), AmSmem<128>::TOTAL, s, a);
    }
}

}  // namespace ember
