// decode_attn_mma.cu -- split-KV decode attention on the warp tensor cores
// (head_dim 64 / 128, up to 16 query heads per kv head).
//
// One CTA = (token b, kv head g, key split); 8 warps.  The G query heads of
// the group are the 16-row A operand (rows >= G are zero): per 128-key tile,
// warp w takes keys 16w..16w+15 and computes S = Q K^T with mma.m16n8k16
// (f16 operands, f32 accumulators; K fragments by ldmatrix from a swizzled
// shared tile), keeps an online softmax per row in the base-2 domain, packs P
// to f16 in registers as the A operand of O += P V (V fragments by
// ldmatrix.trans).  The eight warps' states are merged in shared memory; the
// split partials are merged by the last CTA of the (token, kv head) as in
// the SIMT kernel.  K/V tiles of 128 keys stream through a 2-3 stage ring of
// bulk tensor copies (bf16, 128-byte swizzle) issued as soon as the position
// is known; fragments are converted to f16 in registers.  The prologue (optional
// q/k RMSNorm, RoPE, the new K/V row written as bf16 by the split holding the
// position) is that of grouped-query attention in the Llama / Qwen2 decoder.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "mma_common.cuh"

namespace ember {

namespace {

constexpr int AM_THREADS = 256;
constexpr int AM_WARPS = AM_THREADS / 32;
constexpr int AM_KW = 128 / AM_WARPS;     // keys of a tile per warp (blocks of 16)
constexpr int AM_TK = 128;              // keys per tile (the TMA box height)
constexpr int AM_MIN_CHUNK = 64;        // keys per split at least
constexpr int AM_MAX_SPLITS = 32;       // partial buffer layout (same as the SIMT kernel)
constexpr long long AM_WAIT = 1ll << 31;

__device__ __forceinline__ void mbar_expect_tx_(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                     uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sa_u32(dst)),
        "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(sa_u32(bar))
        : "memory");
}
__device__ __forceinline__ bool am_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = sa_u32(bar);
    uint32_t ok;
    const long long t0 = clock64();
    do {
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(addr), "r"(parity)
            : "memory");
        if (ok) return true;
    } while (clock64() - t0 < AM_WAIT);
    return false;
}

template <int D>
struct AmSmem {
    static constexpr int NS = D == 64 ? 3 : 2;           // ring stages
    static constexpr int TILE = AM_TK * D * 2;           // one bf16 K (or V) tile
    static constexpr int Q = 0;                          // [16][D] f16
    static constexpr int R0 = 4096;                      // ring (1024-aligned)
    static constexpr int BAR = R0 + NS * 2 * TILE;
    static constexpr int END = BAR + 64;
    // after the key loop the ring holds the warps' states [AM_WARPS][16][D + 2] f32
    static_assert(AM_WARPS * 16 * (D + 2) * 4 <= NS * 2 * TILE, "merge scratch");
    static_assert(16 * D * 2 <= R0, "q tile");
    static constexpr int TOTAL = END + 1024;
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(AM_THREADS) k_attn_decode_mma(const __grid_constant__ CUtensorMap k_map,
                                                              const __grid_constant__ CUtensorMap v_map,
                                                              AttnDecodeArgs a) {
    constexpr int H2 = D / 2, C8 = D / 8, NT = D / 8, KS = D / 16, NSUB = D / 64;
    using L = AmSmem<D>;
    constexpr int NS = L::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
    __shared__ float s_q[16][D];
    __shared__ float s_kv[2][D];
    __shared__ float s_cs[D];            // RoPE row of pos: cos | sin
    __shared__ int s_last, s_err;

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = a.NH / a.NKV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // The caller's sequence indices are complete before the step starts, and
    // the barriers are this CTA's own: both before the wait.
    const int seq = a.seqs[b];
    if (tid == 0) {
        s_err = 0;
        for (int st = 0; st < NS; ++st)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa_u32(&full[st])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_trigger();
    pdl_wait();
    const int tok_ok = __ldcg(a.tok_ok + b);
    const int pos = __ldcg(a.positions + b);   // both loads in flight together
    // q of the G heads (rows >= G zero) and the new k / v: independent of the
    // position, so their loads go out with it
    constexpr int QPT = (16 * D + AM_THREADS - 1) / AM_THREADS;
    float qreg[QPT];
    const float* qkv = a.qkv + (size_t)b * a.ld_qkv;
#pragma unroll
    for (int j = 0; j < QPT; ++j) {
        const int e = tid + j * AM_THREADS;
        qreg[j] = (e < 16 * D && e / D < G) ? __ldcg(qkv + (size_t)g * G * D + e) : 0.f;
    }
    const float kvreg = tid < 2 * D ? __ldcg(qkv + (size_t)a.NH * D + (size_t)(tid / D) * a.NKV * D +
                                              (size_t)g * D + tid % D)
                                    : 0.f;
    if (!tok_ok) return;   // the embed kernel flagged this token
    const int n_keys = pos + 1;
    int per = (n_keys + gridDim.x - 1) / gridDim.x;
    per = per < AM_MIN_CHUNK ? AM_MIN_CHUNK : per;
    const int S = (n_keys + per - 1) / per;          // active splits
    if (split >= S) return;
    const int lo = split * per;
    const int hi = min(n_keys, lo + per);
    const int n_tiles = (hi - lo + AM_TK - 1) / AM_TK;
    const int kz = (seq * a.L + a.layer) * a.NKV + g;   // (seq, layer, kv head) plane of the maps
    auto issue = [&](int it) {   // tile it -> stage it % NS
        const int st = it % NS;
        uint8_t* kt = sm + L::R0 + st * 2 * L::TILE;
        mbar_expect_tx_(&full[st], (uint32_t)(2 * L::TILE));
#pragma unroll
        for (int sb = 0; sb < NSUB; ++sb) {
            tma3(kt + sb * AM_TK * 128, &k_map, sb * 64, lo + it * AM_TK, kz, &full[st]);
            tma3(kt + L::TILE + sb * AM_TK * 128, &v_map, sb * 64, lo + it * AM_TK, kz, &full[st]);
        }
    };
    if (tid == 0)
        for (int it = 0; it < NS && it < n_tiles; ++it) issue(it);
    const float* cs = a.cos_t + (size_t)pos * H2;
    const float* sn = a.sin_t + (size_t)pos * H2;
    const size_t head_off = (size_t)kz * a.max_len * D;
    uint16_t* kc = a.kc + head_off;
    uint16_t* vc = a.vc + head_off;
    const float qscale = 1.4426950408889634f * rsqrtf((float)D);   // scores in base 2

    // ---- q of the G heads (rows >= G zero), the new k / v; q/k norm; RoPE ----
#pragma unroll
    for (int j = 0; j < QPT; ++j) {
        const int e = tid + j * AM_THREADS;
        if (e < 16 * D) s_q[e / D][e % D] = qreg[j];
    }
    if (tid < 2 * D) s_kv[tid / D][tid % D] = kvreg;   // 0: k, 1: v
    for (int e = tid; e < D; e += AM_THREADS) s_cs[e] = e < H2 ? cs[e] : sn[e - H2];
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
        rope_pair(v[i], v[i + H2], s_cs[i], s_cs[H2 + i], r0, r1);
        if (h < G) {
            v[i] = r0 * qscale;
            v[i + H2] = r1 * qscale;
        } else {
            v[i] = r0;
            v[i + H2] = r1;
        }
    }
    __syncthreads();
    const bool owner = pos >= lo && pos < hi;
    if (owner) {   // the split holding pos writes the new K/V row (bf16)
        for (int d = tid; d < D; d += AM_THREADS) {
            kc[(size_t)pos * D + d] = f32_to_bf16(s_kv[0][d]);
            vc[(size_t)pos * D + d] = f32_to_bf16(s_kv[1][d]);
        }
    }
    for (int e = tid; e < 16 * C8; e += AM_THREADS) {   // q as the f16 A tile
        const int r = e / C8, c = e % C8;
        const float* q = &s_q[r][c * 8];
        *reinterpret_cast<uint4*>(sm + L::Q + q_off<D>(r, c)) =
            make_uint4(pack_f16x2(q[0], q[1]), pack_f16x2(q[2], q[3]), pack_f16x2(q[4], q[5]),
                       pack_f16x2(q[6], q[7]));
    }
    __syncthreads();
    uint32_t qa[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        const int mi = lane >> 3;
        const int r = (mi & 1) * 8 + (lane & 7), c = 2 * kk + (mi >> 1);
        ldsm4(sa_u32(sm + L::Q + q_off<D>(r, c)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    // ---- keys [lo, hi): tiles of 128 from the ring; warp w takes keys AM_KW*w.. ----
    float o[NT][4];
#pragma unroll
    for (int dn = 0; dn < NT; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows lane/4 and lane/4 + 8
    const int g4 = lane >> 2, q4 = lane & 3;
    for (int it = 0; it < n_tiles; ++it) {
        const int st = it % NS;
        const int t0 = lo + it * AM_TK;
        if (!am_wait(&full[st], (uint32_t)((it / NS) & 1))) s_err = 1;
        uint8_t* kt = sm + L::R0 + st * 2 * L::TILE;
        uint8_t* vt = kt + L::TILE;
        if (owner && pos >= t0 && pos < t0 + AM_TK && tid < C8) {   // the row the copy read stale
            const int r = pos - t0, c = tid;
            const float* kk8 = &s_kv[0][c * 8];
            const float* vv8 = &s_kv[1][c * 8];
            *reinterpret_cast<uint4*>(kt + kv_off(r, c)) =
                make_uint4(pack_bf16x2(kk8[0], kk8[1]), pack_bf16x2(kk8[2], kk8[3]),
                           pack_bf16x2(kk8[4], kk8[5]), pack_bf16x2(kk8[6], kk8[7]));
            *reinterpret_cast<uint4*>(vt + kv_off(r, c)) =
                make_uint4(pack_bf16x2(vv8[0], vv8[1]), pack_bf16x2(vv8[2], vv8[3]),
                           pack_bf16x2(vv8[4], vv8[5]), pack_bf16x2(vv8[6], vv8[7]));
        }
        __syncthreads();
#pragma unroll
        for (int blk = 0; blk < AM_KW / 16; ++blk) {
            const int r0k = warp * AM_KW + blk * 16;    // first key row of this block in the tile
            const int kw = t0 + r0k;
            if (kw >= hi) continue;                     // warp-uniform
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {   // S = Q K^T over 16 keys
                const int mi = lane >> 3;
                const int row = r0k + (mi >> 1) * 8 + (lane & 7), c = 2 * kk + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm4(sa_u32(kt + kv_off(row, c)), b0, b1, b2, b3);
                mma16816(s[0], qa[kk], bf2_to_h2(b0), bf2_to_h2(b1));
                mma16816(s[1], qa[kk], bf2_to_h2(b2), bf2_to_h2(b3));
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
                const int row = r0k + (mi & 1) * 8 + (lane & 7), c = dn + (mi >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm4t(sa_u32(vt + kv_off(row, c)), r0, r1, r2, r3);
                mma16816(o[dn], pa, bf2_to_h2(r0), bf2_to_h2(r1));
                mma16816(o[dn + 1], pa, bf2_to_h2(r2), bf2_to_h2(r3));
            }
        }
        __syncthreads();   // stage st fully read
        if (tid == 0 && it + NS < n_tiles) issue(it + NS);
    }
    if (tid == 0 && s_err) raise_status(a.status, EMBER_ERR_TIMEOUT);

    // ---- merge the warps: [AM_WARPS][16][D + 2] f32 = (m, l, O) per warp and row ----
    l0 += __shfl_xor_sync(FULL_MASK, l0, 1);
    l0 += __shfl_xor_sync(FULL_MASK, l0, 2);
    l1 += __shfl_xor_sync(FULL_MASK, l1, 1);
    l1 += __shfl_xor_sync(FULL_MASK, l1, 2);
    float* ws = reinterpret_cast<float*>(sm + L::R0);   // the ring is no longer read
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
        for (int w = 0; w < AM_WARPS; ++w) {
            const float* st = ws + ((size_t)w * 16 + h) * (D + 2);
            if (st[1] > 0.f) M = fmaxf(M, st[0]);
        }
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < AM_WARPS; ++w) {
            const float* st = ws + ((size_t)w * 16 + h) * (D + 2);
            if (st[1] > 0.f) v = fmaf(k == 0 ? 0.f : st[k], exp2f(st[0] - M), v);
        }
        if (k == 0) v = M;
        if (S == 1) {   // a single split is already the answer
            if (k >= 2) {
                float Ls = 0.f;
#pragma unroll
                for (int w = 0; w < AM_WARPS; ++w) {
                    const float* st = ws + ((size_t)w * 16 + h) * (D + 2);
                    if (st[1] > 0.f) Ls = fmaf(st[1], exp2f(st[0] - M), Ls);
                }
                const float out = Ls > 0.f ? v / Ls : 0.f;
                if (a.att_b) {
                    bool bad = false;
                    a.att_b[out0 + (size_t)h * D + k - 2] = f32_to_f16_chk(out, bad);
                    if (bad) raise_status(a.status, EMBER_ERR_RANGE);
                }
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
        if (a.att_b) {
            bool bad = false;
            a.att_b[out0 + e] = f32_to_f16_chk(O, bad);
            if (bad) raise_status(a.status, EMBER_ERR_RANGE);
        }
        else a.att[out0 + e] = O;
    }
    if (tid == 0) a.counters[b * a.NKV + g] = 0u;
}

bool attn_decode_mma_supported(int D, int G) { return (D == 64 || D == 128) && G >= 1 && G <= 16; }

void launch_attn_decode_mma(const AttnDecodeArgs& a, cudaStream_t s) {
    dim3 grid(a.splits < AM_MAX_SPLITS ? a.splits : AM_MAX_SPLITS, a.NKV, a.nb);
    const CUtensorMap& km = *reinterpret_cast<const CUtensorMap*>(a.k_map);
    const CUtensorMap& vm = *reinterpret_cast<const CUtensorMap*>(a.v_map);
    if (a.D == 64) {
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(k_attn_decode_mma<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AmSmem<64>::TOTAL);
            attr = true;
        }
        launch_k(k_attn_decode_mma<64>, grid, dim3(AM_THREADS), AmSmem<64>::TOTAL, s, km, vm, a);
    } else {
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(k_attn_decode_mma<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AmSmem<128>::TOTAL);
            attr = true;
        }
        launch_k(k_attn_decode_mma<128>, grid, dim3(AM_THREADS), AmSmem<128>::TOTAL, s, km, vm, a);
    }
}

}  // namespace ember
