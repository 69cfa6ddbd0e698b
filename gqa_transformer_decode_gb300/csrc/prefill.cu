// prefill.cu -- whole-prompt side of the forward: RMSNorm to the f16 GEMM
// operand, q/k-norm + RoPE + KV-cache write for n tokens, whole-sequence GQA
// attention (causal over the cache, or bidirectional within a sequence), the
// f32 final norm and the linear label head.
//
// Pages: LowLlamaBasic reference.py predict() (whole-sequence form, causal
// self_attn); PII-Tracer-vLLM serving/reference_forward.py forward() (q/k
// RMSNorm before RoPE, no mask, token_cls_head with bias).
#include "common.cuh"
#include "kernels.h"

namespace ember {

// ============================================================ RMSNorm rows ==
// OUT: 0 = f32, 1 = f16 (projection GEMM operand), 2 = bf16 (tied-head GEMM operand)
// zero (nullable): row t also clears zero[t * zlen, (t + 1) * zlen) -- the
// split-K output of the GEMM that consumes this operand, so that no memset
// node breaks the chain of programmatic launches.
template <int OUT>
__global__ void __launch_bounds__(256) k_rmsnorm(const float* x, const float* w, float eps, int H,
                                                 void* out, int* status, float* zero, int zlen) {
    // one row per CTA; H % 4 == 0 and H <= 8192 (the weights are loaded into
    // registers before the wait, the row in one batch of 16-byte loads)
    constexpr int MAXV = 8;
    __shared__ float red[32];
    const int t = blockIdx.x, H4 = H >> 2;
    float4 wv[MAXV], xv[MAXV];
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
        const int i = threadIdx.x + q * 256;
        wv[q] = i < H4 ? __ldg(reinterpret_cast<const float4*>(w) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_trigger();
    pdl_wait();
    if (zero)
        for (int i = threadIdx.x; i < zlen; i += 256) zero[(size_t)t * zlen + i] = 0.f;
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * H);
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < MAXV; ++q) {
        const int i = threadIdx.x + q * 256;
        xv[q] = i < H4 ? __ldcg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += xv[q].x * xv[q].x + xv[q].y * xv[q].y + xv[q].z * xv[q].z + xv[q].w * xv[q].w;
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) tot += red[k];
    const float ri = rsqrtf(tot / (float)H + eps);
#pragma unroll
    bool bad = false;
    for (int q = 0; q < MAXV; ++q) {
        const int i = threadIdx.x + q * 256;
        if (i >= H4) continue;
        const float a0 = xv[q].x * ri * wv[q].x, a1 = xv[q].y * ri * wv[q].y;
        const float a2 = xv[q].z * ri * wv[q].z, a3 = xv[q].w * ri * wv[q].w;
        if (OUT == 0) {
            reinterpret_cast<float4*>(static_cast<float*>(out) + (size_t)t * H)[i] = make_float4(a0, a1, a2, a3);
        } else {
            uint2* o = reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + (size_t)t * H);
            o[i] = OUT == 1 ? make_uint2(pack_f16x2_chk(a0, a1, bad), pack_f16x2_chk(a2, a3, bad))
                            : make_uint2(pack_bf16x2(a0, a1), pack_bf16x2(a2, a3));
        }
    }
    if (bad) raise_status(status, EMBER_ERR_RANGE);
}

// A warp per row for H <= 2048 (H % 128 == 0) and at least 1024 rows: the
// row in registers (H/128 16-byte loads per lane), a warp reduction, no
// block barrier; 8 rows per CTA.
template <int NV>
__global__ void __launch_bounds__(256) k_rmsnorm_warp(const float* x, const float* w, float eps, int H,
                                                      int n, uint16_t* out, int* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();
    if (t >= n) return;
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * H);
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        v[q] = __ldcg(xr + lane + 32 * q);
        ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
    }
    ss = warp_sum(ss);
    const float ri = rsqrtf(ss / (float)H + eps);
    uint2* o = reinterpret_cast<uint2*>(out + (size_t)t * H);
    bool bad = false;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        const float4 g = __ldg(reinterpret_cast<const float4*>(w) + lane + 32 * q);
        o[lane + 32 * q] = make_uint2(pack_f16x2_chk(v[q].x * ri * g.x, v[q].y * ri * g.y, bad),
                                      pack_f16x2_chk(v[q].z * ri * g.z, v[q].w * ri * g.w, bad));
    }
    if (bad) raise_status(status, EMBER_ERR_RANGE);
}

void launch_rmsnorm_h(const float* x, const float* w, float eps, int n, int H, uint16_t* xb,
                      int* status, cudaStream_t s, float* zero, int zlen) {
    const dim3 g((n + 7) / 8), b(256);
    // a warp per row pays off with many rows; a few rows (decode batches,
    // short prompts) keep a CTA per row so that they spread over the SMs
    if (!zero && n >= 1024 && H % 128 == 0 && H <= 2048) {
        switch (H / 128) {
#define EMBER_RMS_WARP(NV) \
    case NV: launch_k(k_rmsnorm_warp<NV>, g, b, 0, s, x, w, eps, H, n, xb, status); return;
            EMBER_RMS_WARP(1) EMBER_RMS_WARP(2) EMBER_RMS_WARP(3) EMBER_RMS_WARP(4)
            EMBER_RMS_WARP(5) EMBER_RMS_WARP(6) EMBER_RMS_WARP(7) EMBER_RMS_WARP(8)
            EMBER_RMS_WARP(9) EMBER_RMS_WARP(10) EMBER_RMS_WARP(11) EMBER_RMS_WARP(12)
            EMBER_RMS_WARP(13) EMBER_RMS_WARP(14) EMBER_RMS_WARP(15) EMBER_RMS_WARP(16)
#undef EMBER_RMS_WARP
            default: break;
        }
    }
    launch_k(k_rmsnorm<1>, dim3(n), dim3(256), 0, s, x, w, eps, H, (void*)xb, status, zero, zlen);
}
void launch_rmsnorm_bf16(const float* x, const float* w, float eps, int n, int H, uint16_t* xb,
                         cudaStream_t s) {
    launch_k(k_rmsnorm<2>, dim3(n), dim3(256), 0, s, x, w, eps, H, (void*)xb, (int*)nullptr, (float*)nullptr, 0);
}
void launch_rmsnorm_f32(const float* x, const float* w, float eps, int n, int H, float* h,
                        cudaStream_t s) {
    launch_k(k_rmsnorm<0>, dim3(n), dim3(256), 0, s, x, w, eps, H, (void*)h, (int*)nullptr, (float*)nullptr, 0);
}

// =================================================== q/k norm, RoPE, K/V write ==
__global__ void __launch_bounds__(128) k_rope_kv(RopeKVArgs a) {
    extern __shared__ float sm[];   // [(NH + 2*NKV) * D] f32
    const int t = blockIdx.x;
    const int D = a.D, H2 = D / 2;
    const int nq = a.NH * D, nkv = a.NKV * D;
    const int z = t / a.T_per_seq;
    const int pos = a.pos0 + t % a.T_per_seq;
    const float* row = a.qkv + (size_t)t * a.ld_qkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();
    if (!a.q_norm) {   // no per-head norm: four rotate-half pairs per item, in registers
        const int Q4 = H2 / 4;                       // items per head
        const int n_rope = (a.NH + a.NKV) * Q4, n_v = nkv / 4;
        const float* cs = a.cos_t + (size_t)pos * H2;
        const float* sn = a.sin_t + (size_t)pos * H2;
        for (int e = tid; e < n_rope + n_v; e += blockDim.x) {
            if (e < n_rope) {
                const int h = e / Q4, i0 = (e % Q4) * 4;
                const float4 x0 = *reinterpret_cast<const float4*>(row + h * D + i0);
                const float4 x1 = *reinterpret_cast<const float4*>(row + h * D + H2 + i0);
                const float4 cv = *reinterpret_cast<const float4*>(cs + i0);
                const float4 sv = *reinterpret_cast<const float4*>(sn + i0);
                float r0[4], r1[4];
                rope_pair(x0.x, x1.x, cv.x, sv.x, r0[0], r1[0]);
                rope_pair(x0.y, x1.y, cv.y, sv.y, r0[1], r1[1]);
                rope_pair(x0.z, x1.z, cv.z, sv.z, r0[2], r1[2]);
                rope_pair(x0.w, x1.w, cv.w, sv.w, r0[3], r1[3]);
                // queries in f16 (the attention MMA's operand), keys in bf16 (the cache)
                const bool isq = h < a.NH;
                const uint2 lo = isq ? make_uint2(pack_f16x2(r0[0], r0[1]), pack_f16x2(r0[2], r0[3]))
                                     : make_uint2(pack_bf16x2(r0[0], r0[1]), pack_bf16x2(r0[2], r0[3]));
                const uint2 hi = isq ? make_uint2(pack_f16x2(r1[0], r1[1]), pack_f16x2(r1[2], r1[3]))
                                     : make_uint2(pack_bf16x2(r1[0], r1[1]), pack_bf16x2(r1[2], r1[3]));
                uint16_t* dst;
                if (isq) {
                    dst = a.q_out + (size_t)t * nq + h * D;
                } else {
                    dst = a.kc + z * a.seq_stride + (h - a.NH) * a.head_stride + (long long)pos * D;
                    if (a.kh) {   // the same bf16 values, as f16
                        uint16_t* kd = a.kh + ((size_t)(z * a.NKV + h - a.NH) * a.kh_pad + pos) * D;
                        *reinterpret_cast<uint2*>(kd + i0) =
                            make_uint2(pack_f16x2(bf16_lo(lo.x), bf16_hi(lo.x)), pack_f16x2(bf16_lo(lo.y), bf16_hi(lo.y)));
                        *reinterpret_cast<uint2*>(kd + H2 + i0) =
                            make_uint2(pack_f16x2(bf16_lo(hi.x), bf16_hi(hi.x)), pack_f16x2(bf16_lo(hi.y), bf16_hi(hi.y)));
                    }
                }
                *reinterpret_cast<uint2*>(dst + i0) = lo;
                *reinterpret_cast<uint2*>(dst + H2 + i0) = hi;
            } else {
                const int f = (e - n_rope) * 4, g = f / D, d = f % D;
                const float4 v = *reinterpret_cast<const float4*>(row + nq + nkv + f);
                *reinterpret_cast<uint2*>(a.vc + z * a.seq_stride + g * a.head_stride + (long long)pos * D + d) =
                    make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
            }
        }
        return;
    }
    if (D % 64 == 0) {   // per-head RMSNorm, then RoPE: a warp per head, lane l holds
        // rotate-half pairs i = l*PPL .. l*PPL + PPL - 1 (both halves) in registers
        const int PPL = D / 64;   // 1 or 2
        const int i0 = lane * PPL;
        const float* cs = a.cos_t + (size_t)pos * H2;
        const float* sn = a.sin_t + (size_t)pos * H2;
        for (int h = warp; h < a.NH + a.NKV; h += blockDim.x / 32) {
            const float* x = row + h * D;
            const float* w = h < a.NH ? a.q_norm : a.k_norm;
            float lo[2] = {0.f, 0.f}, hi[2] = {0.f, 0.f};
            if (PPL == 2) {
                const float2 u = *reinterpret_cast<const float2*>(x + i0);
                const float2 v = *reinterpret_cast<const float2*>(x + H2 + i0);
                lo[0] = u.x; lo[1] = u.y; hi[0] = v.x; hi[1] = v.y;
            } else {
                lo[0] = x[i0];
                hi[0] = x[H2 + i0];
            }
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < 2; ++k) ss += lo[k] * lo[k] + hi[k] * hi[k];
            ss = warp_sum(ss);
            const float ri = rsqrtf(ss / (float)D + a.eps);
            float r0[2] = {0.f, 0.f}, r1[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (k < PPL) {
                    const int i = i0 + k;
                    rope_pair(lo[k] * ri * w[i], hi[k] * ri * w[H2 + i], cs[i], sn[i], r0[k], r1[k]);
                }
            }
            uint16_t* dst;
            const bool isq = h < a.NH;   // queries f16 (the attention operand), keys bf16 (the cache)
            if (isq) dst = a.q_out + (size_t)t * nq + h * D;
            else dst = a.kc + z * a.seq_stride + (h - a.NH) * a.head_stride + (long long)pos * D;
            if (PPL == 2) {
                *reinterpret_cast<uint32_t*>(dst + i0) = isq ? pack_f16x2(r0[0], r0[1]) : pack_bf16x2(r0[0], r0[1]);
                *reinterpret_cast<uint32_t*>(dst + H2 + i0) = isq ? pack_f16x2(r1[0], r1[1]) : pack_bf16x2(r1[0], r1[1]);
            } else {
                dst[i0] = isq ? f32_to_f16(r0[0]) : f32_to_bf16(r0[0]);
                dst[H2 + i0] = isq ? f32_to_f16(r1[0]) : f32_to_bf16(r1[0]);
            }
            if (!isq && a.kh) {   // the same bf16 values, as f16
                uint16_t* kd = a.kh + ((size_t)(z * a.NKV + h - a.NH) * a.kh_pad + pos) * D;
                if (PPL == 2) {
                    const uint32_t b0 = pack_bf16x2(r0[0], r0[1]), b1 = pack_bf16x2(r1[0], r1[1]);
                    *reinterpret_cast<uint32_t*>(kd + i0) = pack_f16x2(bf16_lo(b0), bf16_hi(b0));
                    *reinterpret_cast<uint32_t*>(kd + H2 + i0) = pack_f16x2(bf16_lo(b1), bf16_hi(b1));
                } else {
                    kd[i0] = f32_to_f16(bf16_to_f32(f32_to_bf16(r0[0])));
                    kd[H2 + i0] = f32_to_f16(bf16_to_f32(f32_to_bf16(r1[0])));
                }
            }
        }
        for (int f = tid * 4; f < nkv; f += blockDim.x * 4) {   // V rows: bf16 into the cache
            const int g = f / D, d = f % D;
            const float4 v = *reinterpret_cast<const float4*>(row + nq + nkv + f);
            *reinterpret_cast<uint2*>(a.vc + z * a.seq_stride + g * a.head_stride + (long long)pos * D + d) =
                make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        }
        return;
    }
    for (int e = tid; e < nq + 2 * nkv; e += blockDim.x) sm[e] = row[e];
    __syncthreads();
    if (a.q_norm) {   // PII-Tracer forward(): per-head RMSNorm of q and k before RoPE
        for (int h = warp; h < a.NH + a.NKV; h += blockDim.x / 32) {
            float* v = sm + h * D;
            const float* w = h < a.NH ? a.q_norm : a.k_norm;
            float ss = 0.f;
            for (int d = lane; d < D; d += 32) ss += v[d] * v[d];
            ss = warp_sum(ss);
            const float ri = rsqrtf(ss / (float)D + a.eps);
            for (int d = lane; d < D; d += 32) v[d] = v[d] * ri * w[d];
        }
        __syncthreads();
    }
    const float* cs = a.cos_t + (size_t)pos * H2;
    const float* sn = a.sin_t + (size_t)pos * H2;
    uint16_t* qo = a.q_out + (size_t)t * nq;
    for (int e = tid; e < (a.NH + a.NKV) * H2; e += blockDim.x) {
        const int h = e / H2, i = e % H2;
        const float* v = sm + h * D;
        float r0, r1;
        rope_pair(v[i], v[i + H2], cs[i], sn[i], r0, r1);
        if (h < a.NH) {
            qo[h * D + i] = f32_to_f16(r0);
            qo[h * D + i + H2] = f32_to_f16(r1);
        } else {
            const int g = h - a.NH;
            uint16_t* kr = a.kc + z * a.seq_stride + g * a.head_stride + (long long)pos * D;
            kr[i] = f32_to_bf16(r0);
            kr[i + H2] = f32_to_bf16(r1);
            if (a.kh) {   // the same bf16 values, as f16
                uint16_t* kd = a.kh + ((size_t)(z * a.NKV + g) * a.kh_pad + pos) * D;
                kd[i] = f32_to_f16(bf16_to_f32(kr[i]));
                kd[i + H2] = f32_to_f16(bf16_to_f32(kr[i + H2]));
            }
        }
    }
    for (int e = tid; e < nkv; e += blockDim.x) {
        const int g = e / D, d = e % D;
        a.vc[z * a.seq_stride + g * a.head_stride + (long long)pos * D + d] =
            f32_to_bf16(sm[nq + nkv + e]);
    }
}

void launch_rope_kv(const RopeKVArgs& a, cudaStream_t s) {
    // only the per-head-norm path for head_dim % 64 != 0 stages the row in shared memory
    const bool staged = a.q_norm && (a.D % 64) != 0;
    const size_t smem = staged ? (size_t)(a.NH + 2 * a.NKV) * a.D * sizeof(float) : 0;
    launch_k(k_rope_kv, dim3(a.n), dim3(128), smem, s, a);
}

// ======================================================== prefill attention ==
// CTA = (query tile of QT rows, kv head g, sequence z), 8 warps.  The QT*G
// (row, head) items are dealt round-robin to the warps; key tiles of 32 rows
// are staged in shared memory, lane j scores key j, the warp keeps an online
// softmax per item and accumulates P.V with lane-owned output columns.
constexpr int APF_THREADS = 256;
constexpr int APF_TK = 32;

template <int D, int IPW>
__global__ void __launch_bounds__(APF_THREADS) k_attn_prefill(AttnPrefillArgs a, int QT) {
    constexpr int KP = D + 2;
    constexpr int DL = D / 32 > 0 ? D / 32 : 1;   // output columns per lane
    extern __shared__ float smq[];                // [QT*G][D] f32 queries
    __shared__ __align__(16) uint16_t s_k[APF_TK][KP];
    __shared__ __align__(16) uint16_t s_v[APF_TK][D];
    const int G = a.NH / a.NKV;
    const int g = blockIdx.y, z = blockIdx.z;
    const int qt0 = blockIdx.x * QT;
    const int rows = min(QT, a.T_per_seq - qt0);
    if (rows <= 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();
    const int items = rows * G;
    const float qk_scale = 1.4426950408889634f * rsqrtf((float)D);

    // stage this tile's queries (item i = r*G + h -> query head g*G + h of row r)
    for (int e = tid; e < items * D; e += APF_THREADS) {
        const int i = e / D, d = e % D, r = i / G, h = i % G;
        const size_t qrow = (size_t)z * a.T_per_seq + qt0 + r;
        smq[e] = __half2float(__ushort_as_half(a.q[qrow * a.NH * D + (size_t)(g * G + h) * D + d])) *
                 qk_scale;
    }
    float m[IPW], l[IPW], acc[IPW][DL];
#pragma unroll
    for (int k = 0; k < IPW; ++k) {
        m[k] = -INFINITY;
        l[k] = 0.f;
#pragma unroll
        for (int c = 0; c < DL; ++c) acc[k][c] = 0.f;
    }
    const int n_all = a.pos0 + a.T_per_seq;                     // keys in the sequence
    const int kend = a.causal ? min(n_all, a.pos0 + qt0 + rows) : n_all;
    const uint16_t* kb = a.kc + z * a.seq_stride + g * a.head_stride;
    const uint16_t* vb = a.vc + z * a.seq_stride + g * a.head_stride;

    for (int t0 = 0; t0 < kend; t0 += APF_TK) {
        const int nt = min(APF_TK, kend - t0);
        __syncthreads();
        constexpr int C8 = D / 8;
        for (int e = tid; e < nt * C8; e += APF_THREADS) {
            const int j = e / C8, c = e % C8;
            const uint4 k4 = *reinterpret_cast<const uint4*>(kb + (size_t)(t0 + j) * D + c * 8);
            const uint4 v4 = *reinterpret_cast<const uint4*>(vb + (size_t)(t0 + j) * D + c * 8);
            uint32_t* kd = reinterpret_cast<uint32_t*>(&s_k[j][c * 8]);
            kd[0] = k4.x; kd[1] = k4.y; kd[2] = k4.z; kd[3] = k4.w;
            *reinterpret_cast<uint4*>(&s_v[j][c * 8]) = v4;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < IPW; ++k) {
            const int i = warp + k * (APF_THREADS / 32);
            if (i >= items) break;
            const int r = i / G;
            const int qpos = a.pos0 + qt0 + r;
            const int kp = t0 + lane;
            const bool vis = lane < nt && (a.causal ? kp <= qpos : true);
            float s = -INFINITY;
            if (vis) {
                const float* qv = smq + (size_t)i * D;
                const uint32_t* kr = reinterpret_cast<const uint32_t*>(s_k[lane]);
                float dot = 0.f;
#pragma unroll 8
                for (int d2 = 0; d2 < D / 2; ++d2) {
                    const uint32_t kk = kr[d2];
                    dot = fmaf(qv[2 * d2], bf16_lo(kk), dot);
                    dot = fmaf(qv[2 * d2 + 1], bf16_hi(kk), dot);
                }
                s = dot;
            }
            const float tm = warp_max(s);
            if (tm == -INFINITY) continue;   // nothing visible for this item in this tile
            const float mn = fmaxf(m[k], tm);
            const float p = exp2f(s - mn);
            const float sc = exp2f(m[k] - mn);
            l[k] = l[k] * sc + warp_sum(p);
            m[k] = mn;
#pragma unroll
            for (int c = 0; c < DL; ++c) acc[k][c] *= sc;
            for (int j = 0; j < nt; ++j) {
                const float pj = __shfl_sync(FULL_MASK, p, j);
#pragma unroll
                for (int c = 0; c < DL; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) acc[k][c] = fmaf(pj, bf16_to_f32(s_v[j][d]), acc[k][c]);
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < IPW; ++k) {
        const int i = warp + k * (APF_THREADS / 32);
        if (i >= items) break;
        const int r = i / G, h = i % G;
        const size_t qrow = (size_t)z * a.T_per_seq + qt0 + r;
        uint16_t* o = a.att + qrow * a.NH * D + (size_t)(g * G + h) * D;
        const float inv = 1.f / l[k];
#pragma unroll
        for (int c = 0; c < DL; ++c) {
            const int d = lane + 32 * c;
            if (d < D) {
                bool bad = false;
                o[d] = f32_to_f16_chk(acc[k][c] * inv, bad);
                if (bad) raise_status(a.status, EMBER_ERR_RANGE);
            }
        }
    }
}

template <int D>
static void launch_apf(const AttnPrefillArgs& a, int QT, dim3 grid, size_t smem, cudaStream_t s) {
    static bool attr = false;   // static K/V tiles + dynamic queries may exceed 48 KB
    if (!attr) {
        cudaFuncSetAttribute(k_attn_prefill<D, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             64 * 1024);
        attr = true;
    }
    launch_k(k_attn_prefill<D, 16>, grid, dim3(APF_THREADS), smem, s, a, QT);
}

void launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t s) {
    const int G = a.NH / a.NKV;
    // QT rows x G heads = items, at most 16 per warp (128 per CTA) and their
    // f32 queries within 48 KB of shared memory.
    const int max_items = 12288 / a.D < 128 ? 12288 / a.D : 128;
    int QT = 64;
    while (QT > 1 && QT * G > max_items) QT >>= 1;
    const int nseq = a.n / a.T_per_seq;
    dim3 grid((a.T_per_seq + QT - 1) / QT, a.NKV, nseq);
    const size_t smem = (size_t)QT * G * a.D * sizeof(float);
    switch (a.D) {
        case 16: launch_apf<16>(a, QT, grid, smem, s); break;
        case 32: launch_apf<32>(a, QT, grid, smem, s); break;
        case 64: launch_apf<64>(a, QT, grid, smem, s); break;
        case 128: launch_apf<128>(a, QT, grid, smem, s); break;
        default: break;
    }
}

// ================================================================ label head ==
__global__ void __launch_bounds__(256) k_cls_head(const float* h, int n, int H, const uint16_t* W,
                                                  const float* b, int labels, float* out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    pdl_trigger();
    pdl_wait();
    if (t >= n) return;
    const float* hr = h + (size_t)t * H;
    for (int j = 0; j < labels; ++j) {
        const uint16_t* w = W + (size_t)j * H;
        float s = 0.f;
        for (int k = lane; k < H; k += 32) s = fmaf(hr[k], bf16_to_f32(w[k]), s);
        s = warp_sum(s);
        if (lane == 0) out[(size_t)t * labels + j] = s + (b ? b[j] : 0.f);
    }
}

void launch_cls_head(const float* h, int n, int H, const uint16_t* W, const float* b, int labels,
                     float* out, cudaStream_t s) {
    launch_k(k_cls_head, dim3((n + 7) / 8), dim3(256), 0, s, h, n, H, W, b, labels, out);
}

// ============================================= mean-pooled (sensitivity) head ==
// Sequence b: the mean over its T rows of h (each column summed in position
// order), then out[b][j] = mean . W[j] + b[j] by block reductions.
__global__ void __launch_bounds__(256) k_pooled_head(const float* h, int T, int H, const uint16_t* W,
                                                     const uint16_t* bias, int n_out, float* out) {
    extern __shared__ float s_mean[];   // [H]
    __shared__ float s_red[32];
    pdl_trigger();
    pdl_wait();
    const float* hb = h + (size_t)blockIdx.x * T * H;
    const float inv = 1.f / (float)T;
    for (int k = threadIdx.x; k < H; k += blockDim.x) {
        float acc = 0.f;
        for (int t = 0; t < T; ++t) acc += __ldg(hb + (size_t)t * H + k);
        s_mean[k] = acc * inv;
    }
    __syncthreads();
    for (int j = 0; j < n_out; ++j) {
        const uint16_t* w = W + (size_t)j * H;
        float s = 0.f;
        for (int k = threadIdx.x; k < H; k += blockDim.x) s = fmaf(s_mean[k], bf16_to_f32(w[k]), s);
        s = block_sum(s, s_red);
        if (threadIdx.x == 0) out[(size_t)blockIdx.x * n_out + j] = s + (bias ? bf16_to_f32(bias[j]) : 0.f);
    }
}

cudaError_t launch_pooled_head(const float* h, int B, int T, int H, const uint16_t* W, const uint16_t* b,
                               int n_out, float* out, cudaStream_t s) {
    return launch_k(k_pooled_head, dim3(B), dim3(256), (size_t)H * sizeof(float), s, h, T, H, W, b, n_out, out);
}

// ================================================================ row copy ==
__global__ void k_copy_f32(float* dst, const float* src, int n) {
    pdl_trigger();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

void launch_copy_f32(float* dst, const float* src, int n, cudaStream_t s) {
    launch_k(k_copy_f32, dim3((n + 255) / 256 < 64 ? (n + 255) / 256 : 64), dim3(256), 0, s, dst, src, n);
}

// ============================================== standalone RoPE + bf16 store ==
__global__ void k_rope_store(const float* x, int n_heads, int D, const float* cos_t,
                             const float* sin_t, uint16_t* out) {
    const int t = blockIdx.x, H2 = D / 2;
    const float* xr = x + (size_t)t * n_heads * D;
    uint16_t* o = out + (size_t)t * n_heads * D;
    const float* cs = cos_t + (size_t)t * H2;
    const float* sn = sin_t + (size_t)t * H2;
    for (int e = threadIdx.x; e < n_heads * H2; e += blockDim.x) {
        const int h = e / H2, i = e % H2;
        float r0, r1;
        rope_pair(xr[h * D + i], xr[h * D + i + H2], cs[i], sn[i], r0, r1);
        o[h * D + i] = f32_to_bf16(r0);
        o[h * D + i + H2] = f32_to_bf16(r1);
    }
}

void launch_rope_store(const float* x, int n_tok, int n_heads, int D, const float* cos_t,
                       const float* sin_t, uint16_t* out, cudaStream_t s) {
    count_launches(1);
    k_rope_store<<<n_tok, 128, 0, s>>>(x, n_heads, D, cos_t, sin_t, out);
}

}  // namespace ember
