// decode.cu -- batch-1..8 decode path: embedding gather, RMSNorm-fused split
// GEMV with its epilogues (bias, residual add, SwiGLU, LM head + argmax),
// split-KV flash-decoding GQA attention with the fused q/k-norm + RoPE + KV
// write, and the end-of-step argmax write-back / cursor advance.
//
// Pages: ember scripts/reference_forward.py forward() (the per-token layer
// loop this path runs, one token per sequence); ember internals "kv cache"
// (cursor advances after all layers, explicit positions) and "grouped-query
// attention" (query head h reads kv head h / G).
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace ember {

// ============================================================== embedding ==
__global__ void k_embed(EmbedArgs a) {
    const int t = blockIdx.x;
    __shared__ int s_id;
    pdl_trigger();
    pdl_wait();   // x is still read by the previous step's LM head
    if (threadIdx.x == 0) {
        int id = a.ids[t];
        int ok = 1;
        if (id < 0 || id >= a.V) {          // Falcon-H1 logits(): token outside vocabulary
            raise_status(a.status, EMBER_ERR_TOKEN);
            id = 0;
            ok = 0;
        }
        if (a.seqs) {
            const int seq = a.seqs[t];
            int pos = -1;
            if (seq < 0 || seq >= a.max_seqs) {
                raise_status(a.status, EMBER_ERR_INVALID_ARG);
                ok = 0;
            } else {
                // no positions array: the token goes at its sequence's cursor
                pos = a.positions ? a.positions[t] : a.cursor[seq];
                if (pos < 0 || pos >= a.max_len) {
                    raise_status(a.status, EMBER_ERR_CAPACITY);
                    ok = 0;
                } else if (pos != a.cursor[seq]) {  // ember internals: explicit pos == cursor
                    raise_status(a.status, EMBER_ERR_STATE);
                }
            }
            a.tok_ok[t] = ok;
            a.tok_pos[t] = pos;
        }
        if (t == 0 && a.pf_seq >= 0 && a.cursor[a.pf_seq] != a.pf_start)
            raise_status(a.status, EMBER_ERR_STATE);
        s_id = id;
    }
    __syncthreads();
    const uint16_t* row = a.E + (size_t)s_id * a.H;
    float* out = a.x + (size_t)t * a.H;
    for (int i = threadIdx.x; i < a.H; i += blockDim.x) out[i] = bf16_to_f32(row[i]);
    if (a.zero0) {
        const int zl = a.zlen > 0 ? a.zlen : a.H;
        for (int i = threadIdx.x; i < zl; i += blockDim.x) {
            a.zero0[(size_t)t * zl + i] = 0.f;
            a.zero1[(size_t)t * zl + i] = 0.f;
        }
    }
}

void launch_embed(const EmbedArgs& a, cudaStream_t s) {
    launch_k(k_embed, dim3(a.n), dim3(256), 0, s, a);
}

// =================================================================== GEMV ==
// One CTA of 256 threads handles tiles of R = 256/TPR consecutive weight rows;
// TPR threads share a row, each issuing up to MAXJ independent 16-byte loads
// before any arithmetic so that ~R*K*2 bytes per CTA are in flight.  The grid
// is persistent (a few CTAs per SM striding over tiles) so the RMSNorm
// statistics of the nb input rows are computed once per CTA.
constexpr int GEMV_THREADS = 256;
constexpr int GEMV_MAXJ = 8;

// Weight formats of the GEMV: bf16, f16, or q8_0 ("ember internals" q8_0
// block quantization: 32 int8 codes per f16 scale d, value q * d; stored here
// as codes [N][K] and scales [N][K/32]).  A unit is 8 consecutive weights of
// a row: 16 bytes of bf16 / f16, 8 bytes of codes.
enum { WF_BF16 = 0, WF_F16 = 1, WF_Q8 = 2 };

__device__ __forceinline__ uint2 ld_stream8(const uint2* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// Issue the weight loads of one row tile (immutable data: may run before
// the predecessor kernel has finished).
template <int TPR, int WF>
__device__ __forceinline__ void gemv_load_tile(const GemvArgs& a, int tile, int r, int sub, int K8,
                                               uint4 (&w)[GEMV_MAXJ], float (&sc)[GEMV_MAXJ]) {
    constexpr int R = GEMV_THREADS / TPR;
    const int row = tile * R + r;
    if (row >= a.N) return;
    if (WF == WF_Q8) {
        const uint2* qrow = reinterpret_cast<const uint2*>(a.Wq + (size_t)row * a.K);
        const __half* drow = reinterpret_cast<const __half*>(a.Wd) + (size_t)row * (a.K / 32);
#pragma unroll
        for (int j = 0; j < GEMV_MAXJ; ++j) {
            const int c = sub + j * TPR;
            if (c < K8) {
                const uint2 q = ld_stream8(qrow + c);
                w[j].x = q.x;
                w[j].y = q.y;
                sc[j] = __half2float(__ldg(drow + (c >> 2)));
            }
        }
    } else {
        const uint4* wrow = reinterpret_cast<const uint4*>(a.W + (size_t)row * a.K);
#pragma unroll
        for (int j = 0; j < GEMV_MAXJ; ++j) {
            const int c = sub + j * TPR;
            if (c < K8) w[j] = ld_stream(wrow + c);
        }
    }
}

// the 8 weights of a unit as f32 (q8_0: code times the block's scale, exact)
template <int WF>
__device__ __forceinline__ void gemv_unpack(const uint4& w, float scale, float* f) {
    if (WF == WF_Q8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[i] = (float)(int8_t)((w.x >> (8 * i)) & 0xFF) * scale;
            f[4 + i] = (float)(int8_t)((w.y >> (8 * i)) & 0xFF) * scale;
        }
    } else {
        unpack8w<WF == WF_F16>(w, f);
    }
}

template <int TPR, int NB, int WF, bool XA = false>
__global__ void __launch_bounds__(GEMV_THREADS) k_gemv(GemvArgs a) {
    constexpr int R = GEMV_THREADS / TPR;
    constexpr int GL = TPR < 32 ? TPR : 32;       // lanes reduced by shuffles
    constexpr int WPR = TPR > 32 ? TPR / 32 : 1;  // warps per row
    __shared__ float s_red[32];
    __shared__ float s_rinv[NB];
    __shared__ float s_part[R][WPR][NB];
    __shared__ unsigned long long s_key[NB];

    const int tid = threadIdx.x;
    const int r = tid / TPR, sub = tid % TPR;
    const int K8 = a.K >> 3;
    const int nb = a.nb;
    const int n_tiles = (a.N + R - 1) / R;

    pdl_trigger();
    // The first tile's weights stream in while the previous kernel drains.
    uint4 w[GEMV_MAXJ];
    int tile = blockIdx.x;
    float wsc[GEMV_MAXJ];   // q8_0: the scale of each unit's block
#pragma unroll
    for (int j = 0; j < GEMV_MAXJ; ++j) wsc[j] = 0.f;
    if (tile < n_tiles) gemv_load_tile<TPR, WF>(a, tile, r, sub, K8, w, wsc);
    pdl_wait();
    // XA (one row): the normalised input rmsnorm(x + x_add) = (x + x_add) *
    // norm_w / rms staged once in shared memory, so that the tile loop reads
    // only weights and this vector
    extern __shared__ float s_xa[];
    if (XA) {
        float ss = 0.f;
        for (int i = tid * 4; i < a.K; i += GEMV_THREADS * 4) {
            float4 t = __ldcg(reinterpret_cast<const float4*>(a.x + i));
            for (int z = 0; z < a.x_add_slots; ++z) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(a.x_add + (size_t)z * a.K + i));
                t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
            }
            ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
            *reinterpret_cast<float4*>(s_xa + i) = t;
        }
        if (a.norm_w) {
            ss = block_sum(ss, s_red);
            const float rinv = rsqrtf(ss / (float)a.K + a.eps);
            for (int i = tid * 4; i < a.K; i += GEMV_THREADS * 4) {   // the elements this thread wrote
                const float4 n = reinterpret_cast<const float4*>(a.norm_w)[i / 4];
                float4 t = *reinterpret_cast<float4*>(s_xa + i);
                t.x *= n.x * rinv; t.y *= n.y * rinv; t.z *= n.z * rinv; t.w *= n.w * rinv;
                *reinterpret_cast<float4*>(s_xa + i) = t;
            }
        }
        __syncthreads();
    }
    const bool wnorm = a.norm_w && !XA;   // otherwise the input already carries the norm

    // RMSNorm statistics of every input row (ember reference_forward.py rmsnorm()).
    for (int b = 0; b < NB; ++b) {
        float rinv = 1.f;
        if (wnorm && b < nb) {
            const float* xb = XA ? s_xa : a.x + (size_t)b * a.ldx;
            float ss = 0.f;
            for (int i = tid; i < a.K; i += GEMV_THREADS) ss += xb[i] * xb[i];
            ss = block_sum(ss, s_red);
            rinv = rsqrtf(ss / (float)a.K + a.eps);
        }
        if (tid == 0) s_rinv[b] = rinv;
    }
    if (tid < NB) s_key[tid] = 0ull;
    __syncthreads();

    unsigned long long best[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) best[b] = 0ull;

    for (; tile < n_tiles; tile += gridDim.x) {
        const int row = tile * R + r;
        const bool rv = row < a.N;
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll
        for (int j = 0; j < GEMV_MAXJ; ++j) {
            const int c = sub + j * TPR;
            if (rv && c < K8) {
                float wf[8];
                gemv_unpack<WF>(w[j], wsc[j], wf);
                if (wnorm) {
                    const float4 n0 = reinterpret_cast<const float4*>(a.norm_w)[2 * c];
                    const float4 n1 = reinterpret_cast<const float4*>(a.norm_w)[2 * c + 1];
                    wf[0] *= n0.x; wf[1] *= n0.y; wf[2] *= n0.z; wf[3] *= n0.w;
                    wf[4] *= n1.x; wf[5] *= n1.y; wf[6] *= n1.z; wf[7] *= n1.w;
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b < nb) {
                        const float4* xp =
                            reinterpret_cast<const float4*>(XA ? s_xa : a.x + (size_t)b * a.ldx) + 2 * c;
                        const float4 x0 = xp[0], x1 = xp[1];
                        float s = acc[b];
                        s = fmaf(wf[0], x0.x, s); s = fmaf(wf[1], x0.y, s);
                        s = fmaf(wf[2], x0.z, s); s = fmaf(wf[3], x0.w, s);
                        s = fmaf(wf[4], x1.x, s); s = fmaf(wf[5], x1.y, s);
                        s = fmaf(wf[6], x1.z, s); s = fmaf(wf[7], x1.w, s);
                        acc[b] = s;
                    }
                }
            }
        }
        // next tile's weights fly during this tile's reduction and epilogue
        if (tile + (int)gridDim.x < n_tiles) gemv_load_tile<TPR, WF>(a, tile + gridDim.x, r, sub, K8, w, wsc);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
#pragma unroll
            for (int o = GL / 2; o > 0; o >>= 1) acc[b] += __shfl_xor_sync(FULL_MASK, acc[b], o);
        }
        if ((tid & (GL - 1)) == 0) {
            const int wp = TPR > 32 ? (sub >> 5) : 0;
#pragma unroll
            for (int b = 0; b < NB; ++b) s_part[r][wp][b] = acc[b];
        }
        __syncthreads();
        // Epilogue: thread e handles (row r_e, token b_e).
        if (tid < R * NB) {
            const int re = tid / NB, be = tid % NB;
            const int rowe = tile * R + re;
            float v = 0.f;
#pragma unroll
            for (int q = 0; q < WPR; ++q) v += s_part[re][q][be];
            v *= s_rinv[be] * pow2f(a.w_exp);
            if (rowe < a.N && be < nb) {
                float* o = a.out + (size_t)be * a.ldo;
                if (a.mode == EPI_STORE) {
                    o[rowe] = a.bias ? v + a.bias[rowe] : v;
                } else if (a.mode == EPI_RESID) {
                    o[rowe] += v;
                } else if (a.mode == EPI_ARGMAX) {
                    if (a.out) o[rowe] = v;
                    const unsigned long long k = argmax_key(v, (uint32_t)rowe);
                    best[be] = k > best[be] ? k : best[be];
                }
            }
            if (a.mode == EPI_SWIGLU) s_part[re][0][be] = v;   // re-used below
        }
        if (a.mode == EPI_SWIGLU) {
            __syncthreads();
            // rows 2i (gate) and 2i+1 (up): act_i = silu(gate) * up
            if (tid < (R / 2) * NB) {
                const int pi = tid / NB, be = tid % NB;
                const int rg = tile * R + 2 * pi;
                if (rg + 1 < a.N && be < nb) {
                    const float g = s_part[2 * pi][0][be], u = s_part[2 * pi + 1][0][be];
                    a.out[(size_t)be * a.ldo + (rg >> 1)] = g / (1.f + __expf(-g)) * u;
                }
            }
        }
        __syncthreads();
    }

    if (a.mode == EPI_ARGMAX) {
        if (tid < R * NB) {
            const int be = tid % NB;
            if (be < nb) atomicMax(&s_key[be], best[be]);
        }
        __syncthreads();
        if (tid < nb) atomicMax(&a.keys[tid], s_key[tid]);
    }
}

template <int TPR>
static cudaError_t gemv_nb(const GemvArgs& a, cudaStream_t s, int grid) {
    const dim3 g(grid), b(GEMV_THREADS);
    if (a.x_add)   // batch-1 head over a residual held as two buffers (K <= 12288)
        return launch_k(k_gemv<TPR, 1, WF_BF16, true>, g, b, (size_t)a.K * 4, s, a);
    if (a.Wq) {
        if (a.nb <= 1) return launch_k(k_gemv<TPR, 1, WF_Q8>, g, b, 0, s, a);
        if (a.nb <= 2) return launch_k(k_gemv<TPR, 2, WF_Q8>, g, b, 0, s, a);
        if (a.nb <= 4) return launch_k(k_gemv<TPR, 4, WF_Q8>, g, b, 0, s, a);
        return launch_k(k_gemv<TPR, 8, WF_Q8>, g, b, 0, s, a);
    }
    if (a.w_f16) {
        if (a.nb <= 1) return launch_k(k_gemv<TPR, 1, WF_F16>, g, b, 0, s, a);
        if (a.nb <= 2) return launch_k(k_gemv<TPR, 2, WF_F16>, g, b, 0, s, a);
        if (a.nb <= 4) return launch_k(k_gemv<TPR, 4, WF_F16>, g, b, 0, s, a);
        return launch_k(k_gemv<TPR, 8, WF_F16>, g, b, 0, s, a);
    }
    if (a.nb <= 1) return launch_k(k_gemv<TPR, 1, WF_BF16>, g, b, 0, s, a);
    if (a.nb <= 2) return launch_k(k_gemv<TPR, 2, WF_BF16>, g, b, 0, s, a);
    if (a.nb <= 4) return launch_k(k_gemv<TPR, 4, WF_BF16>, g, b, 0, s, a);
    return launch_k(k_gemv<TPR, 8, WF_BF16>, g, b, 0, s, a);
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, int num_sms) {
    const int K8 = a.K >> 3;
    int tpr = 8;
    while (tpr * GEMV_MAXJ < K8) tpr <<= 1;   // <= 8 loads per thread
    // SwiGLU pairs rows 2i / 2i+1 inside one tile: at least two rows per tile
    // (model validation keeps K <= 8192 for that projection).
    if (a.mode == EPI_SWIGLU && tpr > 128) tpr = 128;
    const int R = GEMV_THREADS / tpr;
    const int tiles = (a.N + R - 1) / R;
    const int grid = tiles < num_sms * 8 ? tiles : num_sms * 8;
    switch (tpr) {
        case 8: return gemv_nb<8>(a, s, grid);
        case 16: return gemv_nb<16>(a, s, grid);
        case 32: return gemv_nb<32>(a, s, grid);
        case 64: return gemv_nb<64>(a, s, grid);
        case 128: return gemv_nb<128>(a, s, grid);
        default: return gemv_nb<256>(a, s, grid);
    }
}

// ========================================================= decode attention ==
// CTA (split s, kv head g, token b), 128 threads.  Keys [0, pos] are cut into
// at most gridDim.x splits of at least ATT_MIN_CHUNK keys (decided on the
// device from the token's position, so one launch shape serves every
// context length); each active split streams its K/V rows through shared
// memory in tiles of 64 and keeps an online softmax (running max m, sum l,
// output acc) per query head in the base-2 domain.  The last split to finish
// merges the partials (log-sum-exp rescale).
constexpr int ATT_THREADS = 128;
constexpr int ATT_TK = 64;
constexpr int ATT_MAXG = 16;
constexpr int ATT_MIN_CHUNK = 64;
constexpr int ATT_MAX_SPLITS = 32;

template <int D>
__global__ void __launch_bounds__(ATT_THREADS) k_attn_decode(AttnDecodeArgs a) {
    constexpr int H2 = D / 2;
    constexpr int KP = D + 2;   // padded K row (bf16 elements): conflict-free row reads
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = a.NH / a.NKV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    __shared__ float s_q[ATT_MAXG][D];
    __shared__ __align__(16) uint16_t s_k[ATT_TK][KP];
    __shared__ __align__(16) uint16_t s_v[ATT_TK][D];
    __shared__ float s_sc[ATT_MAXG][ATT_TK];   // scores; split statistics at the merge
    static_assert(ATT_MAXG * ATT_TK >= 2 * ATT_MAX_SPLITS * ATT_MAXG, "merge scratch");
    __shared__ float s_m[ATT_MAXG], s_l[ATT_MAXG], s_scale[ATT_MAXG];
    __shared__ float s_kv[2][D];
    __shared__ int s_last;

    pdl_trigger();
    pdl_wait();
    if (!a.tok_ok[b]) return;   // the embed kernel flagged this token
    const int pos = a.positions[b];
    const int seq = a.seqs[b];
    const int n_keys = pos + 1;
    int per = (n_keys + gridDim.x - 1) / gridDim.x;
    per = per < ATT_MIN_CHUNK ? ATT_MIN_CHUNK : per;
    const int S = (n_keys + per - 1) / per;   // active splits
    if (split >= S) return;
    const int lo = split * per;
    const int hi = min(n_keys, lo + per);
    const float* qkv = a.qkv + (size_t)b * a.ld_qkv;
    const float* cs = a.cos_t + (size_t)pos * H2;
    const float* sn = a.sin_t + (size_t)pos * H2;
    const size_t head_off = (((size_t)seq * a.L + a.layer) * a.NKV + g) * (size_t)a.max_len * D;
    uint16_t* kc = a.kc + head_off;
    uint16_t* vc = a.vc + head_off;
    // log2(e)/sqrt(D): scores in the base-2 domain
    const float qscale = 1.4426950408889634f * rsqrtf((float)D);

    // ---- q of the G heads: optional per-head RMSNorm, then RoPE ----
    for (int e = tid; e < G * D; e += ATT_THREADS) s_q[e / D][e % D] = qkv[(g * G) * D + e];
    for (int e = tid; e < 2 * D; e += ATT_THREADS) {
        const int which = e / D, d = e % D;   // 0: k, 1: v
        s_kv[which][d] = qkv[a.NH * D + which * a.NKV * D + g * D + d];
    }
    __syncthreads();
    if (a.q_norm) {   // PII-Tracer forward(): per-head RMSNorm before RoPE
        for (int h = warp; h < G + 1; h += ATT_THREADS / 32) {
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
    // RoPE of q (kept f32, pre-scaled) and of k (rounded to bf16 = the cache value)
    for (int e = tid; e < (G + 1) * H2; e += ATT_THREADS) {
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
    // The split that owns position pos writes the new K/V row before reading.
    if (pos >= lo && pos < hi) {
        for (int d = tid; d < D; d += ATT_THREADS) {
            kc[(size_t)pos * D + d] = f32_to_bf16(s_kv[0][d]);
            vc[(size_t)pos * D + d] = f32_to_bf16(s_kv[1][d]);
        }
    }
    if (tid < G) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    __syncthreads();

    // each thread owns output elements e = tid + i*128 of the [G][D] block
    constexpr int MAXE = (ATT_MAXG * D + ATT_THREADS - 1) / ATT_THREADS;
    float acc[MAXE];
#pragma unroll
    for (int i = 0; i < MAXE; ++i) acc[i] = 0.f;

    // K/V tiles are loaded into registers one tile ahead (all of a tile's
    // 16-byte loads in flight together) and stored to shared memory when
    // the tile's turn comes.
    constexpr int C8 = D / 8;
    constexpr int PER = (ATT_TK * C8 + ATT_THREADS - 1) / ATT_THREADS;
    uint4 kr[PER], vr[PER];
    auto load_tile = [&](int t0) {
        const int nt = min(ATT_TK, hi - t0);
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = tid + u * ATT_THREADS;
            if (e < nt * C8) {
                const int j = e / C8, cc = e % C8;
                kr[u] = __ldcg(reinterpret_cast<const uint4*>(kc + (size_t)(t0 + j) * D + cc * 8));
                vr[u] = __ldcg(reinterpret_cast<const uint4*>(vc + (size_t)(t0 + j) * D + cc * 8));
            }
        }
    };
    if (lo < hi) load_tile(lo);
    for (int t0 = lo; t0 < hi; t0 += ATT_TK) {
        const int nt = min(ATT_TK, hi - t0);
        // stage K (padded rows) and V from the registers, then fetch the next tile
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = tid + u * ATT_THREADS;
            if (e < nt * C8) {
                const int j = e / C8, cc = e % C8;
                uint32_t* kd = reinterpret_cast<uint32_t*>(&s_k[j][cc * 8]);
                kd[0] = kr[u].x; kd[1] = kr[u].y; kd[2] = kr[u].z; kd[3] = kr[u].w;
                *reinterpret_cast<uint4*>(&s_v[j][cc * 8]) = vr[u];
            }
        }
        __syncthreads();
        if (t0 + ATT_TK < hi) load_tile(t0 + ATT_TK);
        // scores: thread -> key j = tid % 64, heads h = tid/64, +2, ...
        {
            const int j = tid % ATT_TK;
            for (int h = tid / ATT_TK; h < G; h += ATT_THREADS / ATT_TK) {
                float sc = -INFINITY;
                if (j < nt) {
                    const uint32_t* kr = reinterpret_cast<const uint32_t*>(s_k[j]);
                    float dot = 0.f;
#pragma unroll 8
                    for (int d2 = 0; d2 < H2; ++d2) {
                        const uint32_t kk = kr[d2];
                        dot = fmaf(s_q[h][2 * d2], bf16_lo(kk), dot);
                        dot = fmaf(s_q[h][2 * d2 + 1], bf16_hi(kk), dot);
                    }
                    sc = dot;
                }
                s_sc[h][j] = sc;
            }
        }
        __syncthreads();
        // online softmax update, one warp per head
        for (int h = warp; h < G; h += ATT_THREADS / 32) {
            const float v0 = s_sc[h][lane], v1 = s_sc[h][lane + 32];
            const float tm = warp_max(fmaxf(v0, v1));
            const float mo = s_m[h];
            const float mn = fmaxf(mo, tm);
            const float p0 = exp2f(v0 - mn), p1 = exp2f(v1 - mn);
            const float ps = warp_sum(p0 + p1);
            s_sc[h][lane] = p0;
            s_sc[h][lane + 32] = p1;
            __syncwarp();
            if (lane == 0) {
                const float sc = exp2f(mo - mn);   // 0 when mo == -inf
                s_scale[h] = sc;
                s_l[h] = s_l[h] * sc + ps;
                s_m[h] = mn;
            }
        }
        __syncthreads();
        // acc = acc*scale + P V
#pragma unroll
        for (int i = 0; i < MAXE; ++i) {
            const int e = tid + i * ATT_THREADS;
            if (e < G * D) {
                const int h = e / D, d = e % D;
                float s = acc[i] * s_scale[h];
                for (int j = 0; j < nt; ++j) s = fmaf(s_sc[h][j], bf16_to_f32(s_v[j][d]), s);
                acc[i] = s;
            }
        }
        __syncthreads();
    }

    const size_t out0 = (size_t)b * a.NH * D + (size_t)(g * G) * D;
    if (S == 1) {   // a single split is already the answer
#pragma unroll
        for (int i = 0; i < MAXE; ++i) {
            const int e = tid + i * ATT_THREADS;
            if (e < G * D) {
                const float o = acc[i] / s_l[e / D];
                if (a.att_b) {
                    bool bad = false;
                    a.att_b[out0 + e] = f32_to_f16_chk(o, bad);
                    if (bad) raise_status(a.status, EMBER_ERR_RANGE);
                }
                else a.att[out0 + e] = o;
            }
        }
        return;
    }

    // ---- write this split's partial (m, l, acc) ----
    float* part = a.part + ((((size_t)b * a.NKV + g) * ATT_MAX_SPLITS + split) * G) * (D + 2);
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = tid + i * ATT_THREADS;
        if (e < G * D) part[(size_t)(e / D) * (D + 2) + 2 + (e % D)] = acc[i];
    }
    if (tid < G) {
        part[(size_t)tid * (D + 2) + 0] = s_m[tid];
        part[(size_t)tid * (D + 2) + 1] = s_l[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned done = atomicAdd(&a.counters[b * a.NKV + g], 1u);
        s_last = (done == (unsigned)(S - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last split: merge the S partials.  All (m, l) pairs are fetched in
    // one parallel pass, then every output element sums S independent loads.
    const float* pb = a.part + (((size_t)b * a.NKV + g) * ATT_MAX_SPLITS) * G * (D + 2);
    float* s_pm = &s_sc[0][0];                       // [S][G] maxima, then weights
    float* s_pl = &s_sc[0][0] + ATT_MAX_SPLITS * ATT_MAXG;   // [S][G] sums
    for (int e = tid; e < S * G; e += ATT_THREADS) {
        const float* ps = pb + (size_t)e * (D + 2);
        s_pm[e] = __ldcg(ps);
        s_pl[e] = __ldcg(ps + 1);
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < S; ++s2)
            if (s_pl[s2 * G + tid] > 0.f) M = fmaxf(M, s_pm[s2 * G + tid]);
        float L = 0.f;
        for (int s2 = 0; s2 < S; ++s2) {
            const float l = s_pl[s2 * G + tid];
            const float f = l > 0.f ? exp2f(s_pm[s2 * G + tid] - M) : 0.f;   // empty: nothing
            s_pm[s2 * G + tid] = f;
            L += l * f;
        }
        s_scale[tid] = 1.f / L;
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += ATT_THREADS) {
        const int h = e / D, d = e % D;
        float O = 0.f;
#pragma unroll 4
        for (int s2 = 0; s2 < S; ++s2)
            O = fmaf(__ldcg(pb + ((size_t)s2 * G + h) * (D + 2) + 2 + d), s_pm[s2 * G + h], O);
        O *= s_scale[h];
        if (a.att_b) {
            bool bad = false;
            a.att_b[out0 + e] = f32_to_f16_chk(O, bad);
            if (bad) raise_status(a.status, EMBER_ERR_RANGE);
        }
        else a.att[out0 + e] = O;
    }
    if (tid == 0) a.counters[b * a.NKV + g] = 0u;
}

void launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t s) {
    if (a.k_map && a.v_map && attn_decode_mma_supported(a.D, a.NH / a.NKV)) {
        launch_attn_decode_mma(a, s);
        return;
    }
    dim3 grid(a.splits < ATT_MAX_SPLITS ? a.splits : ATT_MAX_SPLITS, a.NKV, a.nb);
    switch (a.D) {
        case 16: launch_k(k_attn_decode<16>, grid, dim3(ATT_THREADS), 0, s, a); break;
        case 32: launch_k(k_attn_decode<32>, grid, dim3(ATT_THREADS), 0, s, a); break;
        case 64: launch_k(k_attn_decode<64>, grid, dim3(ATT_THREADS), 0, s, a); break;
        case 128: launch_k(k_attn_decode<128>, grid, dim3(ATT_THREADS), 0, s, a); break;
        default: break;   // rejected by model validation
    }
}

// ================================================================== finish ==
__global__ void k_finish(FinishArgs a) {
    const int b = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    if (b < a.nb) {
        if (a.argmax) a.argmax[b] = argmax_key_index(a.keys[b]);
        a.keys[b] = 0ull;
        if (a.seqs && a.tok_ok[b]) a.cursor[a.seqs[b]] = a.positions[b] + 1;
    }
    if (b == 0 && a.pf_seq >= 0) a.cursor[a.pf_seq] = a.pf_end;
}

void launch_finish(const FinishArgs& a, cudaStream_t s) {
    const int th = a.nb < 32 ? 32 : ((a.nb + 31) / 32) * 32;
    launch_k(k_finish, dim3(1), dim3(th), 0, s, a);
}

// Set one sequence's cursor (value passed by argument: capturable, no host buffer).
__global__ void k_set_cursor(int32_t* cursor, int seq, int pos) { cursor[seq] = pos; }

void launch_set_cursor(int32_t* cursor, int seq, int pos, cudaStream_t s) {
    count_launches(1);
    k_set_cursor<<<1, 1, 0, s>>>(cursor, seq, pos);
}

// ================================================================ repack ==
__global__ void k_bf16_to_f32(const uint16_t* in, float* out, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        out[i] = bf16_to_f32(in[i]);
}

__global__ void k_bf16_to_f16(uint16_t* p, long long n, float scale) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        p[i] = f32_to_f16(bf16_to_f32(p[i]) * scale);
}

void launch_bf16_to_f16_inplace(uint16_t* p, long long n, int exp, cudaStream_t s) {
    if (n <= 0) return;
    count_launches(1);
    long long blocks = (n + 255) / 256;
    k_bf16_to_f16<<<(int)(blocks < 8192 ? blocks : 8192), 256, 0, s>>>(p, n, std::ldexp(1.f, -exp));
}

// q8_0 block quantization of n bf16 values (n % 32 == 0), one warp per block
// of 32: amax = max |x|; the codes are x / (amax / 127) in f32 rounded to the
// nearest integer (ties to even) and clamped to [-127, 127], zero for a block
// of zeros; the block's scale is amax / 127 stored as f16 (nearest even).
// Decoding is q * d ("ember internals", q8_0 block format).  With f16_out
// set, the decoded value times f16_scale is written there as f16 (in place of
// the bf16 input when f16_out == p): the tensor-core GEMMs' copy of the
// quantized matrix.
__global__ void k_q8_0_quantize(const uint16_t* p, long long n, int8_t* q, uint16_t* d, uint16_t* f16_out,
                                float f16_scale) {
    const long long stride = (long long)gridDim.x * blockDim.x;   // a multiple of 32
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
        // n % 32 == 0: the 32 lanes of a warp are all in range or all out
        const float x = bf16_to_f32(p[i]);
        float amax = fabsf(x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, o));
        const float d32 = __fdiv_rn(amax, 127.f);
        float c = d32 > 0.f ? rintf(__fdiv_rn(x, d32)) : 0.f;
        c = fminf(fmaxf(c, -127.f), 127.f);
        q[i] = (int8_t)c;
        const __half dh = __float2half_rn(d32);
        if ((threadIdx.x & 31) == 0) d[i >> 5] = __half_as_ushort(dh);
        if (f16_out) f16_out[i] = f32_to_f16(c * __half2float(dh) * f16_scale);
    }
}

void launch_q8_0_quantize(const uint16_t* p, long long n, int8_t* q, uint16_t* d, uint16_t* f16_out,
                          int f16_exp, cudaStream_t s) {
    if (n <= 0) return;
    count_launches(1);
    long long blocks = (n + 255) / 256;
    k_q8_0_quantize<<<(int)(blocks < 8192 ? blocks : 8192), 256, 0, s>>>(p, n, q, d, f16_out,
                                                                         std::ldexp(1.f, -f16_exp));
}

// out = max |p[i]| over n bf16 values, as f32 bits (non-negative floats order
// like their bits); NaN entries are skipped
__global__ void k_absmax_bf16(const uint16_t* p, long long n, unsigned* out) {
    unsigned m = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const unsigned b = ((unsigned)p[i] & 0x7FFFu) << 16;
        if (b <= 0x7F800000u) m = b > m ? b : m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned t = __shfl_xor_sync(FULL_MASK, m, o);
        m = t > m ? t : m;
    }
    if ((threadIdx.x & 31) == 0) atomicMax(out, m);
}

void launch_absmax_bf16(const uint16_t* p, long long n, unsigned* out, cudaStream_t s) {
    if (n <= 0) return;
    count_launches(1);
    long long blocks = (n + 255) / 256;
    k_absmax_bf16<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(p, n, out);
}

void launch_bf16_to_f32(const uint16_t* in, float* out, long long n, cudaStream_t s) {
    count_launches(1);
    if (n <= 0) return;
    long long blocks = (n + 255) / 256;
    k_bf16_to_f32<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(in, out, n);
}

}  // namespace ember
