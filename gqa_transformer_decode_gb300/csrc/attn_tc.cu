// attn_tc.cu -- whole-prompt GQA attention on the tcgen05 tensor cores.
//
// One CTA = 128 query rows of one query head h (kv head g = h / G: ember
// internals "grouped-query attention").  Per key tile of 128 keys:
//   S = Q . K^T                  tcgen05.mma M=128, N=128, K=D  -> TMEM (f16 Q and K)
//   softmax rows (online)        8 warps: query row r is two threads, one per 64 score columns
//   P -> shared memory           f16, the 128-byte-swizzled K-major A operand
//   O += P . V                   tcgen05.mma (f16) M=128, N=D, K=128, accumulating
//                                in TMEM across all key tiles
// The running row maximum m only moves when a tile's maximum exceeds it by
// more than 2^8 (lazy rescaling): the row's thread then multiplies its O
// columns in TMEM by exp2(m_old - m_new) after the previous P . V is done,
// and l with it.  Every term stays <= 2^8 before the final O / l, far from
// f32 overflow, and the result is the same softmax.
// Causal rows see keys at positions <= their own (LowLlamaBasic reference.py
// self_attn()); the bidirectional encoder sees every key of its sequence
// (PII-Tracer-vLLM forward()).  Q rows come from the RoPE'd f16 queries; K
// and V from f16 copies of the bf16 cache (or the encoder's K / V buffers)
// that k_vt16 writes before the attention: Kh [kv head][keys][D] and the
// transposed Vt [kv head][D][keys], K-major for the MMA (bf16 -> f16 is exact
// for these magnitudes; P in [0, 1] keeps 11 bits instead of bf16's 8).
// Warp 0: TMA producer (Q once; Kh and Vt through a ring of 4 stages for
// head_dim 64, 2 for 128); warp 1: TMEM allocation and the MMA issuer;
// warps 2-9: softmax and output.  Every
// mbarrier wait is bounded; a timeout raises EMBER_ERR_TIMEOUT and the CTA
// drains its copies and frees TMEM.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace ember {

constexpr int AT_THREADS = 320;   // producer, MMA issuer, 8 softmax warps
constexpr int AT_BQ = 128;   // query rows per CTA
constexpr int AT_BK = 128;   // keys per tile

template <int D>
struct AtSmem {
    static constexpr int KB = D / 64;                    // 64-element K blocks of Q / K rows
    static constexpr int Q_BYTES = KB * AT_BQ * 128;
    static constexpr int NSTG = D == 64 ? 4 : 2;        // K/V ring stages (shared memory bound)
    static constexpr int K_BYTES = KB * AT_BK * 128;     // one stage
    static constexpr int V_BLOCK = D * 128;              // [D rows][64 keys] f16
    static constexpr int V_BYTES = 2 * V_BLOCK;          // one stage: 128 keys
    static constexpr int P_BYTES = 2 * AT_BQ * 128;      // [128 rows][128 keys] f16
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NSTG * K_BYTES;
    static constexpr int OFF_P = OFF_V + NSTG * V_BYTES;
    static constexpr int OFF_BAR = OFF_P + P_BYTES;
    static constexpr int TOTAL = OFF_BAR + 256 + 1024;   // + barriers, + alignment slack
    static constexpr uint32_t TMEM_COLS = (128 + D) <= 256 ? 256 : 512;
};

template <int D>
__global__ void __launch_bounds__(AT_THREADS, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, AttnTcArgs a) {
    using L = AtSmem<D>;
    extern __shared__ uint8_t at_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    constexpr int NSTG = L::NSTG;
    uint64_t* q_full = bar + 0;
    uint64_t* s_full = bar + 1;
    uint64_t* p_full = bar + 2;
    uint64_t* o_full = bar + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);
    int* sflag = reinterpret_cast<int*>(bar + 5);   // [0] failed, [1] issued, [2] consumed
    uint64_t* kv_full = bar + 8;    // [NSTG]
    uint64_t* kv_empty = bar + 12;  // [NSTG]
    uint64_t* xb = bar + 20;        // [4] the two softmax halves of a TMEM lane quarter
    __shared__ float s_mx[2][2][AT_BQ];   // [tile parity][half][row] maxima
    __shared__ float s_lh[2][AT_BQ];      // [half][row] final sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = gridDim.x - 1 - blockIdx.x;        // heaviest (last) query tiles first
    const int h = blockIdx.y, z = blockIdx.z;
    const int g = h / a.G;
    const int vz = z * a.NKV + g;                     // Kh and Vt rows of this kv head
    const int q_first = qt * AT_BQ;                    // first query row within the sequence
    const int q_last = min(a.T_per_seq, q_first + AT_BQ) - 1;
    const int nkt = a.causal ? (a.pos0 + q_last) / AT_BK + 1 : (a.n_keys + AT_BK - 1) / AT_BK;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NSTG; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, 256);
        for (int q = 0; q < 4; ++q) mbar_init(&xb[q], 64);
        mbar_init(o_full, 1);
        sflag[0] = 0;
        sflag[1] = 0;
        sflag[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(L::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 128;
    pdl_wait();   // Q, K and Vt are the previous kernels' outputs

    if (warp == 0) {   // ------------------------------------------ TMA producer
        // Up to NSTG tiles are in flight; tile j + NSTG is issued once the
        // MMAs of tile j have freed its stage.
        if (lane == 0) {
            auto issue = [&](int j) {
                const int s = j % NSTG;
                mbar_expect_tx(&kv_full[s], L::K_BYTES + L::V_BYTES);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_3d(sm + L::OFF_K + s * L::K_BYTES + kb * AT_BK * 128, &tmK, kb * 64,
                                j * AT_BK, vz, &kv_full[s]);
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_3d(sm + L::OFF_V + s * L::V_BYTES + kb * L::V_BLOCK, &tmV,
                                j * AT_BK + kb * 64, 0, vz, &kv_full[s]);
            };
            const int qrow0 = z * a.T_per_seq + q_first;
            mbar_expect_tx(q_full, L::Q_BYTES);
            for (int kb = 0; kb < L::KB; ++kb)
                tma_load_2d(sm + L::OFF_Q + kb * AT_BQ * 128, &tmQ, h * D + kb * 64, qrow0, q_full);
            int issued = 0;
            for (; issued < NSTG && issued < nkt; ++issued) issue(issued);
            bool fail = false;
            for (; issued < nkt; ++issued) {   // stage of tile issued - NSTG -> tile issued
                const int j = issued - NSTG;
                if (!mbar_wait(&kv_empty[j % NSTG], (uint32_t)(j / NSTG) & 1u)) {
                    fail = true;
                    break;
                }
                issue(issued);
            }
            if (fail) sflag[0] = 1;
            sflag[1] = issued;
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ------------------------------------------ MMA issuer
            constexpr uint32_t idS = idesc_f16(AT_BQ, AT_BK);   // f16 queries and keys
            constexpr uint32_t idO = idesc_f16(AT_BQ, D);
            bool ok = mbar_wait(q_full, 0);
            int j = 0;
            for (; ok && j < nkt; ++j) {
                const int s = j % NSTG;
                const uint32_t u = (uint32_t)(j / NSTG);
                if (!mbar_wait(&kv_full[s], u & 1u)) break;
                tc_fence_after();
                const uint32_t q0 = smem_u32(sm + L::OFF_Q);
                const uint32_t k0 = smem_u32(sm + L::OFF_K + s * L::K_BYTES);
#pragma unroll
                for (int kb = 0; kb < L::KB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(tS, sdesc_sw128(q0 + kb * AT_BQ * 128 + k * 32),
                                  sdesc_sw128(k0 + kb * AT_BK * 128 + k * 32), idS,
                                  (kb | k) ? 1u : 0u);
                umma_commit(s_full);
                // O += P . V once the softmax warps have written P (and rescaled O)
                if (!mbar_wait(p_full, (uint32_t)j & 1u)) break;
                tc_fence_after();
                const uint32_t p0 = smem_u32(sm + L::OFF_P);
                const uint32_t v0 = smem_u32(sm + L::OFF_V + s * L::V_BYTES);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(tO, sdesc_sw128(p0 + kb * AT_BQ * 128 + k * 32),
                                  sdesc_sw128(v0 + kb * L::V_BLOCK + k * 32), idO,
                                  (j | kb | k) ? 1u : 0u);
                umma_commit(o_full);
                umma_commit(&kv_empty[s]);
            }
            if (j < nkt) sflag[0] = 1;
            sflag[2] = j;
        }
    } else {   // ------------------------------------------------ softmax warps
        // Eight warps: thread = (query row, half); half 0 takes score columns
        // 0-63 and O columns 0..D/2-1, half 1 the rest.  The two threads of a
        // row exchange their halves' maxima through shared memory (pair
        // mbarrier xb[quarter], 64 arrivals per tile).  O accumulates in TMEM
        // across key tiles; the row keeps a reference maximum m and rescales O
        // (and l) only when a tile's maximum exceeds m by more than RESCALE
        // (log2 units), so p = 2^(s - m) stays <= 2^RESCALE (f16-safe).  The
        // rescale is a TMEM read-scale-write after the previous P.V completed.
        constexpr float RESCALE = 8.f;
        constexpr int DH = D / 2;
        const int qw = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = qw * 32 + lane;                 // query row within the tile
        const int qp = a.pos0 + q_first + r;          // its position
        const int qmin = a.pos0 + q_first;            // the tile's first position
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const int cs0 = half * 64;                    // this half's score columns
        const int co0 = half * DH;                    // this half's O columns
        const float sc_log2 = 1.4426950408889634f * rsqrtf((float)D);
        float m = -INFINITY, l = 0.f;
        uint8_t* sP = sm + L::OFF_P;
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            if (!mbar_wait(s_full, (uint32_t)j & 1u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key0 = j * AT_BK;
            const bool full = key0 + AT_BK <= a.n_keys && (!a.causal || key0 + AT_BK - 1 <= qmin);
            // pass 1: this half's 64 scores (kept in registers) and their maximum
            uint32_t v[64];
            tmem_ld32(tS + lane_off + cs0, v);
            tmem_ld32(tS + lane_off + cs0 + 32, v + 32);
            tmem_ld_wait();
            float mt = -INFINITY;
            if (full) {
#pragma unroll
                for (int i = 0; i < 64; ++i) mt = fmaxf(mt, __uint_as_float(v[i]));
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int kp = key0 + cs0 + i;
                    const bool vis = kp < a.n_keys && (!a.causal || kp <= qp);
                    if (!vis) v[i] = __float_as_uint(-INFINITY);
                    mt = fmaxf(mt, __uint_as_float(v[i]));
                }
            }
            s_mx[j & 1][half][r] = mt;
            mbar_arrive(&xb[qw]);
            if (!mbar_wait(&xb[qw], (uint32_t)j & 1u)) {
                ok = false;
                break;
            }
            mt = fmaxf(s_mx[j & 1][0][r], s_mx[j & 1][1][r]) * sc_log2;
            // reference maximum: move it (and rescale O, l) only when it falls behind
            const bool move = mt > m + RESCALE;
            const float mref = move ? mt : m;
            const float corr = (m == -INFINITY) ? 0.f : exp2f(m - mref);   // 1 when not moving
            if (j > 0) {   // PV(j-1) must be complete before O is touched or P is rewritten
                if (!mbar_wait(o_full, (uint32_t)(j - 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(FULL_MASK, move)) {
#pragma unroll
                    for (int c0 = 0; c0 < DH; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + lane_off + co0 + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st16(tO + lane_off + co0 + c0, o);
                        tmem_st16(tO + lane_off + co0 + c0 + 16, o + 16);
                    }
                    tmem_st_wait();
                }
            }
            l *= corr;
            m = mref;
            // pass 2: p = 2^(s - m) (masked scores are -inf: p = 0), row sum,
            // P -> shared (K-major block `half`, 128-byte swizzle)
            float rs = 0.f;
#pragma unroll
            for (int h32 = 0; h32 < 64; h32 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float p0 = ex2(fmaf(__uint_as_float(v[h32 + i]), sc_log2, -m));
                    const float p1 = ex2(fmaf(__uint_as_float(v[h32 + i + 1]), sc_log2, -m));
                    rs += p0 + p1;
                    pk[i / 2] = pack_f16x2(p0, p1);
                }
                uint8_t* rowp = sP + half * AT_BQ * 128 + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int chunk = h32 / 8 + t;
                    *reinterpret_cast<uint4*>(rowp + ((chunk ^ (r & 7)) * 16)) =
                        make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            mbar_arrive(p_full);
            l += rs;
        }
        // the row's sum over both halves (one more phase of the pair barrier)
        if (ok) {
            s_lh[half][r] = l;
            mbar_arrive(&xb[qw]);
            if (!mbar_wait(&xb[qw], (uint32_t)nkt & 1u)) ok = false;
        }
        if (ok && nkt > 0 && !mbar_wait(o_full, (uint32_t)(nkt - 1) & 1u)) ok = false;
        if (!ok) sflag[0] = 1;
        tc_fence_after();
        if (ok) {
            const float inv = 1.f / (s_lh[0][r] + s_lh[1][r]);
            const bool live = q_first + r < a.T_per_seq;
            uint16_t* out = a.att + (size_t)(z * a.T_per_seq + q_first + r) * a.ld_att + h * D + co0;
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + lane_off + co0 + c0, o);
                tmem_ld_wait();
                if (live) {
                    bool bad = false;
#pragma unroll
                    for (int d = 0; d < 32; d += 8) {
                        uint4 w;
                        w.x = pack_f16x2_chk(__uint_as_float(o[d]) * inv, __uint_as_float(o[d + 1]) * inv, bad);
                        w.y = pack_f16x2_chk(__uint_as_float(o[d + 2]) * inv, __uint_as_float(o[d + 3]) * inv, bad);
                        w.z = pack_f16x2_chk(__uint_as_float(o[d + 4]) * inv, __uint_as_float(o[d + 5]) * inv, bad);
                        w.w = pack_f16x2_chk(__uint_as_float(o[d + 6]) * inv, __uint_as_float(o[d + 7]) * inv, bad);
                        *reinterpret_cast<uint4*>(out + c0 + d) = w;
                    }
                    if (bad) raise_status(a.status, EMBER_ERR_RANGE);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && sflag[0]) raise_status(a.status, EMBER_ERR_TIMEOUT);
    if (warp == 0 && lane == 0 && sflag[0]) {
        // drain K/V copies issued but never consumed by the MMA warp
        for (int j = sflag[2]; j < sflag[1]; ++j)
            (void)mbar_wait(&kv_full[j % NSTG], (uint32_t)(j / NSTG) & 1u);
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(L::TMEM_COLS));
    }
}

// Vt[z][d][key] = f16(V[z][key][d]) and Kh[z][key][d] = f16(K[z][key][d]);
// zero past n_keys.
__global__ void __launch_bounds__(256) k_vt(VtArgs a) {
    __shared__ uint16_t tile[64][129];   // [key][d], padded
    const int z = blockIdx.y;
    const int key0 = blockIdx.x * 64;
    const int D = a.D;
    pdl_trigger();
    pdl_wait();
    const uint16_t* src =
        a.v + (size_t)(z / a.nkv) * a.v_z_stride + (size_t)(z % a.nkv) * a.v_h_stride;
    for (int e = threadIdx.x; e < 64 * D; e += blockDim.x) {
        const int k = e / D, d = e % D;
        tile[k][d] = (key0 + k < a.n_keys) ? src[(size_t)(key0 + k) * D + d] : (uint16_t)0;
    }
    __syncthreads();
    uint16_t* dst = a.vt + (size_t)z * D * a.keys_pad;
    for (int e = threadIdx.x; e < 64 * D; e += blockDim.x) {
        const int d = e / 64, k = e % 64;
        if (key0 + k < a.keys_pad)
            dst[(size_t)d * a.keys_pad + key0 + k] =
                __half_as_ushort(__float2half_rn(bf16_to_f32(tile[k][d])));
    }
    if (a.kh) {
        const uint16_t* ks =
            a.k + (size_t)(z / a.nkv) * a.v_z_stride + (size_t)(z % a.nkv) * a.v_h_stride;
        uint16_t* kd = a.kh + (size_t)z * a.keys_pad * D;
        for (int e = threadIdx.x; e < 64 * D; e += blockDim.x) {
            const int k = e / D, d = e % D;
            const int key = key0 + k;
            if (key < a.keys_pad && (key < a.kh_from || key >= a.n_keys))
                kd[(size_t)key * D + d] =
                    key < a.n_keys ? __half_as_ushort(__float2half_rn(bf16_to_f32(ks[(size_t)key * D + d])))
                                   : (uint16_t)0;
        }
    }
}

// The same for D % 8 == 0, D <= 128, with 16-byte accesses on both sides:
// key rows in as 8-value chunks, f16 tile [64 keys][D] (row pitch D + 8),
// 8-key runs of one column out.
__global__ void __launch_bounds__(256) k_vt16(VtArgs a) {
    __shared__ __align__(16) uint16_t tile[64][136];
    const int z = blockIdx.y;
    const int key0 = blockIdx.x * 64;
    const int D = a.D, C8 = D / 8;
    pdl_trigger();
    pdl_wait();
    const uint16_t* src =
        a.v + (size_t)(z / a.nkv) * a.v_z_stride + (size_t)(z % a.nkv) * a.v_h_stride;
    for (int e = threadIdx.x; e < 64 * C8; e += blockDim.x) {
        const int k = e / C8, c = e % C8;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (key0 + k < a.n_keys) {
            const uint4 b = *reinterpret_cast<const uint4*>(src + (size_t)(key0 + k) * D + 8 * c);
            u = make_uint4(pack_f16x2(bf16_lo(b.x), bf16_hi(b.x)), pack_f16x2(bf16_lo(b.y), bf16_hi(b.y)),
                           pack_f16x2(bf16_lo(b.z), bf16_hi(b.z)), pack_f16x2(bf16_lo(b.w), bf16_hi(b.w)));
        }
        *reinterpret_cast<uint4*>(&tile[k][8 * c]) = u;
    }
    __syncthreads();
    uint16_t* dst = a.vt + (size_t)z * D * a.keys_pad;
    for (int e = threadIdx.x; e < D * 8; e += blockDim.x) {
        const int d = e / 8, kc = e % 8;   // column d, keys 8kc..8kc+7 of the block
        if (key0 + 8 * kc >= a.keys_pad) continue;   // keys_pad % 8 == 0: whole runs
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = (uint32_t)tile[8 * kc + 2 * j][d] | ((uint32_t)tile[8 * kc + 2 * j + 1][d] << 16);
        *reinterpret_cast<uint4*>(dst + (size_t)d * a.keys_pad + key0 + 8 * kc) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (a.kh) {   // the K rows of the block, converted in 16-byte chunks
        const uint16_t* ks =
            a.k + (size_t)(z / a.nkv) * a.v_z_stride + (size_t)(z % a.nkv) * a.v_h_stride;
        uint16_t* kd = a.kh + (size_t)z * a.keys_pad * D;
        for (int e = threadIdx.x; e < 64 * C8; e += blockDim.x) {
            const int k = e / C8, c = e % C8;
            if (key0 + k >= a.keys_pad) continue;
            if (key0 + k >= a.kh_from && key0 + k < a.n_keys) continue;   // written by the RoPE kernel
            uint4 u = make_uint4(0, 0, 0, 0);
            if (key0 + k < a.n_keys) {
                const uint4 b = *reinterpret_cast<const uint4*>(ks + (size_t)(key0 + k) * D + 8 * c);
                u = make_uint4(pack_f16x2(bf16_lo(b.x), bf16_hi(b.x)), pack_f16x2(bf16_lo(b.y), bf16_hi(b.y)),
                               pack_f16x2(bf16_lo(b.z), bf16_hi(b.z)), pack_f16x2(bf16_lo(b.w), bf16_hi(b.w)));
            }
            *reinterpret_cast<uint4*>(kd + (size_t)(key0 + k) * D + 8 * c) = u;
        }
    }
}

void launch_vt(const VtArgs& a, int zs, cudaStream_t s) {
    if (a.D % 8 == 0 && a.D <= 128 && a.keys_pad % 8 == 0)
        launch_k(k_vt16, dim3((a.keys_pad + 63) / 64, zs), dim3(256), 0, s, a);
    else
        launch_k(k_vt, dim3((a.keys_pad + 63) / 64, zs), dim3(256), 0, s, a);
}

template <int D>
static void launch_at(const void* mq, const void* mk, const void* mv, const AttnTcArgs& a, int nseq,
                      cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AtSmem<D>::TOTAL);
        attr = true;
    }
    dim3 grid((a.T_per_seq + AT_BQ - 1) / AT_BQ, a.NH, nseq);
    launch_k(k_attn_tc<D>, grid, dim3(AT_THREADS), AtSmem<D>::TOTAL, s,
             *reinterpret_cast<const CUtensorMap*>(mq), *reinterpret_cast<const CUtensorMap*>(mk),
             *reinterpret_cast<const CUtensorMap*>(mv), a);
}

bool attn_tc_supported(int D) { return D == 64 || D == 128; }

void launch_attn_tc(const void* map_q, const void* map_k, const void* map_vt, const AttnTcArgs& a,
                    int nseq, int D, cudaStream_t s) {
    // more than one query tile per sequence: two tiles per CTA in ping-pong
    if (a.T_per_seq > AT_BQ) launch_attn_tc2(map_q, map_k, map_vt, a, nseq, D, s);
    else if (D == 64) launch_at<64>(map_q, map_k, map_vt, a, nseq, s);
    else if (D == 128) launch_at<128>(map_q, map_k, map_vt, a, nseq, s);
}

}  // namespace ember
