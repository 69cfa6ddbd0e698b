// attn_tc2.cu -- whole-prompt GQA attention for head_dim 64 and 128 on the
// tcgen05 tensor cores, two query tiles per CTA in ping-pong.
//
// The same computation as k_attn_tc (attn_tc.cu): per key tile of 128 keys,
// S = Q . K^T into TMEM, the online softmax of each query row, P (f16) and
// O += P . V accumulated in TMEM, with the lazy rescaling of O and l when a
// row's maximum moves by more than 2^8.  What differs is the schedule, and
// that P stays in tensor memory (the A operand of P . V read from TMEM).
// One CTA holds two 128-row query tiles A and B of one head, each with its
// own four softmax warps (one thread per query row, all 128 score columns)
// and its own S, P and O columns of TMEM, and the MMA warp interleaves them
// (head_dim 64):
//     S_A(j+1), PV_A(j)   while the B warps turn S_B(j) into P_B(j)
//     S_B(j+1), PV_B(j)   while the A warps turn S_A(j+1) into P_A(j+1)
// so the tensor cores work on one tile while the CUDA cores exponentiate the
// other (with one tile per CTA the two alternate and each idles while the
// other runs).  S of the next key tile goes ahead of P . V of this one: a
// softmax warp computes its row's P in registers while P . V(j) still reads
// the TMEM copy of P(j), and writes P(j + 1) there once that is done.  (A
// tcgen05.mma of M = 128, K = 16 takes ~112 cycles whatever N <= 128, so the
// N = 64 P . V costs twice the N = 128 S and the tensor pipe sets the pace.)
// With head_dim 128 the four accumulators fill the 512 TMEM columns, so P
// is written over the first half of its tile's S columns and the order is
// PV_t(j), S_t(j + 1) (the MMAs of one thread run in issue order, and S_t(j)
// complete implies PV_t(j - 1) complete).  Both tiles walk the key tiles of tile B (the later one); the
// causal mask zeroes tile A's share of the last one.
// Warp 0: TMA producer (f16 Q, the f16 copy Kh of the keys and the
// transposed Vt, as k_attn_tc reads them); warp 1:
// TMEM allocation and MMA issue; warps 2-5: tile A; warps 6-9: tile B (a
// warp reads the TMEM lanes of its index mod 4, so each group of four covers
// its tile's 128 rows).  Every mbarrier wait is bounded; a timeout raises
// EMBER_ERR_TIMEOUT and the CTA drains its copies and frees TMEM.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace ember {

namespace {

constexpr int P2_THREADS = 320;
constexpr int P2_BQ = 128;    // query rows per tile (two tiles per CTA)
constexpr int P2_BK = 128;    // keys per tile

template <int D>
struct P2Smem {
    static constexpr int KB = D / 64;                   // 64-element blocks of a Q / K row
    static constexpr int TILE = KB * P2_BQ * 128;       // one query tile: KB swizzled [128][64] blocks
    static constexpr int NSTG = D == 64 ? 4 : 2;        // K/V ring stages
    static constexpr int K_BYTES = KB * P2_BK * 128;    // 128 keys x D f16
    static constexpr int V_BLOCK = D * 128;             // [D dims][64 keys] f16
    static constexpr int V_BYTES = 2 * V_BLOCK;         // 128 keys
    static constexpr int OFF_Q = 0;                     // Q_A, Q_B
    static constexpr int OFF_K = OFF_Q + 2 * TILE;
    static constexpr int OFF_V = OFF_K + NSTG * K_BYTES;
    static constexpr int OFF_BAR = OFF_V + NSTG * V_BYTES;
    static constexpr int TOTAL = OFF_BAR + 256 + 1024;     // + barriers, + alignment slack
    // TMEM columns: S_A, S_B (128 f32 each), O_A, O_B (D f32 each); P_A, P_B
    // (128 f16 each, packed two to a column) in their own columns for head_dim
    // 64, over the first half of S_A / S_B for 128
    static constexpr bool ALIAS = D == 128;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_O = 256;
    static constexpr uint32_t col_p(int t) { return ALIAS ? COL_S + t * 128 : 384 + t * 64; }
};

template <int D>
__global__ void __launch_bounds__(P2_THREADS, 1)
    k_attn_tc2(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, AttnTcArgs a) {
    using L = P2Smem<D>;
    constexpr int NSTG = L::NSTG;
    extern __shared__ uint8_t p2_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p2_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
    uint64_t* q_full = bar + 0;
    uint64_t* s_full = bar + 1;     // [2] per tile
    uint64_t* p_full = bar + 3;     // [2]
    uint64_t* o_full = bar + 5;     // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 7);
    int* sflag = reinterpret_cast<int*>(bar + 8);   // [0] failed, [1] issued, [2] consumed
    uint64_t* kv_full = bar + 10;   // [NSTG]
    uint64_t* kv_empty = bar + 16;  // [NSTG]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pt = gridDim.x - 1 - blockIdx.x;         // heaviest (last) tile pairs first
    const int h = blockIdx.y, z = blockIdx.z;
    const int g = h / a.G;
    const int vz = z * a.NKV + g;                      // Kh and Vt rows of this kv head
    const int q_first = pt * 2 * P2_BQ;                 // tile A's first row; tile B at + 128
    const int q_last = min(a.T_per_seq, q_first + 2 * P2_BQ) - 1;
    const int nkt = a.causal ? (a.pos0 + q_last) / P2_BK + 1 : (a.n_keys + P2_BK - 1) / P2_BK;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 128);
            mbar_init(&o_full[t], 1);
        }
        for (int s = 0; s < NSTG; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
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
    pdl_wait();   // Q, K and Vt are the previous kernels' outputs

    if (warp == 0) {   // ------------------------------------------ TMA producer
        if (lane == 0) {
            auto issue = [&](int j) {
                const int s = j % NSTG;
                mbar_expect_tx(&kv_full[s], L::K_BYTES + L::V_BYTES);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_3d(sm + L::OFF_K + s * L::K_BYTES + kb * P2_BK * 128, &tmK, kb * 64, j * P2_BK, vz,
                                &kv_full[s]);
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_3d(sm + L::OFF_V + s * L::V_BYTES + kb * L::V_BLOCK, &tmV,
                                j * P2_BK + kb * 64, 0, vz, &kv_full[s]);
            };
            const int qrow0 = z * a.T_per_seq + q_first;
            mbar_expect_tx(q_full, 2 * L::TILE);
            for (int t = 0; t < 2; ++t)
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_2d(sm + L::OFF_Q + t * L::TILE + kb * P2_BQ * 128, &tmQ, h * D + kb * 64,
                                qrow0 + t * P2_BQ, q_full);
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
            constexpr uint32_t idS = idesc_f16(P2_BQ, P2_BK);
            constexpr uint32_t idO = idesc_f16(P2_BQ, D);
            auto mma_s = [&](int t, int s) {   // S_t = Q_t . K(stage s)^T
                const uint32_t q0 = smem_u32(sm + L::OFF_Q + t * L::TILE);
                const uint32_t k0 = smem_u32(sm + L::OFF_K + s * L::K_BYTES);
#pragma unroll
                for (int kb = 0; kb < L::KB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(tmem + L::COL_S + t * 128, sdesc_sw128(q0 + kb * P2_BQ * 128 + k * 32),
                                  sdesc_sw128(k0 + kb * P2_BK * 128 + k * 32), idS, (kb | k) ? 1u : 0u);
                umma_commit(&s_full[t]);
            };
            auto mma_pv = [&](int t, int s, bool acc) {   // O_t += P_t (TMEM) . V(stage s)
                const uint32_t v0 = smem_u32(sm + L::OFF_V + s * L::V_BYTES);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16_ts(tmem + L::COL_O + t * D, tmem + L::col_p(t) + kb * 32 + k * 8,
                                    sdesc_sw128(v0 + kb * L::V_BLOCK + k * 32), idO, (acc || kb || k) ? 1u : 0u);
                umma_commit(&o_full[t]);
            };
            bool ok = mbar_wait(q_full, 0) && (nkt == 0 || mbar_wait(&kv_full[0], 0));
            int j = 0;
            if (ok && nkt > 0) {
                tc_fence_after();
                mma_s(0, 0);
                mma_s(1, 0);
            }
            for (; ok && j < nkt; ++j) {
                const int s = j % NSTG;
                const bool more = j + 1 < nkt;
                const int s1 = (j + 1) % NSTG;
                // S_t(j + 1) may overwrite S_t(j): p_full[t] says its row
                // values have all been read.  With P over S (head_dim 128)
                // P . V(j) must go first.
                if (!mbar_wait(&p_full[0], (uint32_t)j & 1u)) break;
                tc_fence_after();
                if (L::ALIAS) mma_pv(0, s, j > 0);
                if (more) {
                    if (!mbar_wait(&kv_full[s1], (uint32_t)((j + 1) / NSTG) & 1u)) break;
                    tc_fence_after();
                    mma_s(0, s1);
                }
                if (!L::ALIAS) mma_pv(0, s, j > 0);
                if (!mbar_wait(&p_full[1], (uint32_t)j & 1u)) break;
                tc_fence_after();
                if (L::ALIAS) mma_pv(1, s, j > 0);
                if (more) mma_s(1, s1);
                if (!L::ALIAS) mma_pv(1, s, j > 0);
                umma_commit(&kv_empty[s]);
            }
            if (!ok || j < nkt) sflag[0] = 1;
            sflag[2] = j;
        }
    } else {   // ------------------------------------------------ softmax warps
        constexpr float RESCALE = 8.f;
        const int t = (warp - 2) >> 2;                // query tile: 0 = A, 1 = B
        const int qw = warp & 3;                      // TMEM lane quarter of this warp
        const int r = qw * 32 + lane;                 // query row within the tile
        const int row0 = q_first + t * P2_BQ;         // the tile's first row
        const int qp = a.pos0 + row0 + r;             // this row's position
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const uint32_t tS = tmem + L::COL_S + t * 128 + lane_off;
        const uint32_t tO = tmem + L::COL_O + t * D + lane_off;
        const uint32_t tP = tmem + L::col_p(t) + lane_off;
        const float sc_log2 = 1.4426950408889634f * rsqrtf((float)D);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // p = 2^(s - mr) for the row's 128 scores of the tile (masked: 0), 64
        // columns per TMEM load, packed as f16 pairs into pk (keys 2c, 2c + 1
        // in pk[c]).  Returns the row sum; mt = the tile's largest visible
        // scaled score.  `masked` is warp-uniform: false when every row of
        // the warp sees all 128 keys.
        auto emit = [&](float mr, int lim, bool masked, float& mt, uint32_t (&pk)[64]) -> float {
            const float mo = mr == -INFINITY ? 0.f : mr;   // no visible key yet: every p is 0
            float rs = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 64) {
                uint32_t v[64];
                tmem_ld32(tS + c0, v);
                tmem_ld32(tS + c0 + 32, v + 32);
                tmem_ld_wait();
                if (masked) {
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const float x0 = c0 + c < lim ? __uint_as_float(v[c]) * sc_log2 : -INFINITY;
                        const float x1 = c0 + c + 1 < lim ? __uint_as_float(v[c + 1]) * sc_log2 : -INFINITY;
                        mt = fmaxf(mt, fmaxf(x0, x1));
                        const float p0 = ex2(x0 - mo), p1 = ex2(x1 - mo);
                        rs += p0 + p1;
                        pk[(c0 + c) / 2] = pack_f16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const float x0 = __uint_as_float(v[c]) * sc_log2;
                        const float x1 = __uint_as_float(v[c + 1]) * sc_log2;
                        mt = fmaxf(mt, fmaxf(x0, x1));
                        const float p0 = ex2(x0 - mo), p1 = ex2(x1 - mo);
                        rs += p0 + p1;
                        pk[(c0 + c) / 2] = pack_f16x2(p0, p1);
                    }
                }
            }
            return rs;
        };
        for (int j = 0; j < nkt; ++j) {
            if (!mbar_wait(&s_full[t], (uint32_t)j & 1u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key0 = j * P2_BK;
            int lim = a.n_keys - key0;                        // keys i < lim of the tile are visible
            if (a.causal) lim = min(lim, qp - key0 + 1);
            lim = max(0, min(P2_BK, lim));
            const bool masked = !__all_sync(FULL_MASK, lim == P2_BK);
            if (j == 0) {   // the first tile sets the reference maximum
                float mt = -INFINITY;
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 64) {
                    uint32_t v[64];
                    tmem_ld32(tS + c0, v);
                    tmem_ld32(tS + c0 + 32, v + 32);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (c0 + i < lim) mt = fmaxf(mt, __uint_as_float(v[i]) * sc_log2);
                }
                m = mt;
            }
            // the reference maximum m moves (and O, l are rescaled) only when
            // the tile's maximum exceeds it by more than RESCALE (log2 units),
            // so p stays <= 2^RESCALE (f16-safe); then the tile is redone
            uint32_t pk[64];
            float mt = -INFINITY;
            float rs = emit(m, lim, masked, mt, pk);
            const bool move = mt > m + RESCALE;
            const bool any_move = __any_sync(FULL_MASK, move);
            float corr = 1.f;
            if (any_move) {
                const float mnew = move ? mt : m;
                corr = move ? exp2f(m - mnew) : 1.f;
                float mt2 = -INFINITY;
                rs = emit(mnew, lim, masked, mt2, pk);
                l *= corr;
                m = mnew;
            }
            if (j > 0) {   // P . V(j - 1) must be complete before O is touched or P is rewritten
                if (!mbar_wait(&o_full[t], (uint32_t)(j - 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (any_move) {
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld16(tO + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                        tmem_st16(tO + c0, o);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < 64; c += 16) tmem_st16(tP + c, pk + c);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
            l += rs;
        }
        if (ok && nkt > 0 && !mbar_wait(&o_full[t], (uint32_t)(nkt - 1) & 1u)) ok = false;
        if (!ok) sflag[0] = 1;
        tc_fence_after();
        if (ok) {
            const float inv = 1.f / l;
            const bool live = row0 + r < a.T_per_seq;
            uint16_t* out = a.att + (size_t)(z * a.T_per_seq + row0 + r) * a.ld_att + h * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
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

}  // namespace

template <int D>
static void launch_pp(const void* mq, const void* mk, const void* mv, const AttnTcArgs& a, int nseq,
                      cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_tc2<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, P2Smem<D>::TOTAL);
        attr = true;
    }
    dim3 grid((a.T_per_seq + 2 * P2_BQ - 1) / (2 * P2_BQ), a.NH, nseq);
    launch_k(k_attn_tc2<D>, grid, dim3(P2_THREADS), P2Smem<D>::TOTAL, s,
             *reinterpret_cast<const CUtensorMap*>(mq), *reinterpret_cast<const CUtensorMap*>(mk),
             *reinterpret_cast<const CUtensorMap*>(mv), a);
}

void launch_attn_tc2(const void* mq, const void* mk, const void* mv, const AttnTcArgs& a, int nseq, int D,
                     cudaStream_t s) {
    if (D == 64) launch_pp<64>(mq, mk, mv, a, nseq, s);
    else if (D == 128) launch_pp<128>(mq, mk, mv, a, nseq, s);
}

}  // namespace ember
