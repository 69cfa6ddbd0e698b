// gemm_persistent.cu -- persistent tcgen05 GEMM for many-row operands
// (prefill and encoder projections, M > 128).
//
//   D[M,N] = A[M,K] . B[N,K]^T      (f16 or bf16 operands, f32 accumulation)
//
// One CTA per SM walks the 128 x BN output tiles (row tiles fastest, so the
// CTAs running at the same time share weight tiles in L2).  Warp 0 streams A
// and B k-blocks through a STAGES-deep shared-memory ring across tile
// boundaries; warp 1 issues tcgen05.mma into one of two TMEM accumulators
// (2 x BN columns), so the epilogue warps 2-5 drain tile i while tile i + 1
// accumulates.  Accumulator hand-off: acc_full[b] (MMA commit -> epilogue),
// acc_empty[b] (128 epilogue arrivals -> MMA).  Every wait is bounded; a
// timeout raises EMBER_ERR_TIMEOUT, drains the copies in flight and frees
// TMEM.  Epilogues: bias store, residual add, SwiGLU (f16 out), argmax.
// With an output tensor map the store / residual / SwiGLU epilogues stage
// 32-column slices (f32) or the whole tile (f16) in a swizzled shared buffer
// and write them with TMA (the residual as an f32 reduce-add), so the output
// leaves in whole 128-byte lines instead of one 16-byte piece per row.
// The residual epilogue adds, so that GEMM is split stream-K style: CTA b
// takes the b-th contiguous 1/gridDim share of the (tile, k-block) work, a
// tile's k-range may be shared by two or three CTAs, and each adds its
// partial sum (every SM busy whatever the tile count; no inter-CTA waits).
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace ember {

namespace {

constexpr int GP_BM = 128;
constexpr int GP_BK = 64;
constexpr int GP_THREADS = 192;

// Epilogue of one accumulator tile: this thread's row `row`, columns
// [n0, n0 + BN), read from TMEM at tbase (lane quadrant already applied).
template <int BN>
__device__ __forceinline__ void tile_epilogue(const GemmEpilogue& e, uint32_t tbase, int row, int n0,
                                              int M, int N, unsigned long long& best, bool& f16bad) {
    const float wsc = pow2f(e.w_exp);   // the weights' storage scale
    for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld16(tbase + c, r);
        tmem_ld16(tbase + c + 16, r + 16);
        tmem_ld_wait();
        const int n = n0 + c;
        if (row >= M || n >= N) continue;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * wsc;
        const bool fullc = (n + 32 <= N);
        if (e.mode == EPI_ARGMAX) {
            if (e.out_f32) {
                float* o = e.out_f32 + (size_t)row * e.ldo + n;
                for (int i = 0; i < 32 && n + i < N; ++i) o[i] = v[i];
            }
            for (int i = 0; i < 32 && n + i < N; ++i) {
                const unsigned long long kk = argmax_key(v[i], (uint32_t)(n + i));
                best = kk > best ? kk : best;
            }
        } else if (e.mode == EPI_SWIGLU) {
            // columns 2i / 2i+1 = gate_i / up_i -> output column n/2 + i
            uint16_t* o = e.out_h + (size_t)row * e.ldo + (n >> 1);
            if (fullc) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float g0 = v[4 * i], u0 = v[4 * i + 1];
                    const float g1 = v[4 * i + 2], u1 = v[4 * i + 3];
                    pk[i] = pack_f16x2_chk(__fdividef(g0, 1.f + __expf(-g0)) * u0,
                                           __fdividef(g1, 1.f + __expf(-g1)) * u1, f16bad);
                }
                uint4* o4 = reinterpret_cast<uint4*>(o);
                o4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                o4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else {
                for (int i = 0; i < 16 && n + 2 * i + 1 < N; ++i) {
                    const float g = v[2 * i], u = v[2 * i + 1];
                    o[i] = f32_to_f16_chk(__fdividef(g, 1.f + __expf(-g)) * u, f16bad);
                }
            }
        } else {
            float* o = e.out_f32 + (size_t)row * e.ldo + n;
            if (e.mode == EPI_STORE && e.bias) {
                for (int i = 0; i < 32; ++i)
                    if (n + i < N) v[i] += e.bias[n + i];
            }
            if (fullc) {
                float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float4 t = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    if (e.mode == EPI_RESID) {
                        const float4 x = o4[i];
                        t.x += x.x; t.y += x.y; t.z += x.z; t.w += x.w;
                    }
                    o4[i] = t;
                }
            } else {
                for (int i = 0; i < 32 && n + i < N; ++i)
                    o[i] = (e.mode == EPI_RESID) ? o[i] + v[i] : v[i];
            }
        }
    }
}

constexpr int GP_STAGING = 32768;   // output staging: two 16 KB f32 slices or one f16 tile

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// the same barrier, returning whether every epilogue thread passed `ok`
__device__ __forceinline__ bool epi_bar_and(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

// The same epilogues through TMA: thread `r` (0..127) holds tile row m0 + r.
// f32 modes: the slices the kernel writes (32 columns each; none past N)
// alternate, by their running count `slice`, between the two 16 KB halves of
// stg ([128 rows][32 f32], 16-byte chunk k of row r at chunk k ^ (r & 7), the
// map's 128-byte swizzle); one copy (one bulk group) per slice, and the slice
// written two slices ago must have been read by its copy first.  SwiGLU: the tile's BN/2 f16 outputs per row as
// BN/128 blocks of [128 rows][64 f16] in the same layout.  Rows >= M are
// written as zeros (the map clips at its own row count).
template <int BN>
__device__ __forceinline__ void tile_epilogue_tma(const GemmEpilogue& e, const CUtensorMap* tmO, uint32_t tbase,
                                                  int r, int m0, int n0, int M, int N, uint8_t* stg,
                                                  int& slice, bool& f16bad) {
    const float wsc = pow2f(e.w_exp);
    const bool live = m0 + r < M;
    const bool leader = threadIdx.x == 64;   // first epilogue thread issues the copies
    if (e.mode == EPI_SWIGLU) {
        if (leader) bulk_wait_read<0>();
        epi_bar();
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
            uint32_t u[32];
            tmem_ld16(tbase + c, u);
            tmem_ld16(tbase + c + 16, u + 16);
            tmem_ld_wait();
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float g0 = __uint_as_float(u[4 * i]) * wsc, u0 = __uint_as_float(u[4 * i + 1]) * wsc;
                const float g1 = __uint_as_float(u[4 * i + 2]) * wsc, u1 = __uint_as_float(u[4 * i + 3]) * wsc;
                const float y0 = __fdividef(g0, 1.f + __expf(-g0)) * u0;
                const float y1 = __fdividef(g1, 1.f + __expf(-g1)) * u1;
                pk[i] = live && n0 + c + 4 * i < N ? pack_f16x2_chk(y0, y1, f16bad) : 0u;
            }
            uint8_t* rowp = stg + (c >> 7) * 16384 + r * 128;
            const int k0 = (c & 127) >> 4;   // 16-byte chunk of the 32 outputs' first half
            *reinterpret_cast<uint4*>(rowp + ((k0 ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(rowp + (((k0 + 1) ^ (r & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epi_bar();
        if (leader) {
            for (int b = 0; b < BN / 128; ++b)
                if (n0 / 2 + b * 64 < N / 2) tma_store_2d(tmO, stg + b * 16384, n0 / 2 + b * 64, m0);
            bulk_commit();
        }
        return;
    }
#pragma unroll 1
    for (int c = 0; c < BN && n0 + c < N; c += 32) {
        uint32_t u[32];
        tmem_ld16(tbase + c, u);
        tmem_ld16(tbase + c + 16, u + 16);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = live ? __uint_as_float(u[i]) * wsc : 0.f;
        if (e.mode == EPI_STORE && e.bias && live) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (n0 + c + i < N) v[i] += e.bias[n0 + c + i];
        }
        uint8_t* buf = stg + (slice & 1) * 16384;
        ++slice;
        if (leader) bulk_wait_read<1>();   // the copy of the slice before last has read buf
        epi_bar();
        uint8_t* rowp = buf + r * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(rowp + ((k ^ (r & 7)) << 4)) =
                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epi_bar();
        if (leader) {
            if (e.mode == EPI_RESID) tma_reduce_add_2d(tmO, buf, n0 + c, m0);
            else tma_store_2d(tmO, buf, n0 + c, m0);
            bulk_commit();
        }
    }
}

}  // namespace

template <int BN, int STAGES>
__global__ void __launch_bounds__(GP_THREADS, 1)
    k_gemm_tcp(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmO, int M, int N, int K, uint32_t idesc, GemmEpilogue e,
               int* status) {
    constexpr int A_BYTES = GP_BM * GP_BK * 2;
    constexpr int B_BYTES = BN * GP_BK * 2;
    constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stg = smem + STAGES * STAGE_BYTES;   // output staging (1024-aligned)
    uint64_t* full = reinterpret_cast<uint64_t*>(stg + GP_STAGING);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;     // [2]
    uint64_t* acc_empty = acc_full + 2;      // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    int* sflag = reinterpret_cast<int*>(tmem_slot + 1);   // [0] failed, [1] issued, [2] consumed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = (K + GP_BK - 1) / GP_BK;
    const int n_mt = (M + GP_BM - 1) / GP_BM, n_nt = (N + BN - 1) / BN;
    const int n_tiles = n_mt * n_nt;
    // Work segments of this CTA: whole tiles b, b + grid, ... or, stream-K
    // (residual epilogue through TMA), the k-blocks [w0, w1) of the
    // tile-major (tile, k-block) sequence, cut at tile boundaries.
    const bool sk = e.mode == EPI_RESID && e.out_map != nullptr;
    const long long W = (long long)n_tiles * nk;
    const long long w0 = sk ? W * blockIdx.x / gridDim.x : 0;
    const long long w1 = sk ? W * (blockIdx.x + 1) / gridDim.x : 0;
    const int my_tiles = sk ? (w1 > w0 ? (int)((w1 - 1) / nk - w0 / nk) + 1 : 0)
                            : ((int)blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0);
    auto tile_mn = [&](int li, int& m0, int& n0, int& kb0, int& kb1) {
        int t;
        if (sk) {
            t = (int)(w0 / nk) + li;
            kb0 = li == 0 ? (int)(w0 % nk) : 0;
            kb1 = (int)((w1 - (long long)t * nk) < nk ? (w1 - (long long)t * nk) : nk);
        } else {
            t = (int)blockIdx.x + li * (int)gridDim.x;
            kb0 = 0;
            kb1 = nk;
        }
        m0 = (t % n_mt) * GP_BM;
        n0 = (t / n_mt) * BN;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 128);
        }
        sflag[0] = 0;
        sflag[1] = 0;
        sflag[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (my_tiles > 0) {   // the first segment's weights do not depend on the previous kernel
            int m0, n0, kb0, kb1;
            tile_mn(0, m0, n0, kb0, kb1);
            const int pre = kb1 - kb0 < STAGES ? kb1 - kb0 : STAGES;
            for (int i = 0; i < pre; ++i) {
                mbar_expect_tx(&full[i], STAGE_BYTES);
                tma_load_2d(smem + i * STAGE_BYTES + A_BYTES, &tmB, (kb0 + i) * GP_BK, n0, &full[i]);
            }
        }
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(tmem_slot)),
            "r"((uint32_t)(2 * BN)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // activations and the residual stream are the previous kernels' outputs

    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer, k-blocks of all my segments
            int g = 0;     // global k-block count
            bool fail = false;
            int pre = 0;   // B blocks of the first segment already issued
            for (int li = 0; li < my_tiles && !fail; ++li) {
                int m0, n0, kb0, kb1;
                tile_mn(li, m0, n0, kb0, kb1);
                if (li == 0) pre = kb1 - kb0 < STAGES ? kb1 - kb0 : STAGES;
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % STAGES;
                    uint8_t* sa = smem + s * STAGE_BYTES;
                    if (g >= pre) {
                        if (g >= STAGES &&
                            !mbar_wait(&empty[s], ((uint32_t)(g / STAGES) & 1u) ^ 1u)) {
                            fail = true;
                            break;
                        }
                        mbar_expect_tx(&full[s], STAGE_BYTES);
                        tma_load_2d(sa + A_BYTES, &tmB, kb * GP_BK, n0, &full[s]);
                    }
                    tma_load_2d(sa, &tmA, kb * GP_BK, m0, &full[s]);
                }
            }
            if (fail) sflag[0] = 1;
            sflag[1] = g;
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------- MMA issuer
            int g = 0;
            bool fail = false;
            for (int li = 0; li < my_tiles && !fail; ++li) {
                const int b = li & 1;
                int m0, n0, kb0, kb1;
                tile_mn(li, m0, n0, kb0, kb1);
                if (!mbar_wait(&acc_empty[b], ((uint32_t)(li >> 1) & 1u) ^ 1u)) {
                    fail = true;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * BN);
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % STAGES;
                    if (!mbar_wait(&full[s], (uint32_t)(g / STAGES) & 1u)) {
                        fail = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                    for (int k = 0; k < GP_BK / 16; ++k)
                        umma_bf16(acc, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                                  (kb > kb0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);   // the stage is free once these MMAs read it
                }
                if (!fail) umma_commit(&acc_full[b]);
            }
            if (fail) sflag[0] = 1;
            sflag[2] = g;
        }
    } else {   // ---------------- epilogue warps 2..5
        const int q = warp & 3;
        unsigned long long best = 0ull;
        int best_row = -1;
        bool f16bad = false;   // EPI_SWIGLU: an output beyond the f16 range
        int slice = 0;         // f32 slices written through TMA so far
        const bool tma_out = e.out_map && e.mode != EPI_ARGMAX && (e.mode != EPI_SWIGLU || BN >= 128);
        for (int li = 0; li < my_tiles; ++li) {
            const int b = li & 1;
            int m0, n0, kb0, kb1;
            tile_mn(li, m0, n0, kb0, kb1);
            const int row = m0 + q * 32 + lane;
            bool got = mbar_wait(&acc_full[b], (uint32_t)(li >> 1) & 1u);
            if (tma_out) got = epi_bar_and(got);   // the TMA epilogue's barriers need all 128 threads
            if (!got) {
                sflag[0] = 1;
                break;
            }
            tc_fence_after();
            if (e.mode == EPI_ARGMAX && row != best_row) {   // a new row tile: flush the last key
                if (best && best_row >= 0 && best_row < M) atomicMax(e.keys + best_row, best);
                best = 0ull;
                best_row = row;
            }
            if (tma_out)
                tile_epilogue_tma<BN>(e, &tmO, tmem + (uint32_t)(b * BN) + ((uint32_t)(q * 32) << 16), q * 32 + lane,
                                      m0, n0, M, N, stg, slice, f16bad);
            else
                tile_epilogue<BN>(e, tmem + (uint32_t)(b * BN) + ((uint32_t)(q * 32) << 16), row, n0, M, N,
                                  best, f16bad);
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
        }
        if (e.mode == EPI_ARGMAX && best && best_row >= 0 && best_row < M)
            atomicMax(e.keys + best_row, best);
        if (f16bad) raise_status(status, EMBER_ERR_RANGE);
        if (tma_out && threadIdx.x == 64) bulk_wait<0>();   // every output copy complete before exit
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && sflag[0]) raise_status(status, EMBER_ERR_TIMEOUT);
    if (warp == 0 && lane == 0 && sflag[0]) {   // copies issued but never consumed
        for (int g = sflag[2]; g < sflag[1]; ++g)
            (void)mbar_wait(&full[g % STAGES], (uint32_t)(g / STAGES) & 1u);
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)(2 * BN)));
    }
}

template <int BN, int STAGES>
static void launch_p(const void* tmA, const void* tmB, int m_rows, int N, int K, uint32_t idesc,
                     const GemmEpilogue& e, int* status, int sms, cudaStream_t s) {
    constexpr int STAGE_BYTES = (GP_BM + BN) * GP_BK * 2;
    constexpr int SMEM = STAGES * STAGE_BYTES + GP_STAGING + 1024 + 256;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_tcp<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        attr = true;
    }
    const int tiles = ((m_rows + GP_BM - 1) / GP_BM) * ((N + BN - 1) / BN);
    // stream-K (residual through TMA): every SM, as long as each gets a k-block
    const long long work = e.mode == EPI_RESID && e.out_map ? (long long)tiles * ((K + GP_BK - 1) / GP_BK) : tiles;
    const int grid = work < sms ? (int)work : sms;
    static const CUtensorMap no_map{};   // unused when e.out_map is null
    const CUtensorMap* tmO = e.out_map ? reinterpret_cast<const CUtensorMap*>(e.out_map) : &no_map;
    launch_k(k_gemm_tcp<BN, STAGES>, dim3(grid), dim3(GP_THREADS), SMEM, s,
             *reinterpret_cast<const CUtensorMap*>(tmA), *reinterpret_cast<const CUtensorMap*>(tmB), *tmO,
             m_rows, N, K, idesc, e, status);
}

void launch_gemm_persistent(const void* tmA, const void* tmB, int bn, int m_rows, int N, int K,
                            uint32_t idesc, const GemmEpilogue& e, int* status, int sms,
                            cudaStream_t s) {
    switch (bn) {
        case 64: launch_p<64, 8>(tmA, tmB, m_rows, N, K, idesc, e, status, sms, s); break;
        case 128: launch_p<128, 6>(tmA, tmB, m_rows, N, K, idesc, e, status, sms, s); break;
        default: launch_p<256, 4>(tmA, tmB, m_rows, N, K, idesc, e, status, sms, s); break;
    }
}

}  // namespace ember
