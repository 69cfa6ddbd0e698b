// gemm.cu -- tcgen05 / TMEM tensor-core GEMM fed by TMA, with the fused
// epilogues of the projections (bias, residual add, SwiGLU).
//
//   D[M,N] = A[M,K] . B[N,K]^T      A: activations (bf16, K contiguous)
//                                   B: weights, HF [out, in] (bf16, K contiguous)
//
// k_gemm_tc serves calls of at most one row tile (decode batches up to 128
// tokens, narrow heads), with 64-column tiles and the K range split over
// grid.z for the additive epilogues; more rows go to the persistent kernel
// (gemm_persistent.cu).  One CTA computes a BM x BN tile (BM = 128 rows of
// A = 128 TMEM lanes, BN f32 accumulator columns).  Warp roles:
//   warp 0   one thread issues the TMA loads of A and B k-blocks (BK = 64
//            elements = one 128-byte swizzle span) into a STAGES-deep ring;
//   warp 1   allocates TMEM; one thread issues tcgen05.mma (M=128, N=BN,
//            K=16 per instruction, 4 per k-block) and commits each stage back
//            to the producer, then commits the finished accumulator;
//   warps 2-5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//            32*(w%4)..+31), apply the fused epilogue, store to global.
// Every mbarrier wait is bounded (~1 s of clock64); a timeout raises
// EMBER_ERR_TIMEOUT, waits (bounded) for copies still in flight, frees TMEM
// and returns.
//
// The projections this serves: q/k/v (+bias), o_proj (+residual), gate/up
// (SwiGLU) and down (+residual) of ember scripts/reference_forward.py
// forward(), in the whole-sequence form of LowLlamaBasic reference.py.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace ember {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;
constexpr int GEMM_THREADS = 192;
template <int BN, int STAGES>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              int M, int N, int K, uint32_t idesc, GemmEpilogue e, int* status) {
    constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    constexpr int B_BYTES = BN * GEMM_BK * 2;
    constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
    int* sflag = reinterpret_cast<int*>(tmem_slot + 1);   // [0] failed, [1] issued, [2] consumed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * GEMM_BM;
    // this CTA's k-blocks [kb0, kb0 + nk) (split-K over grid.z)
    const int nk_all = (K + GEMM_BK - 1) / GEMM_BK;
    const int per = (nk_all + (int)gridDim.z - 1) / (int)gridDim.z;
    const int kb0 = (int)blockIdx.z * per;
    const int nk = max(0, min(nk_all, kb0 + per) - kb0);
    const bool split = gridDim.z > 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        sflag[0] = 0;
        sflag[1] = 0;
        sflag[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // the weights (B) of the first stages do not depend on the previous
        // kernel: start them now, under its tail
        for (int kb = 0; kb < nk && kb < STAGES; ++kb) {
            uint8_t* sa = smem + kb * STAGE_BYTES;
            mbar_expect_tx(&full[kb], STAGE_BYTES);
            tma_load_2d(sa + A_BYTES, &tmB, (kb0 + kb) * GEMM_BK, n0, &full[kb]);
        }
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(tmem_slot)),
            "r"((uint32_t)BN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // barrier init and TMEM allocation overlapped the previous kernel's tail;
    // activations (A) and the residual stream are its outputs.
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer
            int kb = 0;
            for (; kb < nk; ++kb) {
                const int s = kb % STAGES;
                const uint32_t it = (uint32_t)(kb / STAGES);
                uint8_t* sa = smem + s * STAGE_BYTES;
                if (kb >= STAGES) {   // the first STAGES got their weights before the wait
                    if (!mbar_wait(&empty[s], (it & 1u) ^ 1u)) {
                        sflag[0] = 1;
                        break;
                    }
                    mbar_expect_tx(&full[s], STAGE_BYTES);
                    tma_load_2d(sa + A_BYTES, &tmB, (kb0 + kb) * GEMM_BK, n0, &full[s]);
                }
                tma_load_2d(sa, &tmA, (kb0 + kb) * GEMM_BK, m0, &full[s]);
            }
            sflag[1] = kb;
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------- MMA issuer
            int kb = 0;
            for (; kb < nk; ++kb) {
                const int s = kb % STAGES;
                const uint32_t it = (uint32_t)(kb / STAGES);
                if (!mbar_wait(&full[s], it & 1u)) {
                    sflag[0] = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + s * STAGE_BYTES);
                const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                for (int k = 0; k < GEMM_BK / 16; ++k) {
                    umma_bf16(tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                              (kb > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);   // frees the stage once these MMAs have read it
            }
            sflag[2] = kb;
            umma_commit(tfull);           // accumulator complete (after all issued MMAs)
        }
    } else {   // ---------------- epilogue warps 2..5
        const int q = warp & 3;
        const int row = m0 + q * 32 + lane;
        unsigned long long best = 0ull;   // EPI_ARGMAX
        bool f16bad = false;              // EPI_SWIGLU: an output beyond the f16 range
        const float wsc = pow2f(e.w_exp);   // the weights' storage scale
        if (!mbar_wait(tfull, 0)) {
            sflag[0] = 1;
        } else {
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld16(tbase + c, r);
                tmem_ld16(tbase + c + 16, r + 16);
                tmem_ld_wait();
                const int n = n0 + c;
                if (row >= M || n >= N || nk == 0) continue;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * wsc;
                const bool fullc = (n + 32 <= N);
                if (e.mode == EPI_ARGMAX) {   // logits (optional) and the row's best key
                    if (e.out_f32) {
                        float* o = e.out_f32 + (size_t)row * e.ldo + n;
                        for (int i = 0; i < 32 && n + i < N; ++i) o[i] = v[i];
                    }
                    for (int i = 0; i < 32 && n + i < N; ++i) {
                        const unsigned long long kk = argmax_key(v[i], (uint32_t)(n + i));
                        best = kk > best ? kk : best;
                    }
                } else if (split) {   // partial sums of a K split: add into the output
                    float* o = e.out_f32 + (size_t)row * e.ldo + n;
                    if (e.mode == EPI_STORE && e.bias && blockIdx.z == 0) {
                        for (int i = 0; i < 32; ++i)
                            if (n + i < N) v[i] += e.bias[n + i];
                    }
                    if (fullc) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(o + 4 * i),
                                         "f"(v[4 * i]), "f"(v[4 * i + 1]), "f"(v[4 * i + 2]),
                                         "f"(v[4 * i + 3])
                                         : "memory");
                    } else {
                        for (int i = 0; i < 32 && n + i < N; ++i) atomicAdd(o + i, v[i]);
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
                            pk[i] = pack_f16x2_chk(g0 / (1.f + __expf(-g0)) * u0,
                                                   g1 / (1.f + __expf(-g1)) * u1, f16bad);
                        }
                        uint4* o4 = reinterpret_cast<uint4*>(o);
                        o4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        o4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    } else {
                        for (int i = 0; i < 16 && n + 2 * i + 1 < N; ++i) {
                            const float g = v[2 * i], u = v[2 * i + 1];
                            o[i] = f32_to_f16_chk(g / (1.f + __expf(-g)) * u, f16bad);
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
            if (e.mode == EPI_ARGMAX && row < M && best) atomicMax(e.keys + row, best);
            if (f16bad) raise_status(status, EMBER_ERR_RANGE);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && sflag[0]) raise_status(status, EMBER_ERR_TIMEOUT);
    if (warp == 0 && lane == 0 && sflag[0]) {
        // drain TMA copies that were issued but never consumed
        for (int kb = sflag[2]; kb < sflag[1]; ++kb)
            (void)mbar_wait(&full[kb % STAGES], (uint32_t)(kb / STAGES) & 1u);
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)BN));
    }
}

// ------------------------------------------------------------------- host --
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

static bool encode_map_t(void* out, const void* ptr, CUtensorMapDataType dt, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box) {
    auto enc = encode_fn();
    if (!enc || rank < 2 || rank > 5) return false;
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) {
            if (strides[i] % 16) return false;
            st[i] = strides[i];
        }
    }
    CUresult r = enc(reinterpret_cast<CUtensorMap*>(out), dt,
                     (cuuint32_t)rank, const_cast<void*>(ptr), d, st, bx, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_map_bf16(void* out, const void* ptr, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
    return encode_map_t(out, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, dims, strides, box);
}

bool make_out_map(void* out, const void* ptr, int rows, int cols, int ld, bool f16) {
    if (rows <= 0 || cols <= 0 || cols > ld) return false;
    const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)ld * (f16 ? 2 : 4)};
    const uint32_t box[2] = {f16 ? 64u : 32u, 128u};
    return encode_map_t(out, ptr, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dims,
                        strides, box);
}

static bool make_map(void* out, const uint16_t* ptr, int rows, int ld, int K, int box_rows) {
    if ((ld % 8) || (K % 8)) return false;
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)ld * 2};
    const uint32_t box[2] = {(uint32_t)GEMM_BK, (uint32_t)box_rows};
    return encode_map_bf16(out, ptr, 2, dims, strides, box);
}

// N tile of the many-row GEMM: an M = 128, N = 256 tcgen05.mma takes ~171
// cycles against ~112 for N = 128 (the minimum per instruction), so 256
// columns do 31 % more work per cycle -- worth a partly empty last tile
// unless N is small
static int pick_bn(int N) {
    if (N <= 64) return 64;
    if (N <= 512) return 128;
    return 256;
}

bool make_gemm_plan(GemmPlan& p, const uint16_t* A, int M, int lda, const uint16_t* B, int N,
                    int ldb, int K, bool f16) {
    p.f16 = f16;
    static_assert(sizeof(CUtensorMap) <= sizeof(p.tmA), "tensor map size");
    p.M = M;
    p.N = N;
    p.K = K;
    p.bn = pick_bn(N);
    int dev = 0;
    p.sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&p.sms, cudaDevAttrMultiProcessorCount, dev);
    p.ok = make_map(p.tmA, A, M, lda, K, GEMM_BM) && make_map(p.tmB, B, N, ldb, K, p.bn) &&
           make_map(p.tmB64, B, N, ldb, K, 64);
    return p.ok;
}

int gemm_splits(const GemmPlan& p, int m_rows, int mode) {
    if (m_rows > GEMM_BM || (mode != EPI_STORE && mode != EPI_RESID)) return 1;
    const int tiles = (p.N + 63) / 64;
    const int nk = (p.K + GEMM_BK - 1) / GEMM_BK;
    int ks = p.sms / tiles;
    if (ks > nk) ks = nk;
    if (ks <= 1) return 1;
    const int per = (nk + ks - 1) / ks;
    return (nk + per - 1) / per;   // no empty split
}

template <int BN, int STAGES>
static void launch_bn(const GemmPlan& p, int m_rows, const GemmEpilogue& e, int* status,
                      cudaStream_t s, int ksplit = 1) {
    constexpr int STAGE_BYTES = (GEMM_BM + BN) * GEMM_BK * 2;
    constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_tc<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM);
        attr = true;
    }
    dim3 grid((p.N + BN - 1) / BN, (m_rows + GEMM_BM - 1) / GEMM_BM, ksplit);
    const CUtensorMap* ta = reinterpret_cast<const CUtensorMap*>(p.tmA);
    const CUtensorMap* tb = reinterpret_cast<const CUtensorMap*>(BN == p.bn ? p.tmB : p.tmB64);
    const uint32_t idesc = p.f16 ? idesc_f16(GEMM_BM, BN) : idesc_bf16(GEMM_BM, BN);
    launch_k(k_gemm_tc<BN, STAGES>, grid, dim3(GEMM_THREADS), SMEM, s, *ta, *tb, m_rows, p.N, p.K,
             idesc, e, status);
}

void launch_gemm(const GemmPlan& p, int m_rows, const GemmEpilogue& e, int* status,
                 cudaStream_t s) {
    if (m_rows <= 0) return;
    // one row tile: narrow tiles, K split for the additive epilogues -- except
    // a wide argmax head (the tied LM head over the vocabulary), which the
    // persistent kernel serves with 256-column tiles: a quarter of the tiles,
    // so a quarter of the activation re-reads, and one key flush per row
    if (m_rows <= GEMM_BM && !(e.mode == EPI_ARGMAX && p.N >= 16 * 256 && p.bn == 256)) {
        GemmEpilogue e2 = e;
        int ks = gemm_splits(p, m_rows, e.mode);
        if (e.mode == EPI_STORE && !e.zeroed) ks = 1;
        e2.ksplit = ks;
        launch_bn<64, 8>(p, m_rows, e2, status, s, ks);
        return;
    }
    // many rows: persistent tiles with a double-buffered accumulator
    const uint32_t idesc = p.f16 ? (p.bn == 64 ? idesc_f16(GEMM_BM, 64) : p.bn == 128 ? idesc_f16(GEMM_BM, 128) : idesc_f16(GEMM_BM, 256))
                                 : (p.bn == 64 ? idesc_bf16(GEMM_BM, 64) : p.bn == 128 ? idesc_bf16(GEMM_BM, 128) : idesc_bf16(GEMM_BM, 256));
    launch_gemm_persistent(p.tmA, p.tmB, p.bn, m_rows, p.N, p.K, idesc, e, status, p.sms, s);
}

}  // namespace ember
