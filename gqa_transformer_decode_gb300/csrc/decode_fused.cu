// decode_fused.cu -- batch-1 decode as two kernels per decoder layer.
//
// D1 (k_fused_attn): one thread-block cluster of C CTAs per kv head g.  Each
//   CTA RMS-normalises x, computes its share of the group's q/k/v rows
//   (weights bulk-loaded into shared memory before the programmatic-launch
//   wait), and sends them with st.async into the shared memory of the CTAs
//   that run attention (all C, or CTA 0 alone for contexts up to FA_SOLO
//   keys), where an mbarrier counts the bytes.  Those apply the optional q/k
//   RMSNorm and RoPE, write the new K/V row (the CTA whose key range holds
//   the position), run flash attention over their key ranges for all G query
//   heads of the group and merge the partial softmaxes through distributed
//   shared memory; the merged heads reach every CTA the same way, and each
//   multiplies them by its rows of the group's o_proj column block, adding
//   the result into the residual.  A CTA leaves only after every store aimed
//   at its shared memory has been counted on its own barrier.
// D2 (k_fused_mlp): every CTA owns chunks of FC intermediate features:
//   RMSNorm, the gate/up rows of those features, SwiGLU, and their columns of
//   down_proj (a transposed f16 copy, so each chunk is 4 contiguous rows),
//   adding its partial down_proj output into the residual.
//
// The split-K additions use red.global.add into a zeroed accumulator, so the
// residual stream of kernel n is x_n = X[n-1] + Z[n-1]: kernel n reads
// X[(n-1)%2] and Z[(n-1)%3], writes X[n%2] = x_n, zeroes Z[(n-2)%3] and
// accumulates into Z[n%3] -- no kernel writes a buffer that one of its own
// CTAs may still read.  (Llama / Qwen2 decoder layer: x += o_proj(attn(
// rmsnorm(x))); x += down(silu(gate(rmsnorm(x))) * up(rmsnorm(x))).)
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "mma_common.cuh"

#include <cstdlib>

namespace ember {

namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// split cluster barrier: arrive (relaxed) early, wait (acquire) later
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of shared variable p in CTA `cta` of this cluster
__device__ __forceinline__ uint32_t dsmem(const void* p, uint32_t cta) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(cta));
    return r;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
// 8-byte store (two 32-bit words) into the shared memory of a CTA of this
// cluster whose completion counts 8 bytes on that CTA's mbarrier (both
// addresses from mapa)
__device__ __forceinline__ void st_async2u(uint32_t addr, uint32_t a, uint32_t b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "r"(a), "r"(b), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async1(uint32_t addr, float a, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
                 "r"(__float_as_uint(a)), "r"(bar)
                 : "memory");
}
// mbarrier wait whose completion orders the stores of other CTAs of the
// cluster (st.async complete_tx releases at cluster scope); false once
// `budget` SM cycles have passed without it
__device__ __forceinline__ bool mbar_wait_cluster_for(uint64_t* bar, uint32_t parity, long long budget) {
    const uint32_t addr = smem_u32(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(addr), "r"(parity)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > budget) return false;
    }
}
// the kernels' cluster wait: false after ~1 s
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    return mbar_wait_cluster_for(bar, parity, TC_WAIT_CYCLES);
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// relaxed load (a hint read while another kernel may write the word)
__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// 16-byte shared-memory load (explicit state space: short-scoreboard path)
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}
__device__ __forceinline__ void red_add(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// RMSNorm of the residual x = x_in + the sum of the ZI copies of z_in (H
// floats, H % 4 == 0, H <= 4096 for 256 threads).  The weights are loaded
// into registers before the programmatic-launch wait (load_w); apply() issues
// all of its 16-byte loads at once, writes this CTA's slice of x_out (= x) and
// of the ZZ copies of z_zero (= 0) from the values it holds, and leaves
// f16(x * rsqrt(mean(x^2) + eps) * w) in s_xh (the projections' input, at the
// precision of the tensor-core GEMM operands).  The MLP block accumulates into
// ZSLOTS copies (152+ CTAs add into every element), the attention block into
// one (one cluster per kv head adds into an element): the attention block
// reads ZSLOTS copies and clears ZSLOTS for the MLP block after it, the MLP
// block reads one and clears one.
struct ResidualNorm {
    static constexpr int MAXV = 4;
    float4 w[MAXV];
    __device__ __forceinline__ void load_w(const float* wp, int H) {
        const int H4 = H >> 2;
#pragma unroll
        for (int q = 0; q < MAXV; ++q) {
            const int i = threadIdx.x + q * blockDim.x;
            w[q] = i < H4 ? __ldg(reinterpret_cast<const float4*>(wp) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    template <int ZMAX>
    __device__ __forceinline__ void apply(const float* x_in, const float* z_in, float* x_out, float* z_zero,
                                          float eps, int H, int cta, int ncta, uint16_t* s_xh, float* s_red,
                                          int* status, int ZI, int ZZ) {
        const int H4 = H >> 2;
        const int per = (H4 + ncta - 1) / ncta;
        const int e0 = cta * per, e1 = e0 + per;
        float4 v[MAXV];
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < MAXV; ++q) {
            const int i = threadIdx.x + q * blockDim.x;
            if (i < H4) {
                float4 b[ZMAX];
#pragma unroll
                for (int z = 0; z < ZMAX; ++z)
                    b[z] = z < ZI ? __ldcg(reinterpret_cast<const float4*>(z_in + (size_t)z * H) + i)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                float4 t = __ldcg(reinterpret_cast<const float4*>(x_in) + i);
#pragma unroll
                for (int z = 0; z < ZMAX; ++z) {
                    t.x += b[z].x; t.y += b[z].y; t.z += b[z].z; t.w += b[z].w;
                }
                v[q] = t;
            }
        }
#pragma unroll
        for (int q = 0; q < MAXV; ++q) {
            const int i = threadIdx.x + q * blockDim.x;
            if (i < H4) {
                ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
                if (i >= e0 && i < e1) {
                    reinterpret_cast<float4*>(x_out)[i] = v[q];
#pragma unroll
                    for (int z = 0; z < ZMAX; ++z)
                        if (z < ZZ) reinterpret_cast<float4*>(z_zero + (size_t)z * H)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int k = 0; k < (int)(blockDim.x >> 5); ++k) tot += s_red[k];
        const float ri = rsqrtf(tot / (float)H + eps);
        bool bad = false;
#pragma unroll
        for (int q = 0; q < MAXV; ++q) {
            const int i = threadIdx.x + q * blockDim.x;
            if (i < H4)
                reinterpret_cast<uint2*>(s_xh)[i] =
                    make_uint2(pack_f16x2_chk(v[q].x * ri * w[q].x, v[q].y * ri * w[q].y, bad),
                               pack_f16x2_chk(v[q].z * ri * w[q].z, v[q].w * ri * w[q].w, bad));
        }
        if (bad) raise_status(status, EMBER_ERR_RANGE);
        __syncthreads();
    }
};

// Row dot products by whole warps with the input vector held in registers:
// lane l keeps chunks c = l + 32*i (8 f16 values each) of the input, so
// shared memory only streams the weights.  Eight partial sums per lane, then
// a 5-step butterfly (every lane gets the row's value).
// XI chunks per lane: input length <= XI * 32 * 8 (XI = 4: 1024, 8: 2048); the
// kernels are instantiated for both so that short inputs run no dead code.
template <int XI>
struct XRegs {
    uint4 v[XI];
    __device__ __forceinline__ void load(const uint16_t* xh, int n8) {   // f16 input
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int i = 0; i < XI; ++i) {
            const int c = lane + 32 * i;
            v[i] = c < n8 ? reinterpret_cast<const uint4*>(xh)[c] : make_uint4(0, 0, 0, 0);
        }
    }
};
// Two f16 products accumulated in f32 (fma.rn.f32.f16 takes f16 operands,
// which are exact in f32, so this rounds exactly like fmaf on the converted
// values while skipping the separate conversions).
__device__ __forceinline__ float fma2_h(uint32_t w, uint32_t x, float acc) {
    float d;
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t.reg .f32 t;\n\t"
        "mov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.f16 t, wl, xl, %3;\n\tfma.rn.f32.f16 %0, wh, xh, t;\n\t}"
        : "=f"(d)
        : "r"(w), "r"(x), "f"(acc));
    return d;
}
// dot product of eight f16 pairs, accumulated in order from 0
__device__ __forceinline__ float fma8_h(const uint4& w, const uint4& x) {
    float a = fma2_h(w.x, x.x, 0.f);
    a = fma2_h(w.y, x.y, a);
    a = fma2_h(w.z, x.z, a);
    return fma2_h(w.w, x.w, a);
}

// Four rows at once: the same per-lane chunks for rows r[0..3] (four
// independent streams of loads and FMAs), then a transposing butterfly that
// leaves row ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1) summed in every lane of
// its group of 8 (6 shuffles instead of 20).  Rows may repeat (padding).
template <int XI>
__device__ __forceinline__ float wdot4_f16(const uint4* r0, const uint4* r1, const uint4* r2,
                                           const uint4* r3, const XRegs<XI>& x, int n8) {
    const int lane = threadIdx.x & 31;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int i = 0; i < XI; ++i) {
        const int c = lane + 32 * i;
        if (c < n8) {
            const uint4 xv = x.v[i];
            const uint4 u0 = lds128(r0 + c), u1 = lds128(r1 + c), u2 = lds128(r2 + c), u3 = lds128(r3 + c);
            s0 += fma8_h(u0, xv);
            s1 += fma8_h(u1, xv);
            s2 += fma8_h(u2, xv);
            s3 += fma8_h(u3, xv);
        }
    }
    // lanes 0-15 keep rows 0,1 and lanes 16-31 rows 2,3
    const bool lo16 = lane < 16;
    const float v1 = __shfl_xor_sync(FULL_MASK, lo16 ? s2 : s0, 16);
    const float v2 = __shfl_xor_sync(FULL_MASK, lo16 ? s3 : s1, 16);
    const float a = (lo16 ? s0 : s2) + v1, b = (lo16 ? s1 : s3) + v2;
    // lanes with bit 3 clear keep the first of their two rows
    const bool lo8 = (lane & 8) == 0;
    float t = (lo8 ? a : b) + __shfl_xor_sync(FULL_MASK, lo8 ? b : a, 8);
    t += __shfl_xor_sync(FULL_MASK, t, 4);
    t += __shfl_xor_sync(FULL_MASK, t, 2);
    t += __shfl_xor_sync(FULL_MASK, t, 1);
    return t;
}

}  // namespace

// ================================================================== D1 ==
constexpr int FA_KT = 128;     // keys per K/V tile (the TMA box height)
constexpr int FA_C = 16;       // CTAs per cluster at most (one cluster per kv head)
constexpr int FA_SOLO = 384;   // up to this many keys one CTA of the cluster does the attention

// Shared-memory plan of D1 (host and device compute it the same way).
// Resident (res): two K/V tile buffers and separate q/k/v and o_proj weight
// buffers, all filled before the programmatic-launch wait.  Otherwise one
// tile buffer, and one weight buffer that takes the q/k/v rows, then the
// o_proj rows (or, for CTA 0 alone over more than one tile, the second tile).
struct FaLayout {
    int k, v, k1, v1, w, wo, x, qkv, part, att, qh, wm, cs, red, bar, total;
};
__host__ __device__ inline FaLayout fa_layout(int D, int G, int H, int nr, int no, bool res, int nw = 8) {
    FaLayout L;
    const int tile = FA_KT * D * 2;              // one K (or V) tile, bf16
    int o = 0;
    L.k = o; o += tile;
    L.v = o; o += tile;
    L.k1 = L.v1 = 0;
    if (res) {
        L.k1 = o; o += tile;
        L.v1 = o; o += tile;
    }
    L.w = o;
    const int wb = res ? 2 * nr * H : 2 * (nr * H > no * G * D ? nr * H : no * G * D);
    o += (wb + 1023) / 1024 * 1024;
    L.wo = L.w;
    if (res) {
        L.wo = o;
        o += (2 * no * G * D + 1023) / 1024 * 1024;
    }
    L.x = o; o += ((H * 4 + 15) / 16) * 16;
    L.qkv = o; o += (((G + 2) * D * 4 + 15) / 16) * 16;
    L.part = o; o += ((G * (D + 2) * 4 + 15) / 16) * 16;
    L.att = o; o += ((G * D * 4 + 15) / 16) * 16;
    L.qh = o; o += 16 * D * 2;                    // q as the f16 A tile of the key mma
    L.wm = o; o += nw * G * (D + 2) * 4;          // the warps' (m, l, O) per head
    L.cs = o; o += D * 4;                         // RoPE row of the position: cos | sin
    L.red = o; o += 32 * 4;
    L.bar = o; o += 8 * 8;
    L.total = o + 1024;                           // room to align the base to 1024
    return L;
}

// NW warps: 8 (two CTAs may share an SM), or 16 in the partitioned plan,
// where the CTA has its SM alone and a pass over the keys takes two tiles.
template <int D, int XI, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 2 : 1) k_fused_attn(const __grid_constant__ CUtensorMap k_map,
                                                           const __grid_constant__ CUtensorMap v_map,
                                                           FusedAttnArgs a) {
    constexpr int H2 = D / 2;
    constexpr int NTH = NW * 32;   // threads
    constexpr int TPI = NW / 8;   // K/V tiles per pass (warp w takes keys 16*(w % 8) of tile w / 8)
    constexpr int NSUB = D / 64;               // 64-column TMA sub-tiles per row
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, G = a.NH / a.NKV;
    const int C = a.C;   // CTAs of the cluster (<= FA_C)
    const int Rg = (G + 2) * D;
    const bool res = a.resident != 0;
    const FaLayout Lo = fa_layout(D, G, H, a.nr, a.no, res, NW);
    uint8_t* sK = sm + Lo.k;
    uint8_t* sV = sm + Lo.v;
    uint16_t* sW = reinterpret_cast<uint16_t*>(sm + Lo.w);
    uint16_t* sWo = reinterpret_cast<uint16_t*>(sm + Lo.wo);  // o_proj rows (== sW unless res)
    uint16_t* s_xh = reinterpret_cast<uint16_t*>(sm + Lo.x);  // normed input, f16
    float* s_qkv = reinterpret_cast<float*>(sm + Lo.qkv);    // [G*D q | D k | D v]
    float* s_part = reinterpret_cast<float*>(sm + Lo.part);  // [G][m, l, acc[D]]
    uint16_t* s_atth = reinterpret_cast<uint16_t*>(sm + Lo.att);   // [G*D] merged heads, f16
    uint8_t* sQh = sm + Lo.qh;                                 // [16][D] f16, swizzled
    float* s_wm = reinterpret_cast<float*>(sm + Lo.wm);      // [NW][G][D + 2]
    float* s_red = reinterpret_cast<float*>(sm + Lo.red);
    // mbarriers: 0 q/k/v weights, 1 K/V tile, 2 o_proj weights, 3 q/k/v rows
    // received from the cluster, 4 attention output received from the cluster,
    // 5 second K/V tile buffer
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lo.bar);
    __shared__ int s_err;
    __shared__ int s_ph[2];   // resident mode: phases of the two tile barriers after the speculative copies
    __shared__ float s_sc[16 * NW];   // per head and warp: the weight of the warp's softmax state
    __shared__ float s_ml[2 * 16];    // per head: the maximum and the total of the weighted sums

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = (int)cluster_rank();
    const int g = blockIdx.y;
    const int r0 = r * a.nr, r1 = min(Rg, r0 + a.nr);     // this CTA's rows of the group
    const int o0 = r * a.no, o1 = min(H, o0 + a.no);      // this CTA's o_proj rows
    const int GD = G * D;
    const size_t rowb = (size_t)H * 2;

    // ---- before the wait: immutable weights only ----
    if (tid == 0) {
        s_err = 0;
        for (int i = 0; i < 6; ++i) mbar_init(&bar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (r1 > r0) {
            mbar_expect_tx(&bar[0], (uint32_t)((r1 - r0) * rowb));
            // the group's rows are three runs of the fused [q; k; v] matrix
            int i = r0;
            while (i < r1) {
                int src, run_end;
                if (i < GD) { src = g * GD + i; run_end = GD; }
                else if (i < GD + D) { src = a.NH * D + g * D + (i - GD); run_end = GD + D; }
                else { src = a.NH * D + a.NKV * D + g * D + (i - GD - D); run_end = Rg; }
                const int n = min(r1, run_end) - i;
                bulk_g2s(sW + (size_t)(i - r0) * H, a.wqkv + (size_t)src * H, (uint32_t)(n * rowb), &bar[0]);
                i += n;
            }
        }
    }
    // o_proj rows of this CTA (group g's block, contiguous): resident mode
    // copies them now, otherwise into L2 now and shared memory later
    const uint16_t* wo_cta = a.wo + ((size_t)g * H + o0) * GD;
    const uint32_t wo_bytes = o1 > o0 ? (uint32_t)((o1 - o0) * GD * 2) : 0u;
    auto issue_wo = [&]() {   // one bulk copy: the slice is contiguous
        mbar_expect_tx(&bar[2], wo_bytes);
        bulk_g2s(sWo, wo_cta, wo_bytes, &bar[2]);
    };
    if (res) {
        if (tid == 0 && o1 > o0) issue_wo();
    } else {
        for (uint32_t off = (uint32_t)tid * 16384u; off < wo_bytes; off += NTH * 16384u)
            prefetch_l2(reinterpret_cast<const uint8_t*>(wo_cta) + off, min(16384u, wo_bytes - off));
    }
    constexpr int TILE = FA_KT * D * 2;
    uint8_t* sK1 = res ? sm + Lo.k1 : reinterpret_cast<uint8_t*>(sW);
    uint8_t* sV1 = res ? sm + Lo.v1 : reinterpret_cast<uint8_t*>(sW) + TILE;
    // K/V tile t0.. of plane kz into buffer 0 (sK/sV, barrier 1) or 1 (sK1/sV1, barrier 5)
    auto issue_tile = [&](int t0, int buf, int kz) {
        uint8_t* kd = buf ? sK1 : sK;
        uint8_t* vd = buf ? sV1 : sV;
        uint64_t* b = buf ? &bar[5] : &bar[1];
        mbar_expect_tx(b, (uint32_t)(2 * TILE));
        for (int sb = 0; sb < NSUB; ++sb) {
            tma_load_3d(kd + sb * FA_KT * 128, &k_map, sb * 64, t0, kz, b);
            tma_load_3d(vd + sb * FA_KT * 128, &v_map, sb * 64, t0, kz, b);
        }
    };
    // this CTA's key range [lo, hi) for n_keys keys
    auto key_range = [&](int n_keys, int& lo_, int& hi_) {
        const int per_ = n_keys <= FA_SOLO ? n_keys : (n_keys + C - 1) / C;
        lo_ = n_keys <= FA_SOLO ? (r == 0 ? 0 : n_keys) : min(n_keys, r * per_);
        hi_ = n_keys <= FA_SOLO ? n_keys : min(n_keys, lo_ + per_);
    };
    // Resident mode: the first two K/V tiles of the position the step will
    // use, issued now.  That position is already fixed (an explicit position,
    // or the cursor the previous step left); the rows before it were written
    // by earlier steps.  The embed kernel's checks are read after the wait,
    // and a token they reject or move makes the CTA drain these copies and
    // issue the right ones.
    int spec_seq = -1, spec_pos = -1, spec_n = 0;
    if (res && tid == 0) {
        const int sq = ld_relaxed(a.seqs);
        if (sq >= 0 && sq < a.max_seqs) {
            const int ps = a.positions ? ld_relaxed(a.positions) : ld_relaxed(a.cursor + sq);
            if (ps >= 0 && ps < a.max_len) {
                int slo, shi;
                key_range(ps + 1, slo, shi);
                const int kzs = (sq * a.L + a.layer) * a.NKV + g;
                for (int j = 0; j < 2 && slo + j * FA_KT < shi; ++j) {
                    issue_tile(slo + j * FA_KT, j, kzs);
                    ++spec_n;
                }
                spec_seq = sq;
                spec_pos = ps;
            }
        }
    }
    // The K/V rows this CTA will read, into L2 before the wait: the position
    // is taken from the previous step's resolved position (a hint; the real
    // one is read after the wait), so all keys but the newest are prefetched.
    if (!res) {
        const int hseq = ld_relaxed(a.seqs);
        const int hpos = ld_relaxed(a.tok_pos) + 1;
        if (hseq >= 0 && hseq < a.max_seqs && hpos > 0 && hpos < a.max_len) {
            const int hn = hpos + 1;
            const int hper = hn <= FA_SOLO ? hn : (hn + C - 1) / C;
            const int hlo = hn <= FA_SOLO ? (r == 0 ? 0 : hn) : min(hn, r * hper);
            const int hhi = hn <= FA_SOLO ? hn : min(hn, hlo + hper);
            const size_t row0 = ((size_t)((hseq * a.L + a.layer) * a.NKV + g) * a.max_len + hlo) * D;
            const uint32_t bytes = (uint32_t)(hhi - hlo) * D * 2;
            for (uint32_t off = (uint32_t)tid * 16384u; off < bytes; off += NTH * 16384u) {
                prefetch_l2(reinterpret_cast<const uint8_t*>(a.kc + row0) + off, min(16384u, bytes - off));
                prefetch_l2(reinterpret_cast<const uint8_t*>(a.vc + row0) + off, min(16384u, bytes - off));
            }
        }
    }
    ResidualNorm rn;
    rn.load_w(a.norm_w, H);
    float* s_bias = s_part;   // the biases of this CTA's rows, until the partials are written
    if (a.bqkv && tid < r1 - r0) {
        const int i = r0 + tid;
        int src;
        if (i < GD) src = g * GD + i;
        else if (i < GD + D) src = a.NH * D + g * D + (i - GD);
        else src = a.NH * D + a.NKV * D + g * D + (i - GD - D);
        s_bias[tid] = a.bqkv[src];
    }
    __syncthreads();
    // every CTA's barriers initialised before any remote store: the whole
    // cluster barrier runs before the wait, off the critical path
    cluster_arrive_relaxed();
    cluster_wait();
    pdl_trigger();
    pdl_wait();

    // the step's token state, loaded beside the residual (used after the norm)
    const int ok_raw = __ldcg(a.tok_ok);
    const int pos_raw = __ldcg(a.tok_pos);
    rn.apply<ZSLOTS>(a.x_in, a.z_in, a.x_out, a.z_zero, a.eps, H, g * C + r, a.NKV * C, s_xh, s_red, a.status,
                     a.zs, a.zs);

    const int ok = ok_raw;
    const int pos = ok ? pos_raw : 0;
    const int n_keys = ok ? pos + 1 : 0;
    // short contexts: CTA 0 takes every key and no partials need merging
    const bool solo = n_keys <= FA_SOLO;
    int lo, hi;
    key_range(n_keys, lo, hi);
    const int seq = ok ? a.seqs[0] : 0;
    const int kz = (seq * a.L + a.layer) * a.NKV + g;     // (seq, layer, kv head) plane
    const bool owner = ok && pos >= lo && pos < hi;
    const bool attn_cta = !solo || r == 0;                // receives q/k/v and runs attention
    // Two tiles in flight: always in resident mode; otherwise for CTA 0 alone
    // over more than one tile, the second tile going to the q/k/v weight
    // buffer as soon as the rows are done (the CTA's o_proj rows follow there
    // after attention).
    const bool dual = res || (solo && r == 0 && n_keys > FA_KT && Lo.x - Lo.w >= 2 * TILE);
    if (tid == 0) {
        if (res) {
            // the speculative tiles stand when the step uses their position;
            // otherwise they are drained before the buffers are refilled
            const bool keep = ok && seq == spec_seq && pos == spec_pos;
            int ph0 = 0, ph1 = 0;
            if (!keep) {
                if (spec_n > 0 && !mbar_wait(&bar[1], 0)) s_err = 1;
                if (spec_n > 1 && !mbar_wait(&bar[5], 0)) s_err = 1;
                ph0 = spec_n > 0;
                ph1 = spec_n > 1;
                for (int j = 0; j < 2 && lo + j * FA_KT < hi; ++j) issue_tile(lo + j * FA_KT, j, kz);
            }
            s_ph[0] = ph0;
            s_ph[1] = ph1;
        } else if (hi > lo) {
            issue_tile(lo, 0, kz);
        }
        if (attn_cta) mbar_expect_tx(&bar[3], (uint32_t)(Rg * 4));
        mbar_expect_tx(&bar[4], (uint32_t)(GD * 2));
    }
    float cs_v = 0.f;   // RoPE row of pos (cos | sin), stored to shared memory after the rows
    if (attn_cta && ok && tid < D)
        cs_v = tid < H2 ? __ldg(a.cos_t + (size_t)pos * H2 + tid) : __ldg(a.sin_t + (size_t)pos * H2 + tid - H2);
    float* s_cs = reinterpret_cast<float*>(sm + Lo.cs);

    // ---- this CTA's q/k/v rows (a warp a row quad), sent to the CTAs that
    // run attention: st.async into their shared memory, counted on their
    // barrier 3 ----
    if (r1 > r0 && !mbar_wait(&bar[0], 0)) s_err = 1;
    {
        XRegs<XI> xr;
        xr.load(s_xh, H / 8);
        const int nrow = r1 - r0;
        const int my = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1), l8 = lane & 7;
        for (int base = warp * 4; base < nrow; base += NTH / 8) {   // 4 rows per warp
            const uint4* rp[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                rp[k] = reinterpret_cast<const uint4*>(sW + (size_t)min(base + k, nrow - 1) * H);
            float v = wdot4_f16(rp[0], rp[1], rp[2], rp[3], xr, H / 8) * pow2f(a.qkv_exp);
            const int ri = base + my;
            if (ri < nrow) {
                if (a.bqkv) v += s_bias[ri];
                if (solo) {
                    if (l8 == 0) st_async1(dsmem(&s_qkv[r0 + ri], 0), v, dsmem(&bar[3], 0));
                } else {   // to every CTA of the cluster: lane l8 serves ranks l8, l8 + 8 (< C)
                    for (int cc = l8; cc < C; cc += 8)
                        st_async1(dsmem(&s_qkv[r0 + ri], cc), v, dsmem(&bar[3], cc));
                }
            }
        }
    }
    if (attn_cta && ok && tid < D) s_cs[tid] = cs_v;
    __syncthreads();   // the q/k/v weights are consumed; s_cs is complete

    // o_proj rows into the (now free) weight buffer, while attention runs --
    // or, where the buffer takes the second K/V tile, after attention
    if (tid == 0 && !res) {
        if (dual) issue_tile(lo + FA_KT, 1, kz);
        else if (o1 > o0) issue_wo();
    }

    if (attn_cta) {
        if (!mbar_wait_cluster(&bar[3], 0)) s_err = 1;
        // ---- optional per-head q/k RMSNorm, then RoPE (q pre-scaled, base 2) ----
        if (a.q_norm) {
            for (int h = warp; h < G + 1; h += NTH / 32) {
                float* v = h < G ? s_qkv + h * D : s_qkv + GD;
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
        const float qscale = 1.4426950408889634f * rsqrtf((float)D);
        if (ok) {
            const float* cs = s_cs;
            const float* sn = s_cs + H2;
            for (int e = tid; e < (G + 1) * H2; e += NTH) {
                const int h = e / H2, i = e % H2;
                float* v = h < G ? s_qkv + h * D : s_qkv + GD;
                float r0v, r1v;
                rope_pair(v[i], v[i + H2], cs[i], sn[i], r0v, r1v);
                if (h < G) {
                    v[i] = r0v * qscale;
                    v[i + H2] = r1v * qscale;
                } else {
                    v[i] = r0v;
                    v[i + H2] = r1v;
                }
            }
        }
        __syncthreads();
        if (owner) {   // the new K/V row: to the cache (bf16) and, below, into the tile
            const size_t off = ((size_t)kz * a.max_len + pos) * D;
            for (int d = tid; d < D; d += NTH) {
                a.kc[off + d] = f32_to_bf16(s_qkv[GD + d]);
                a.vc[off + d] = f32_to_bf16(s_qkv[GD + D + d]);
            }
        }

        // ---- flash attention over keys [lo, hi): the G heads are the 16-row A
        // operand of mma.m16n8k16 (rows >= G zero), warp w takes keys 16w..16w+15
        // of each 128-key tile; online softmax per row in registers; P (f16) is
        // the A operand of O += P V ----
        constexpr int KS = D / 16, NT = D / 8;
        for (int e = tid; e < 16 * (D / 8); e += NTH) {
            const int rq = e / (D / 8), cq = e % (D / 8);
            uint4 val = make_uint4(0, 0, 0, 0);
            if (rq < G) {
                const float* q = s_qkv + rq * D + cq * 8;
                val = make_uint4(pack_f16x2(q[0], q[1]), pack_f16x2(q[2], q[3]), pack_f16x2(q[4], q[5]),
                                 pack_f16x2(q[6], q[7]));
            }
            *reinterpret_cast<uint4*>(sQh + q_off<D>(rq, cq)) = val;
        }
        __syncthreads();
        uint32_t qa[KS][4];
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const int mi = lane >> 3;
            ldsm4(sa_u32(sQh + q_off<D>((mi & 1) * 8 + (lane & 7), 2 * kk + (mi >> 1))), qa[kk][0],
                  qa[kk][1], qa[kk][2], qa[kk][3]);
        }
        float o[NT][4];
#pragma unroll
        for (int dn = 0; dn < NT; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows lane/4, lane/4 + 8
        const int g4 = lane >> 2, q4 = lane & 3;
        uint32_t ph0 = res ? (uint32_t)s_ph[0] : 0u, ph1 = res ? (uint32_t)s_ph[1] : 0u;
        for (int t0 = lo, j = 0; t0 < hi; t0 += TPI * FA_KT, j += TPI) {
            // every thread waits for every tile of the pass (uniform phases)
#pragma unroll
            for (int v = 0; v < TPI; ++v) {
                const int tv = t0 + v * FA_KT;
                if (tv < hi) {
                    const int bv = dual ? ((j + v) & 1) : 0;
                    if (!mbar_wait(bv ? &bar[5] : &bar[1], bv ? ph1 : ph0)) s_err = 1;
                    if (bv) ph1 ^= 1;
                    else ph0 ^= 1;
                    if (owner && pos >= tv && pos < min(hi, tv + FA_KT) && tid < D / 8) {   // the row the TMA read stale
                        uint8_t* kt = bv ? sK1 : sK;
                        uint8_t* vt = bv ? sV1 : sV;
                        const int jr = pos - tv, cq = tid;
                        const float* kk8 = s_qkv + GD + cq * 8;
                        const float* vv8 = s_qkv + GD + D + cq * 8;
                        *reinterpret_cast<uint4*>(kt + kv_off(jr, cq)) =
                            make_uint4(pack_bf16x2(kk8[0], kk8[1]), pack_bf16x2(kk8[2], kk8[3]),
                                       pack_bf16x2(kk8[4], kk8[5]), pack_bf16x2(kk8[6], kk8[7]));
                        *reinterpret_cast<uint4*>(vt + kv_off(jr, cq)) =
                            make_uint4(pack_bf16x2(vv8[0], vv8[1]), pack_bf16x2(vv8[2], vv8[3]),
                                       pack_bf16x2(vv8[4], vv8[5]), pack_bf16x2(vv8[6], vv8[7]));
                    }
                }
            }
            __syncthreads();
            const int u = warp / 8, tu = t0 + u * FA_KT;
            const int nt = min(FA_KT, hi - tu);   // <= 0 when this warp's tile is past the range
            const int b = dual ? ((j + u) & 1) : 0;
            uint8_t* sKt = b ? sK1 : sK;
            uint8_t* sVt = b ? sV1 : sV;
            const int r0k = (warp % 8) * 16;
            if (r0k < nt) {   // warp-uniform
                float s[2][4];
#pragma unroll
                for (int n8 = 0; n8 < 2; ++n8) s[n8][0] = s[n8][1] = s[n8][2] = s[n8][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const int mi = lane >> 3;
                    uint32_t b0, b1, b2, b3;
                    ldsm4(sa_u32(sKt + kv_off(r0k + (mi >> 1) * 8 + (lane & 7), 2 * kk + (mi & 1))), b0, b1, b2, b3);
                    mma16816(s[0], qa[kk], bf2_to_h2(b0), bf2_to_h2(b1));
                    mma16816(s[1], qa[kk], bf2_to_h2(b2), bf2_to_h2(b3));
                }
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int n8 = 0; n8 < 2; ++n8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (r0k + n8 * 8 + 2 * q4 + (i & 1) >= nt) s[n8][i] = -INFINITY;
                        if (i < 2) mx0 = fmaxf(mx0, s[n8][i]);
                        else mx1 = fmaxf(mx1, s[n8][i]);
                    }
                mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: key r0k is valid
                const float sc0 = exp2f(m0 - mn0), sc1 = exp2f(m1 - mn1);
                float p[2][4];
#pragma unroll
                for (int n8 = 0; n8 < 2; ++n8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) p[n8][i] = exp2f(s[n8][i] - (i < 2 ? mn0 : mn1));
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
                for (int dn = 0; dn < NT; dn += 2) {
                    const int mi = lane >> 3;
                    uint32_t v0, v1, v2, v3;
                    ldsm4t(sa_u32(sVt + kv_off(r0k + (mi & 1) * 8 + (lane & 7), dn + (mi >> 1))), v0, v1, v2, v3);
                    mma16816(o[dn], pa, bf2_to_h2(v0), bf2_to_h2(v1));
                    mma16816(o[dn + 1], pa, bf2_to_h2(v2), bf2_to_h2(v3));
                }
            }
            __syncthreads();
            // refill the pass's buffers: with two buffers the tiles two on, else the next
            if (tid == 0)
#pragma unroll
                for (int v = 0; v < TPI; ++v) {
                    const int nx = t0 + v * FA_KT + (dual ? 2 : 1) * FA_KT;
                    if (nx < hi) issue_tile(nx, dual ? ((j + v) & 1) : 0, kz);
                }
        }
        if (!res && dual && tid == 0 && o1 > o0) issue_wo();   // the second buffer has been read
        // the 8 warps' states -> this CTA's partial (m, l, acc) per head
        l0 += __shfl_xor_sync(FULL_MASK, l0, 1);
        l0 += __shfl_xor_sync(FULL_MASK, l0, 2);
        l1 += __shfl_xor_sync(FULL_MASK, l1, 1);
        l1 += __shfl_xor_sync(FULL_MASK, l1, 2);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = g4 + 8 * half;
            if (row < G) {
                float* w = s_wm + ((size_t)warp * G + row) * (D + 2);
                if (q4 == 0) {
                    w[0] = half ? m1 : m0;
                    w[1] = half ? l1 : l0;
                }
#pragma unroll
                for (int dn = 0; dn < NT; ++dn) {
                    w[2 + dn * 8 + 2 * q4] = o[dn][2 * half];
                    w[3 + dn * 8 + 2 * q4] = o[dn][2 * half + 1];
                }
            }
        }
        __syncthreads();
        // per head (a warp each): the warps' maxima -> weight f_w of each warp's
        // state and the head's total l; the combine then reads each state once
        for (int hh = warp; hh < G; hh += NW) {
            float mw = -INFINITY, lw = 0.f;
            if (lane < NW) {
                const float* st = s_wm + ((size_t)lane * G + hh) * (D + 2);
                lw = st[1];
                if (lw > 0.f) mw = st[0];
            }
            const float M = warp_max(mw);
            const float f = lw > 0.f ? exp2f(mw - M) : 0.f;
            const float Ls = warp_sum(f * lw);
            if (lane < NW) s_sc[hh * NW + lane] = f;
            if (lane == 0) {
                s_ml[2 * hh] = M;
                s_ml[2 * hh + 1] = Ls;
            }
        }
        __syncthreads();
        // the merged heads go out already rounded to the f16 of the o_proj
        // operand (half the bytes of f32; the range check is the sender's)
        bool bad = false;
        if (solo) {   // CTA 0 holds the whole softmax: normalise and send the heads to every CTA
            for (int e = 4 * tid; e < GD; e += 4 * NTH) {   // D % 4 == 0: one head per quad
                const int hh = e / D, d = e % D;
                float O0 = 0.f, O1 = 0.f, O2 = 0.f, O3 = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float f = s_sc[hh * NW + w];
                    const float* acc = s_wm + ((size_t)w * G + hh) * (D + 2) + 2 + d;
                    O0 = fmaf(acc[0], f, O0);
                    O1 = fmaf(acc[1], f, O1);
                    O2 = fmaf(acc[2], f, O2);
                    O3 = fmaf(acc[3], f, O3);
                }
                const float l = s_ml[2 * hh + 1];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                O0 *= inv; O1 *= inv; O2 *= inv; O3 *= inv;
                const uint32_t h01 = pack_f16x2_chk(O0, O1, bad), h23 = pack_f16x2_chk(O2, O3, bad);
#pragma unroll 4
                for (int cc = 0; cc < C; ++cc) st_async2u(dsmem(&s_atth[e], cc), h01, h23, dsmem(&bar[4], cc));
            }
        } else {
        // this CTA's partial (m, l, acc) per head, for the merge across the cluster
        for (int e = tid; e < G * (D + 2); e += NTH) {
            const int hh = e / (D + 2), k = e % (D + 2);
            float v;
            if (k < 2) {
                v = s_ml[2 * hh + k];
            } else {
                v = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w)
                    v = fmaf(s_wm[((size_t)w * G + hh) * (D + 2) + k], s_sc[hh * NW + w], v);
            }
            s_part[e] = v;
        }
        cluster_sync_all();   // every CTA's partial is in its shared memory

        // ---- merge: CTA r merges element pairs [r*np, (r+1)*np) and broadcasts them ----
        {
            const int GP = GD / 2;   // D is even: a pair never straddles two heads
            const int np = (GP + C - 1) / C;
            const int pi = r * np + tid;
            if (tid < np && pi < GP) {
                const int e = 2 * pi;
                const int h = e / D, d = e % D;
                // log-sum-exp merge of the C partials (empty ranges have l = 0); all
                // 4*C remote loads are issued before the first is used
                float mc[FA_C], lc[FA_C], oa[FA_C], ob[FA_C];
#pragma unroll
                for (int cc = 0; cc < FA_C; ++cc) {
                    mc[cc] = oa[cc] = ob[cc] = 0.f;
                    lc[cc] = 0.f;
                    if (cc < C) {
                        mc[cc] = ld_dsmem(dsmem(&s_part[h * (D + 2)], cc));
                        lc[cc] = ld_dsmem(dsmem(&s_part[h * (D + 2) + 1], cc));
                        oa[cc] = ld_dsmem(dsmem(&s_part[h * (D + 2) + 2 + d], cc));
                        ob[cc] = ld_dsmem(dsmem(&s_part[h * (D + 2) + 3 + d], cc));
                    }
                }
                float M = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < FA_C; ++cc)
                    if (lc[cc] > 0.f) M = fmaxf(M, mc[cc]);
                float Ls = 0.f, Oa = 0.f, Ob = 0.f;
#pragma unroll
                for (int cc = 0; cc < FA_C; ++cc) {
                    if (lc[cc] > 0.f) {
                        const float f = exp2f(mc[cc] - M);
                        Ls = fmaf(lc[cc], f, Ls);
                        Oa = fmaf(oa[cc], f, Oa);
                        Ob = fmaf(ob[cc], f, Ob);
                    }
                }
                const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
                const uint32_t hab = pack_f16x2_chk(Oa * inv, Ob * inv, bad);
#pragma unroll 4
                for (int cc = 0; cc < C; ++cc)
                    st_async1(dsmem(&s_atth[e], cc), __uint_as_float(hab), dsmem(&bar[4], cc));
            }
        }
        }   // !solo
        if (bad) raise_status(a.status, EMBER_ERR_RANGE);
    }   // attn_cta
    // the merged heads, GD f16 values from the cluster; a CTA leaves only
    // after every store aimed at its shared memory has landed
    if (!mbar_wait_cluster(&bar[4], 0)) s_err = 1;

    // ---- o_proj: this CTA's rows of the group's column block, into the residual ----
    if (o1 > o0 && !mbar_wait(&bar[2], 0)) s_err = 1;
    {
        XRegs<XI> xr;
        xr.load(s_atth, GD / 8);
        const int nrow = o1 - o0;
        const int my = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
        for (int base = warp * 4; base < nrow; base += NTH / 8) {   // 4 rows per warp
            const uint4* rp[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                rp[k] = reinterpret_cast<const uint4*>(sWo + (size_t)min(base + k, nrow - 1) * GD);
            const float v = wdot4_f16(rp[0], rp[1], rp[2], rp[3], xr, GD / 8) * pow2f(a.o_exp);
            const int ri = base + my;
            if (ri < nrow && (lane & 7) == 0) red_add(a.z_acc + o0 + ri, v);
        }
    }
    if (tid == 0 && s_err) raise_status(a.status, EMBER_ERR_TIMEOUT);
}

// ================================================================== D2 ==
constexpr int FM_THREADS = 256;

// Chunk = FC intermediate features: 2*FC gate/up rows then FC down_proj^T
// rows, 6*FC*H bytes.  Phase 1 keeps all eight warps on the chunk's gate/up
// rows: a warp takes a quad of rows over one of 16/FC slices of the hidden
// dimension, and the slices' partial sums meet in shared memory.  Phase 2
// (down_proj) gives each thread 8 outputs; when the hidden size leaves half
// of the threads idle, the two halves take the two halves of the chunk's
// features and their sums are added once at the end.
template <int FC, int XI>
__global__ void __launch_bounds__(FM_THREADS, 2) k_fused_mlp(FusedMlpArgs a) {
    constexpr int MAXHG = 2;                      // h-groups of 8 per thread: H <= 4096
    constexpr int QUADS = FC / 2;                 // row quads of a chunk's 2*FC gate/up rows
    constexpr int KSL = (FM_THREADS / 32) / QUADS;   // hidden-dimension slices per quad
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int H = a.H, ns = a.ns, H8 = H / 8;
    const uint32_t stage_bytes = (uint32_t)(6 * FC * H);
    uint8_t* ring = sm;
    uint16_t* s_xh = reinterpret_cast<uint16_t*>(sm + (size_t)ns * stage_bytes);       // normed input
    float* s_y = reinterpret_cast<float*>(sm + (size_t)ns * stage_bytes + ((H * 2 + 15) / 16) * 16);  // [H]
    __shared__ float s_red[32];
    __shared__ float s_g[2][KSL][2 * FC];
    __shared__ __align__(8) uint64_t bar[8];
    __shared__ int s_err;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_chunks = a.F / FC;
    const int my_n = (int)blockIdx.x < n_chunks ? (n_chunks - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto issue = [&](int k) {   // chunk k of this CTA into stage k % ns
        const int ch = blockIdx.x + k * gridDim.x;
        uint8_t* st = ring + (size_t)(k % ns) * stage_bytes;
        mbar_expect_tx(&bar[k % ns], stage_bytes);
        bulk_g2s(st, a.wgu + (size_t)ch * 2 * FC * H, (uint32_t)(4 * FC * H), &bar[k % ns]);
        bulk_g2s(st + 4 * FC * H, a.wdT + (size_t)ch * FC * H, (uint32_t)(2 * FC * H), &bar[k % ns]);
    };
    if (tid == 0) {
        s_err = 0;
        for (int s = 0; s < ns; ++s) mbar_init(&bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int k = 0; k < my_n && k < ns; ++k) issue(k);
    }
    for (int k = ns + tid; k < my_n; k += FM_THREADS) {   // the rest: into L2 now
        const int ch = blockIdx.x + k * gridDim.x;
        prefetch_l2(a.wgu + (size_t)ch * 2 * FC * H, (uint32_t)(4 * FC * H));
        prefetch_l2(a.wdT + (size_t)ch * FC * H, (uint32_t)(2 * FC * H));
    }
    // The last pf_late CTAs launch only when the attention CTAs leave their
    // SMs; the E CTAs before them run beside the attention, so CTA b < E
    // prefetches the chunks of late CTAs E + b, E + b + E, ... into L2 while
    // the attention block computes.
    {
        const int E = (int)gridDim.x - a.pf_late;
        if (a.pf_late > 0 && E > 0 && (int)blockIdx.x < E) {
            for (int lb = E + (int)blockIdx.x; lb < (int)gridDim.x; lb += E)
                for (int ch = lb + tid * (int)gridDim.x; ch < n_chunks; ch += FM_THREADS * (int)gridDim.x) {
                    prefetch_l2(a.wgu + (size_t)ch * 2 * FC * H, (uint32_t)(4 * FC * H));
                    prefetch_l2(a.wdT + (size_t)ch * FC * H, (uint32_t)(2 * FC * H));
                }
        }
    }
    ResidualNorm rn;
    rn.load_w(a.norm_w, H);
    // phase-1 role: row quad qd over the hidden slice [c0, c1) (16-byte units)
    const int qd = warp % QUADS, ks = warp / QUADS;
    const int seg = (H8 + KSL - 1) / KSL;
    const int c0 = min(H8, ks * seg), c1 = min(H8, c0 + seg);
    // phase-2 role: two halves of the features when 2 * H8 threads suffice
    const bool halves = 2 * H8 <= FM_THREADS;
    const int part = halves && tid >= H8 ? 1 : 0;
    const int hgp = tid - part * H8;              // this thread's h-group in halves mode
    __syncthreads();
    pdl_trigger();
    pdl_wait();

    rn.apply<1>(a.x_in, a.z_in, a.x_out, a.z_zero, a.eps, H, blockIdx.x, gridDim.x, s_xh, s_red, a.status, 1, 1);
    XRegs<XI> xr;
    xr.load(s_xh + c0 * 8, c1 - c0);

    float y[MAXHG][8];
#pragma unroll
    for (int q = 0; q < MAXHG; ++q)
#pragma unroll
        for (int u = 0; u < 8; ++u) y[q][u] = 0.f;

    for (int k = 0; k < my_n; ++k) {
        const int s = k % ns;
        if (!mbar_wait(&bar[s], (uint32_t)((k / ns) & 1))) s_err = 1;
        const uint8_t* st = ring + (size_t)s * stage_bytes;
        {   // gate / up rows 4qd..4qd+3 over this warp's slice
            const uint4* rp[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) rp[q] = reinterpret_cast<const uint4*>(st + (size_t)(qd * 4 + q) * H * 2) + c0;
            const float v = wdot4_f16(rp[0], rp[1], rp[2], rp[3], xr, c1 - c0) * pow2f(a.gu_exp);
            const int rr = qd * 4 + ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            if ((lane & 7) == 0) s_g[k & 1][ks][rr] = v;
        }
        __syncthreads();   // s_g[k & 1] complete; chunk k - 1 fully consumed
        if (tid == 0 && k >= 1 && k - 1 + ns < my_n) issue(k - 1 + ns);
        const uint4* wd = reinterpret_cast<const uint4*>(st + (size_t)4 * FC * H);
        if (halves) {
            if (tid < 2 * H8) {
#pragma unroll
                for (int jj = 0; jj < FC / 2; ++jj) {
                    const int j = part * (FC / 2) + jj;
                    float gt = 0.f, up = 0.f;
#pragma unroll
                    for (int z = 0; z < KSL; ++z) {
                        gt += s_g[k & 1][z][2 * j];
                        up += s_g[k & 1][z][2 * j + 1];
                    }
                    const float act = __fdividef(gt, 1.f + __expf(-gt)) * up * pow2f(a.d_exp);
                    float w[8];
                    unpack8_f16(lds128(wd + (size_t)j * H8 + hgp), w);
#pragma unroll
                    for (int u = 0; u < 8; ++u) y[0][u] = fmaf(w[u], act, y[0][u]);
                }
            }
        } else {
            float act[FC];
#pragma unroll
            for (int j = 0; j < FC; ++j) {
                float gt = 0.f, up = 0.f;
#pragma unroll
                for (int z = 0; z < KSL; ++z) {
                    gt += s_g[k & 1][z][2 * j];
                    up += s_g[k & 1][z][2 * j + 1];
                }
                act[j] = __fdividef(gt, 1.f + __expf(-gt)) * up * pow2f(a.d_exp);
            }
#pragma unroll
            for (int q = 0; q < MAXHG; ++q) {
                const int hg = tid + q * FM_THREADS;
                if (hg < H8) {
#pragma unroll
                    for (int j = 0; j < FC; ++j) {
                        float w[8];
                        unpack8_f16(lds128(wd + (size_t)j * H8 + hg), w);
#pragma unroll
                        for (int u = 0; u < 8; ++u) y[q][u] = fmaf(w[u], act[j], y[q][u]);
                    }
                }
            }
        }
    }
    float* z_acc = a.z_acc + (size_t)(blockIdx.x % a.zs) * H;
    if (halves) {   // the second half's sums join the first half's
        if (part == 1 && tid < 2 * H8) {
            reinterpret_cast<float4*>(s_y)[2 * hgp] = make_float4(y[0][0], y[0][1], y[0][2], y[0][3]);
            reinterpret_cast<float4*>(s_y)[2 * hgp + 1] = make_float4(y[0][4], y[0][5], y[0][6], y[0][7]);
        }
        __syncthreads();
        if (part == 0 && tid < H8 && my_n > 0) {
            const float4 b0 = reinterpret_cast<const float4*>(s_y)[2 * tid];
            const float4 b1 = reinterpret_cast<const float4*>(s_y)[2 * tid + 1];
            red_add4(z_acc + 8 * tid, y[0][0] + b0.x, y[0][1] + b0.y, y[0][2] + b0.z, y[0][3] + b0.w);
            red_add4(z_acc + 8 * tid + 4, y[0][4] + b1.x, y[0][5] + b1.y, y[0][6] + b1.z, y[0][7] + b1.w);
        }
    } else {
#pragma unroll
        for (int q = 0; q < MAXHG; ++q) {
            const int hg = tid + q * FM_THREADS;
            if (hg < H8 && my_n > 0) {
                red_add4(z_acc + 8 * hg, y[q][0], y[q][1], y[q][2], y[q][3]);
                red_add4(z_acc + 8 * hg + 4, y[q][4], y[q][5], y[q][6], y[q][7]);
            }
        }
    }
    if (tid == 0 && s_err) raise_status(a.status, EMBER_ERR_TIMEOUT);
}

// ============================================================ D2, resident ==
// The MLP block on its own SMs (the partitioned plan): CTA b owns the
// contiguous features [b*F/grid, (b+1)*F/grid), all of whose gate/up rows and
// down_proj^T rows sit in shared memory before the wait.  Phase 1: the
// gate/up rows in row quads, the hidden dimension in two slices (a warp keeps its slice of the
// normalised input in registers), partial sums in s_g; then SwiGLU per
// feature into s_act.  Phase 2: thread t takes outputs 8*(t % H8).. over one
// of S = 512 / H8 feature slices, the slices meet in the freed gate/up
// buffer, and one red.add.v4 per four outputs goes into the CTA's
// accumulator copy.
constexpr int FR_THREADS = 512;
constexpr int FR_KSL = 2;

__host__ __device__ inline int fr_smem(int nf, int H) {
    return nf * 6 * H + ((H * 2 + 15) / 16) * 16 + ((FR_KSL * 2 * nf * 4 + 15) / 16) * 16 +
           ((nf * 4 + 15) / 16) * 16 + 128;
}

template <int XI>
__global__ void __launch_bounds__(FR_THREADS, 1) k_fused_mlp_res(FusedMlpArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int H = a.H, H8 = H / 8;
    const int f0 = (int)(((long long)blockIdx.x * a.F) / gridDim.x);
    const int f1 = (int)(((long long)(blockIdx.x + 1) * a.F) / gridDim.x);
    const int nf = f1 - f0;
    uint16_t* s_gu = reinterpret_cast<uint16_t*>(sm);                        // [2 nf][H]
    uint16_t* s_wd = s_gu + (size_t)2 * nf * H;                               // [nf][H]
    uint16_t* s_xh = s_wd + (size_t)nf * H;                                   // [H]
    float* s_g = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(s_xh) + ((H * 2 + 15) / 16) * 16);  // [KSL][2 nf]
    float* s_act = s_g + ((FR_KSL * 2 * nf + 3) / 4) * 4;                      // [nf]
    float* s_y = reinterpret_cast<float*>(sm);                                // [S][H] after phase 1
    __shared__ float s_red[32];
    __shared__ __align__(8) uint64_t bar[1];
    __shared__ int s_err;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_err = 0;
        mbar_init(&bar[0], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    ResidualNorm rn;
    rn.load_w(a.norm_w, H);
    // phase-1 role: the warps split into FR_KSL groups, one per hidden slice
    constexpr int WPS = (FR_THREADS / 32) / FR_KSL;   // warps per slice
    const int ks = warp / WPS, wq = warp % WPS;
    const int seg = (H8 + FR_KSL - 1) / FR_KSL;
    const int c0 = min(H8, ks * seg), c1 = min(H8, c0 + seg);
    __syncthreads();
    pdl_trigger();
    // The CTA's weights, ~220 KB, copied by the last thread.  The CTAs of
    // this kernel arrive as the previous MLP block leaves, just when the
    // attention block reads the residual from L2; a 26 MB burst of copies
    // then stalls those reads (measured: 1.2 -> 3-4 us), so the copies start
    // load_delay_ns later (0 without programmatic launch overlap).
    if (tid == FR_THREADS - 1 && nf > 0) {
        if (a.load_delay_ns > 0) {
            const unsigned long long t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < (unsigned long long)a.load_delay_ns) {
            }
        }
        const uint32_t gu_b = (uint32_t)(2 * nf * H * 2), wd_b = (uint32_t)(nf * H * 2);
        mbar_expect_tx(&bar[0], gu_b + wd_b);
        const uint8_t* g_src = reinterpret_cast<const uint8_t*>(a.wgu + (size_t)2 * f0 * H);
        const uint8_t* d_src = reinterpret_cast<const uint8_t*>(a.wdT + (size_t)f0 * H);
        for (uint32_t o = 0; o < gu_b; o += 32768u)
            bulk_g2s(reinterpret_cast<uint8_t*>(s_gu) + o, g_src + o, min(32768u, gu_b - o), &bar[0]);
        for (uint32_t o = 0; o < wd_b; o += 32768u)
            bulk_g2s(reinterpret_cast<uint8_t*>(s_wd) + o, d_src + o, min(32768u, wd_b - o), &bar[0]);
    }
    pdl_wait();

    rn.apply<1>(a.x_in, a.z_in, a.x_out, a.z_zero, a.eps, H, blockIdx.x, gridDim.x, s_xh, s_red, a.status, 1, 1);
    XRegs<XI> xr;
    xr.load(s_xh + c0 * 8, c1 - c0);
    if (nf > 0 && !mbar_wait(&bar[0], 0)) s_err = 1;

    // ---- phase 1: gate / up rows (2 nf of them) over this warp's slice ----
    const int nrow = 2 * nf;
    for (int base = wq * 4; base < nrow; base += WPS * 4) {
        const uint4* rp[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            rp[q] = reinterpret_cast<const uint4*>(s_gu + (size_t)min(base + q, nrow - 1) * H) + c0;
        const float v = wdot4_f16(rp[0], rp[1], rp[2], rp[3], xr, c1 - c0) * pow2f(a.gu_exp);
        const int rr = base + ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
        if ((lane & 7) == 0 && rr < nrow) s_g[ks * nrow + rr] = v;
    }
    __syncthreads();   // s_g complete; the gate/up buffer is free for s_y
    for (int j = tid; j < nf; j += FR_THREADS) {
        float gt = 0.f, up = 0.f;
#pragma unroll
        for (int z = 0; z < FR_KSL; ++z) {
            gt += s_g[z * nrow + 2 * j];
            up += s_g[z * nrow + 2 * j + 1];
        }
        s_act[j] = __fdividef(gt, 1.f + __expf(-gt)) * up * pow2f(a.d_exp);
    }
    __syncthreads();

    // ---- phase 2: SwiGLU and down_proj over feature slice sl, outputs 8 hg.. ----
    const int S = max(1, min(FR_THREADS / H8, nf));
    const int hg = tid % H8, sl = tid / H8;
    if (sl < S && nf > 0) {
        const int j0 = (sl * nf) / S, j1 = ((sl + 1) * nf) / S;
        float y[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = 0.f;
        const uint4* wd = reinterpret_cast<const uint4*>(s_wd);
        for (int j = j0; j < j1; ++j) {
            const float act = s_act[j];
            float w[8];
            unpack8_f16(lds128(wd + (size_t)j * H8 + hg), w);
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] = fmaf(w[u], act, y[u]);
        }
        float4* yo = reinterpret_cast<float4*>(s_y + (size_t)sl * H + 8 * hg);
        yo[0] = make_float4(y[0], y[1], y[2], y[3]);
        yo[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
    __syncthreads();
    float* z_acc = a.z_acc + (size_t)(blockIdx.x % a.zs) * H;
    if (nf > 0)
        for (int i = tid; i < H / 4; i += FR_THREADS) {
            float4 t = reinterpret_cast<const float4*>(s_y)[i];
            for (int q = 1; q < S; ++q) {
                const float4 u = reinterpret_cast<const float4*>(s_y + (size_t)q * H)[i];
                t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
            }
            red_add4(z_acc + 4 * i, t.x, t.y, t.z, t.w);
        }
    if (tid == 0 && s_err) raise_status(a.status, EMBER_ERR_TIMEOUT);
}

// ============================================================= wait probe ==
// Runs one of the kernels' bounded waits on an mbarrier that nothing ever
// completes, with the given budget: the wait gives up, the kernel raises
// EMBER_ERR_TIMEOUT into the status word and returns -- the path every
// waiting kernel takes when a copy or a peer never arrives.
__global__ void k_wait_probe(int which, long long budget, int* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const bool ok = which == 0 ? mbar_wait_for(&bar, 0, budget) : mbar_wait_cluster_for(&bar, 0, budget);
    if (!ok && threadIdx.x == 0) raise_status(status, EMBER_ERR_TIMEOUT);
}

void launch_wait_probe(int which, long long budget, int* status, cudaStream_t s) {
    count_launches(1);
    k_wait_probe<<<1, 32, 0, s>>>(which, budget, status);
}

// ================================================================ host ==
static bool plan_impl(FusedPlan& p, int H, int NH, int NKV, int D, int F, int num_sms, bool allow_part) {
    p = FusedPlan{};
    auto no = [&](const char* why) {
        p.why = why;
        cudaGetLastError();
        return false;
    };
    if (D != 64 && D != 128) return no("head_dim is not 64 or 128");
    if (NH % NKV) return no("n_heads % n_kv_heads != 0");
    const int G = NH / NKV;
    if (G > 16 || H % 8 || H > 2048 || G * D > 2048 || F % 4 || (G * D) % 8)
        return no("group > 16 heads, hidden % 8, hidden or group width > 2048, or ff % 4");
    p.xi = (H <= 1024 && G * D <= 1024) ? 4 : 8;
    const int C = FA_C;
    p.C = C;
    p.nr = ((G + 2) * D + C - 1) / C;
    p.no = (H + C - 1) / C;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return no("device attributes unavailable");
    // Partitioned plan (a layer small enough to sit on chip): the attention
    // clusters take C * NKV SMs with their q/k/v and o_proj rows and two K/V
    // tiles resident, the MLP block takes every other SM with all of its
    // features resident, and neither fits beside the other -- so while one
    // block computes, the next launch of the other is already on its own SMs
    // loading its weights.
    {
        const int n_attn = C * NKV, mg = num_sms - n_attn;
        const int smem_a = fa_layout(D, G, H, p.nr, p.no, true).total;
        if (allow_part && D == 64 && mg >= 1 && F >= mg) {
            const int nfm = (F + mg - 1) / mg;
            const int smem_m = fr_smem(nfm, H);
            // static shared memory of the two kernels, with slack
            if (smem_a <= optin - 4096 && smem_m <= optin - 1024 && smem_a + smem_m > 228 * 1024 &&
                smem_a > 116 * 1024) {
                p.part = true;
                p.zs = ZSLOTS;
                p.mlp_delay_ns = 2000;
                p.smem_attn = smem_a;
                p.smem_mlp = smem_m;
                p.mlp_grid = mg;
            }
        }
    }
    if (!p.part) {
    // more than half an SM's shared memory: one attention CTA per SM, so a
    // cluster spreads over 16 SMs instead of packing two CTAs onto each
    p.smem_attn = fa_layout(D, G, H, p.nr, p.no, false).total;
    if (p.smem_attn < 116 * 1024) p.smem_attn = 116 * 1024;
    if (p.smem_attn > 200 * 1024) return no("attention block needs > 200 KB of shared memory");
    // MLP plan.  Resident: the CTA's chunks all fit its shared memory, so the
    // weights are in place before the wait and nothing is refilled after it;
    // the grid has two CTAs per SM and a CTA fits beside an attention CTA (the
    // CTAs that find no room launch when the attention CTAs leave, their
    // weights prefetched to L2 by the first CTAs).  Otherwise a ring: the
    // largest FC in {16, 8, 4} (dividing F) whose two-stage ring still fits
    // beside the attention kernel on one SM (else FC = 4), one CTA per SM,
    // chunks beyond the ring refilled from L2.
    const int fixed = ((H * 2 + 15) / 16) * 16 + H * 4 + 256;   // s_xh (f16) + s_y (f32) + alignment
    const int budget = 227 * 1024 - p.smem_attn - 2 * 1024;
    p.fc = 0;
    for (int fc : {16, 8, 4}) {
        if (F % fc) continue;
        const int n_chunks = F / fc;
        const int cpc = (n_chunks + 2 * num_sms - 1) / (2 * num_sms);
        const int smem = cpc * 6 * fc * H + fixed;
        if (cpc <= 8 && smem <= budget && 2 * (smem + 1024) <= 228 * 1024) {
            p.fc = fc;
            p.ns = cpc;
            p.mlp_grid = (n_chunks + cpc - 1) / cpc;
            p.smem_mlp = smem;
            p.resident = true;
            p.zs = ZSLOTS;
            p.pf_late = C * NKV < p.mlp_grid ? C * NKV : 0;
            break;
        }
    }
    if (!p.resident) {
        for (int fc : {16, 8, 4})
            if (F % fc == 0 && 2 * 6 * fc * H + fixed <= budget) {
                p.fc = fc;
                break;
            }
        const bool coresident = p.fc != 0;
        if (!coresident) p.fc = 4;
        const int stage = 6 * p.fc * H;
        const int n_chunks = F / p.fc;
        p.mlp_grid = n_chunks < num_sms ? n_chunks : num_sms;
        const int per_cta = (n_chunks + p.mlp_grid - 1) / p.mlp_grid;
        int ns = ((coresident ? budget : 200 * 1024) - fixed) / stage;
        if (ns > per_cta) ns = per_cta;
        if (ns > 8) ns = 8;
        if (ns < 2) ns = 2;
        p.ns = ns;
        p.smem_mlp = ns * stage + fixed;
        // without room beside an attention CTA, the MLP CTAs on the
        // attention's SMs start late: the others prefetch their chunks
        if (!coresident) p.pf_late = C * NKV < p.mlp_grid ? C * NKV : 0;
    }
    if (p.smem_mlp > 227 * 1024) return no("MLP ring does not fit shared memory");
    }   // !p.part
    // The limit is a property of the function, shared by every model in the
    // process: raise it to the device maximum so that no model lowers it
    // below what another one launches with.
    if (p.smem_attn > optin - 1024 || p.smem_mlp > optin - 1024)
        return no("shared memory above the device limit");
    auto setup = [&](auto kern, int) {   // the limit covers static + dynamic shared memory
        cudaFuncAttributes fa{};
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - (int)fa.sharedSizeBytes);
    };
    auto setup_attn = [&](auto kern) {
        setup(kern, p.smem_attn);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    };
    setup_attn(k_fused_attn<64, 4, 8>);
    setup_attn(k_fused_attn<64, 8, 8>);
    setup_attn(k_fused_attn<128, 4, 8>);
    setup_attn(k_fused_attn<128, 8, 8>);
    setup(k_fused_mlp<4, 4>, p.smem_mlp);
    setup(k_fused_mlp<8, 4>, p.smem_mlp);
    setup(k_fused_mlp<16, 4>, p.smem_mlp);
    setup(k_fused_mlp<4, 8>, p.smem_mlp);
    setup(k_fused_mlp<8, 8>, p.smem_mlp);
    setup(k_fused_mlp<16, 8>, p.smem_mlp);
    setup(k_fused_mlp_res<2>, p.smem_mlp);
    setup(k_fused_mlp_res<4>, p.smem_mlp);
    if (e != cudaSuccess) return no("kernel attributes rejected");
    if (p.part) {   // the partitioned MLP kernel's static shared memory must leave room
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, p.xi == 4 ? k_fused_mlp_res<2> : k_fused_mlp_res<4>);
        if (e != cudaSuccess || p.smem_mlp + (int)fa.sharedSizeBytes > optin) p.part = false;
        if (!p.part) return plan_impl(p, H, NH, NKV, D, F, num_sms, false);
    }
    // one cluster of C CTAs must fit somewhere on the chip
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, NKV);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = p.smem_attn;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    e = D == 64 ? (p.xi == 4 ? cudaOccupancyMaxActiveClusters(&n, k_fused_attn<64, 4, 8>, &cfg)
                                 : cudaOccupancyMaxActiveClusters(&n, k_fused_attn<64, 8, 8>, &cfg))
                    : (p.xi == 4 ? cudaOccupancyMaxActiveClusters(&n, k_fused_attn<128, 4, 8>, &cfg)
                                 : cudaOccupancyMaxActiveClusters(&n, k_fused_attn<128, 8, 8>, &cfg));
    if (e != cudaSuccess) return no("cluster occupancy query failed");
    if (n < 1) return no("a cluster of 16 CTAs does not fit");
    // All NKV clusters should be on the chip at once: a cluster that finds no
    // 16 SMs of one GPC free waits for another to finish (on a GB300, seven
    // clusters of 16 fit: the eighth of a Llama-3.2-1B layer started 12 us
    // late).  Fewer CTAs per cluster, each with more of the group's rows, as
    // long as its shared memory allows.
    // EMBER_FUSED_CLUSTER=c (8..15) asks for clusters of c CTAs outright (the
    // same search, started there: tests reach the smaller clusters with it)
    const char* want = getenv("EMBER_FUSED_CLUSTER");
    const int cwant = want ? atoi(want) : 0;
    if (!p.part && (n < NKV || (cwant >= 8 && cwant < C))) {
        for (int c2 = (cwant >= 8 && cwant < C) ? cwant : C - 1; c2 >= 8; --c2) {
            const int nr2 = ((G + 2) * D + c2 - 1) / c2, no2 = (H + c2 - 1) / c2;
            int sm2 = fa_layout(D, G, H, nr2, no2, false).total;
            if (sm2 < 116 * 1024) sm2 = 116 * 1024;
            if (sm2 > 200 * 1024) break;
            cfg.gridDim = dim3(c2, NKV);
            cfg.dynamicSmemBytes = sm2;
            at[0].val.clusterDim.x = c2;
            int n2 = 0;
            e = D == 64 ? (p.xi == 4 ? cudaOccupancyMaxActiveClusters(&n2, k_fused_attn<64, 4, 8>, &cfg)
                                      : cudaOccupancyMaxActiveClusters(&n2, k_fused_attn<64, 8, 8>, &cfg))
                        : (p.xi == 4 ? cudaOccupancyMaxActiveClusters(&n2, k_fused_attn<128, 4, 8>, &cfg)
                                      : cudaOccupancyMaxActiveClusters(&n2, k_fused_attn<128, 8, 8>, &cfg));
            if (e != cudaSuccess) {
                cudaGetLastError();
                e = cudaSuccess;
                break;
            }
            if (n2 >= NKV || c2 == cwant) {
                p.C = c2;
                p.nr = nr2;
                p.no = no2;
                p.smem_attn = sm2;
                if (p.pf_late) p.pf_late = c2 * NKV < p.mlp_grid ? c2 * NKV : 0;   // the attention's SMs
                break;
            }
        }
    }
    p.ok = true;
    p.why = "";
    return true;
}

bool fused_decode_plan(FusedPlan& p, int H, int NH, int NKV, int D, int F, int num_sms) {
    return plan_impl(p, H, NH, NKV, D, F, num_sms, !(getenv("EMBER_NO_PARTITION") && atoi(getenv("EMBER_NO_PARTITION"))));
}

void launch_fused_attn(const void* k_map, const void* v_map, const FusedAttnArgs& a, int xi, int smem,
                       cudaStream_t s) {
    count_launches(1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.C, a.NKV);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = a.C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    const CUtensorMap& km = *reinterpret_cast<const CUtensorMap*>(k_map);
    const CUtensorMap& vm = *reinterpret_cast<const CUtensorMap*>(v_map);
    auto kern = a.D == 64 ? (xi == 4 ? k_fused_attn<64, 4, 8> : k_fused_attn<64, 8, 8>)
                          : (xi == 4 ? k_fused_attn<128, 4, 8> : k_fused_attn<128, 8, 8>);
    trace_launch(reinterpret_cast<const void*>(kern), s);
    cudaLaunchKernelEx(&cfg, kern, km, vm, a);
}

void launch_fused_mlp_res(const FusedMlpArgs& a, int xi, int grid, int smem, cudaStream_t s) {
    const dim3 g(grid), b(FR_THREADS);
    if (xi == 4) launch_k(k_fused_mlp_res<2>, g, b, (size_t)smem, s, a);
    else launch_k(k_fused_mlp_res<4>, g, b, (size_t)smem, s, a);
}

void launch_fused_mlp(const FusedMlpArgs& a, int fc, int xi, int grid, int smem, cudaStream_t s) {
    const dim3 g(grid), b(FM_THREADS);
    if (xi == 4) {
        if (fc == 16) launch_k(k_fused_mlp<16, 4>, g, b, (size_t)smem, s, a);
        else if (fc == 8) launch_k(k_fused_mlp<8, 4>, g, b, (size_t)smem, s, a);
        else launch_k(k_fused_mlp<4, 4>, g, b, (size_t)smem, s, a);
    } else {
        if (fc == 16) launch_k(k_fused_mlp<16, 8>, g, b, (size_t)smem, s, a);
        else if (fc == 8) launch_k(k_fused_mlp<8, 8>, g, b, (size_t)smem, s, a);
        else launch_k(k_fused_mlp<4, 8>, g, b, (size_t)smem, s, a);
    }
}

// wdT[f][h] = wd[h][f] (16-bit elements), 32x32 tiles through shared memory
__global__ void k_transpose16(const uint16_t* in, uint16_t* out, int rows, int cols) {
    __shared__ uint16_t t[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int rr = r0 + i, cc = c0 + threadIdx.x;
        if (rr < rows && cc < cols) t[i][threadIdx.x] = in[(size_t)rr * cols + cc];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int cc = c0 + i, rr = r0 + threadIdx.x;
        if (rr < rows && cc < cols) out[(size_t)cc * rows + rr] = t[threadIdx.x][i];
    }
}

void launch_transpose16(const uint16_t* in, uint16_t* out, int rows, int cols, cudaStream_t s) {
    count_launches(1);
    k_transpose16<<<dim3((cols + 31) / 32, (rows + 31) / 32), dim3(32, 8), 0, s>>>(in, out, rows, cols);
}

}  // namespace ember
