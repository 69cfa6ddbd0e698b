// decode_persistent.cuh -- one batch-1 decode step as a single persistent
// kernel that streams the weights.
//
// One CTA per SM (cooperative launch, all CTAs co-resident).  Warp 0 is the
// producer: one thread walks this CTA's share of every weight matrix in the
// order the step consumes them (per layer: fused q|k|v rows, o_proj rows,
// interleaved gate/up rows, down rows; then the tied LM head) and copies it,
// in chunks of contiguous rows, into a ring of shared-memory slots with
// cp.async.bulk (completion counted on an mbarrier per slot).  Weights never
// depend on activations, so the producer runs ahead across phase and layer
// boundaries, limited only by the ring.  Warps 1..7 are consumers: they stage
// the phase's input vector in shared memory (with the RMSNorm applied), take
// the ring's chunks in order, compute their rows' dot products from shared
// memory and release the slots.  Phases are separated by a grid barrier
// (bounded wait): every phase's input is the whole output of the previous
// one.
//
// Per layer (ember scripts/reference_forward.py forward(), one token):
//   QKV  : qkv = Wqkv . (RMSNorm(x) * w) + b
//   ATTN : per kv head (and split of the keys): q/k-norm, RoPE, K/V row write,
//          GQA attention over the cache (ember internals "grouped-query
//          attention": query head h reads kv head h / G); splits merged by
//          the last one to finish
//   O    : x += Wo . att
//   GU   : act = silu(Wg . xn) * (Wu . xn),  xn = RMSNorm(x) * w
//   D    : x += Wd . act
// then HEAD: logits = E . (RMSNorm(x) * w) with the greedy argmax key, and
// the argmax / cursor write-back.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace ember {

constexpr int PK_CONSUMERS = 7;                         // consumer warps
constexpr int PK_THREADS = 32 * (PK_CONSUMERS + 1);     // + producer warp
constexpr int PK_CT = 32 * PK_CONSUMERS;                // consumer threads
constexpr int PK_MAXG = 16;
constexpr int PK_MAX_SPLITS = 32;                       // as the split-KV partial buffer
constexpr long long PK_WAIT_CYCLES = 1ll << 31;         // ~1 s at 2 GHz
constexpr int PK_MAX_CTAS = 1024;                       // barrier epoch slots
constexpr int PK_MAX_ROWS = PK_CT;                      // rows of a residual / bias phase per CTA

enum PhaseKind : int { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_D = 3, PH_HEAD = 4 };

__device__ __forceinline__ uint32_t pk_smem(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void pk_mbar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(pk_smem(b)), "r"(n));
}
__device__ __forceinline__ bool pk_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(pk_smem(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on an mbarrier phase; false after ~1 s.
__device__ __forceinline__ bool pk_wait(uint64_t* b, uint32_t parity) {
    if (pk_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!pk_try_wait(b, parity))
        if (clock64() - t0 > PK_WAIT_CYCLES) return false;
    return true;
}
__device__ __forceinline__ void pk_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(pk_smem(b)) : "memory");
}
__device__ __forceinline__ void pk_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(pk_smem(b)),
                 "r"(bytes)
                 : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned address and size).
__device__ __forceinline__ void pk_bulk_load(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(pk_smem(dst)),
        "l"(src), "r"(bytes), "r"(pk_smem(bar))
        : "memory");
}
// Named barrier over the consumer warps only (the producer keeps streaming).
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(PK_CT) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Loads through L2 written as volatile asm: the compiler keeps a batch of
// them back to back, so they are all in flight before the first use.
__device__ __forceinline__ uint4 ldcg_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldcg_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ldcg_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier over all CTAs (their consumer threads).  bar[0] = abort word,
// bar[32 + i] = epoch of CTA i.  Each CTA publishes its new epoch with a
// release store; the first consumer warp polls every CTA's epoch (no atomic
// hot spot) until all have reached it, then acquires.  The wait is bounded: a
// timeout raises EMBER_ERR_TIMEOUT and sets abort, after which every barrier
// passes at once, so a stuck CTA cannot hang the others.
__device__ __forceinline__ void grid_sync(unsigned* bar, unsigned& epoch, int* status) {
    consumer_sync();
    if (threadIdx.x >= 32 && threadIdx.x < 64) {   // the first consumer warp
        const int lane = threadIdx.x & 31;
        unsigned* flags = bar + 32;
        ++epoch;
        if (lane == 0) st_release(flags + blockIdx.x, epoch);
        const long long t0 = clock64();
        while (true) {
            bool all = true;
            for (int j = lane; j < (int)gridDim.x; j += 32)
                all &= (int)(ld_relaxed(flags + j) - epoch) >= 0;
            if (__all_sync(FULL_MASK, all)) break;
            if (ld_relaxed(bar)) break;
            if (clock64() - t0 > PK_WAIT_CYCLES) {
                if (lane == 0) {
                    atomicExch(bar, 1u);
                    raise_status(status, EMBER_ERR_TIMEOUT);
                }
                break;
            }
        }
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    consumer_sync();
}

// Rows [r0, r1) of a phase's matrix owned by CTA `cta`: an even number of
// consecutive rows (gate/up pairs stay together).
__device__ __forceinline__ void pk_rows(int N, int cta, int ncta, int& r0, int& r1) {
    int per = (N + ncta - 1) / ncta;
    per += per & 1;
    r0 = min(N, cta * per);
    r1 = min(N, r0 + per);
}

struct PkMat {
    const uint16_t* W;
    int N, K;
};

__device__ __forceinline__ PkMat pk_mat(const PersistArgs& a, int kind, int l) {
    const PersistLayer& L = a.layers[l];
    switch (kind) {
        case PH_QKV: return {L.wqkv, a.qkv_n, a.H};
        case PH_O: return {L.wo, a.H, a.NH * a.D};
        case PH_GU: return {L.wgu, 2 * a.F, a.H};
        case PH_D: return {L.wd, a.H, a.F};
        default: return {a.embed, a.V, a.H};
    }
}

// Rows per ring chunk for a matrix of row length K (even, >= 2).
__device__ __forceinline__ int pk_chunk_rows(const PersistArgs& a, int K) {
    int r = a.chunk_bytes / (K * 2);
    r -= r & 1;
    return r < 2 ? 2 : r;
}

// ------------------------------------------------------------- producer --
static __device__ void pk_producer(const PersistArgs& a, uint8_t* ring, uint64_t* full, uint64_t* empty) {
    const int cta = blockIdx.x, ncta = gridDim.x;
    uint32_t n = 0;   // chunk counter (the consumers count identically)
    auto stream_phase = [&](int kind, int l) -> bool {
        const PkMat m = pk_mat(a, kind, l);
        int r0, r1;
        pk_rows(m.N, cta, ncta, r0, r1);
        const int rc = pk_chunk_rows(a, m.K);
        for (int r = r0; r < r1; r += rc, ++n) {
            const int rows = min(rc, r1 - r);
            const uint32_t slot = n % a.ring_slots, it = n / a.ring_slots;
            if (!pk_wait(&empty[slot], (it & 1u) ^ 1u)) return false;
            const uint32_t bytes = (uint32_t)rows * m.K * 2;
            pk_expect_tx(&full[slot], bytes);
            pk_bulk_load(ring + (size_t)slot * a.chunk_bytes, m.W + (size_t)r * m.K, bytes,
                         &full[slot]);
        }
        return true;
    };
    for (int l = 0; l < a.L; ++l)
        for (int kind = PH_QKV; kind <= PH_D; ++kind)
            if (!stream_phase(kind, l)) return;
    stream_phase(PH_HEAD, 0);
}

// ------------------------------------------------------------- consumers --
struct PkCtx {
    const PersistArgs* a;
    uint8_t* ring;
    uint64_t* full;
    uint64_t* empty;
    float* xs;          // staged phase input (f32)
    uint32_t n;         // chunk counter
    int ctid, cw, lane;
    bool ok;            // false after a ring timeout: stop consuming
    unsigned epoch;     // this CTA's grid-barrier epoch
    float* rows;        // [PK_MAX_ROWS] per-row epilogue operand of this CTA's rows
};

// Consume this CTA's chunks of one phase and hand (row, value[, value of
// the pair's second row]) to the epilogue.  Two mappings:
//  * row mode (a chunk has at least as many rows as there are consumer
//    warps): each warp takes RB rows at once (RB/2 gate/up pairs), lanes
//    stride over K, so every staged input element is loaded once for RB
//    independent dot products;
//  * split-K mode (fewer rows than warps, long rows): every warp takes a
//    slice of K for all of the chunk's rows; partial sums meet in shared
//    memory.
constexpr int PK_RB = 4;          // rows per warp per pass (row mode)
constexpr int PK_SPLIT_ROWS = 16;  // a wave with at most this many rows runs split-K

// Address of row `row` of a wave that starts at row wr0 in ring chunk n0.
__device__ __forceinline__ const uint4* pk_row_ptr(const PkCtx& c, int row, int wr0, uint32_t n0,
                                                   int rc, int K) {
    const int k = (row - wr0) / rc, within = (row - wr0) - k * rc;
    const uint32_t slot = (n0 + k) % c.a->ring_slots;
    return reinterpret_cast<const uint4*>(c.ring + (size_t)slot * c.a->chunk_bytes +
                                          (size_t)within * K * 2);
}

// Split-K pass over the R (>= rows) rows of a wave: thread t takes pieces
// p = t + k*PK_CT of every row; rows past `rows` re-read the first row and are
// dropped; per-warp sums meet in red_rows[warp][R].
template <int R>
__device__ __forceinline__ void pk_split_pass(const PkCtx& c, int rows, int wr0, uint32_t n0,
                                              int rc, int K, const float4* xs4, float* red_rows,
                                              bool f16) {
    const int K8 = K >> 3;
    const uint4* wq[R];
#pragma unroll
    for (int q = 0; q < R; ++q) wq[q] = pk_row_ptr(c, wr0 + (q < rows ? q : 0), wr0, n0, rc, K);
    float acc[R];
#pragma unroll
    for (int q = 0; q < R; ++q) acc[q] = 0.f;
#pragma unroll 2
    for (int p = c.ctid; p < K8; p += PK_CT) {
        const float4 x0 = xs4[2 * p], x1 = xs4[2 * p + 1];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            float wf[8];
            if (f16) unpack8_f16(wq[q][p], wf); else unpack8(wq[q][p], wf);
            float s = acc[q];
            s = fmaf(wf[0], x0.x, s); s = fmaf(wf[1], x0.y, s);
            s = fmaf(wf[2], x0.z, s); s = fmaf(wf[3], x0.w, s);
            s = fmaf(wf[4], x1.x, s); s = fmaf(wf[5], x1.y, s);
            s = fmaf(wf[6], x1.z, s); s = fmaf(wf[7], x1.w, s);
            acc[q] = s;
        }
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
        const float v = warp_sum(acc[q]);
        if (c.lane == 0) red_rows[c.cw * PK_SPLIT_ROWS + q] = v;
    }
}

// Consume this CTA's rows of one phase and hand (row, value[, value of the
// pair's second row]) to the epilogue.  The rows arrive in ring chunks; they
// are taken in waves of up to ring_slots - 2 chunks (the producer keeps
// streaming into the other slots): wait for the wave's chunks, spread all its
// rows over the consumer warps, release the slots.  Mapping per wave:
//  * row mode (many rows): each warp takes PK_RB rows at once (gate/up pairs
//    stay together), lanes stride over K, so every staged input element is
//    loaded once for PK_RB independent dot products;
//  * split-K mode (few, long rows): every thread takes a slice of K for all
//    the wave's rows; partial sums meet in shared memory.
template <class Epi>
__device__ __forceinline__ void pk_consume(PkCtx& c, int kind, int l, float* red_rows, Epi epi) {
    const PersistArgs& a = *c.a;
    const PkMat m = pk_mat(a, kind, l);
    int r0, r1;
    pk_rows(m.N, blockIdx.x, gridDim.x, r0, r1);
    const int rc = pk_chunk_rows(a, m.K);
    const int K8 = m.K >> 3;
    const bool pairs = (kind == PH_GU);
    const bool f16 = (kind != PH_HEAD);   // layer matrices are f16, the tied head bf16
    const float4* xs4 = reinterpret_cast<const float4*>(c.xs);
    const int nchunks = (r1 - r0 + rc - 1) / rc;
    const int W = a.ring_slots > 2 ? a.ring_slots - 2 : 1;
    for (int c0 = 0; c0 < nchunks; c0 += W) {
        const int nc = min(W, nchunks - c0);
        const uint32_t n0 = c.n;
        for (int k = 0; k < nc; ++k) {
            const uint32_t n = n0 + k;
            if (c.ok && !pk_wait(&c.full[n % a.ring_slots], (n / a.ring_slots) & 1u)) {
                c.ok = false;
                raise_status(a.status, EMBER_ERR_TIMEOUT);
            }
        }
        const int wr0 = r0 + c0 * rc;
        const int wrows = min(r1, wr0 + nc * rc) - wr0;
        if (wrows > PK_SPLIT_ROWS) {
            // ---- row mode
            for (int rb = c.cw * PK_RB; c.ok && rb < wrows; rb += PK_CONSUMERS * PK_RB) {
                const int nr = min(PK_RB, wrows - rb);
                const uint4* wq[PK_RB];
#pragma unroll
                for (int q = 0; q < PK_RB; ++q)
                    wq[q] = pk_row_ptr(c, wr0 + rb + (q < nr ? q : nr - 1), wr0, n0, rc, m.K);
                float acc[PK_RB];
#pragma unroll
                for (int q = 0; q < PK_RB; ++q) acc[q] = 0.f;
#pragma unroll 2
                for (int p = c.lane; p < K8; p += 32) {
                    const float4 x0 = xs4[2 * p], x1 = xs4[2 * p + 1];
#pragma unroll
                    for (int q = 0; q < PK_RB; ++q) {
                        float wf[8];
                        if (f16) unpack8_f16(wq[q][p], wf); else unpack8(wq[q][p], wf);
                        float s = acc[q];
                        s = fmaf(wf[0], x0.x, s); s = fmaf(wf[1], x0.y, s);
                        s = fmaf(wf[2], x0.z, s); s = fmaf(wf[3], x0.w, s);
                        s = fmaf(wf[4], x1.x, s); s = fmaf(wf[5], x1.y, s);
                        s = fmaf(wf[6], x1.z, s); s = fmaf(wf[7], x1.w, s);
                        acc[q] = s;
                    }
                }
#pragma unroll
                for (int q = 0; q < PK_RB; ++q) acc[q] = warp_sum(acc[q]);
                if (c.lane == 0) {
                    if (pairs) {
#pragma unroll
                        for (int q = 0; q < PK_RB; q += 2)
                            if (q < nr) epi(wr0 + rb + q, acc[q], acc[q + 1]);
                    } else {
#pragma unroll
                        for (int q = 0; q < PK_RB; ++q)
                            if (q < nr) epi(wr0 + rb + q, acc[q], 0.f);
                    }
                }
            }
        } else {
            // ---- split-K mode; the barriers run whatever c.ok says
            if (c.ok) {
                if (wrows <= 2) pk_split_pass<2>(c, wrows, wr0, n0, rc, m.K, xs4, red_rows, f16);
                else if (wrows <= 4) pk_split_pass<4>(c, wrows, wr0, n0, rc, m.K, xs4, red_rows, f16);
                else if (wrows <= 8) pk_split_pass<8>(c, wrows, wr0, n0, rc, m.K, xs4, red_rows, f16);
                else pk_split_pass<PK_SPLIT_ROWS>(c, wrows, wr0, n0, rc, m.K, xs4, red_rows, f16);
            }
            consumer_sync();
            const int step = pairs ? 2 : 1;
            if (c.ok && c.ctid * step < wrows) {
                const int q = c.ctid * step;
                float v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int w = 0; w < PK_CONSUMERS; ++w) {
                    v0 += red_rows[w * PK_SPLIT_ROWS + q];
                    if (pairs) v1 += red_rows[w * PK_SPLIT_ROWS + q + 1];
                }
                epi(wr0 + q, v0, v1);
            }
            consumer_sync();
        }
        __syncwarp();
        if (c.lane == 0)
            for (int k = 0; k < nc; ++k) pk_arrive(&c.empty[(n0 + k) % a.ring_slots]);
        c.n = n0 + nc;
    }
}

// xs[k] = v[k] * rinv * w[k] over K elements (K % 8 == 0, K <= 8192), rinv =
// 1/sqrt(mean(v^2)+eps) when w != nullptr (RMSNorm; ember
// reference_forward.py rmsnorm()).  v is f32 in global memory, copied with
// cp.async.cg (through L2: other CTAs wrote it; no registers, every copy in
// flight at once), or, when emb != nullptr, the bf16 embedding row.  rsrc /
// [r0, r1): the epilogue's per-row operand (residual x or bias), fetched in
// the same round trip.
static __device__ void pk_stage(PkCtx& c, const float* v, const uint16_t* emb, const float* w, int K,
                                float eps, float* red, const float* rsrc = nullptr, int r0 = 0,
                                int r1 = 0) {
    const int K4 = K >> 2;
    if (rsrc && c.ctid < r1 - r0) c.rows[c.ctid] = __ldcg(rsrc + r0 + c.ctid);
    if (emb) {
        for (int idx = c.ctid; idx < K4; idx += PK_CT) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(emb) + idx);
            reinterpret_cast<float4*>(c.xs)[idx] =
                make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
        }
    } else {
        for (int idx = c.ctid; idx < K4; idx += PK_CT)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(pk_smem(c.xs + 4 * idx)),
                         "l"(v + 4 * idx)
                         : "memory");
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    }
    consumer_sync();
    if (!w) return;
    float ss = 0.f;
    for (int idx = c.ctid; idx < K4; idx += PK_CT) {
        const float4 t = reinterpret_cast<const float4*>(c.xs)[idx];
        ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
    }
    ss = warp_sum(ss);
    if (c.lane == 0) red[c.cw] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < PK_CONSUMERS; ++i) tot += red[i];
    const float rinv = rsqrtf(tot / (float)K + eps);
    for (int idx = c.ctid; idx < K4; idx += PK_CT) {
        const float4 t = reinterpret_cast<const float4*>(c.xs)[idx];
        const float4 ww = __ldg(reinterpret_cast<const float4*>(w) + idx);
        reinterpret_cast<float4*>(c.xs)[idx] =
            make_float4(t.x * rinv * ww.x, t.y * rinv * ww.y, t.z * rinv * ww.z, t.w * rinv * ww.w);
    }
    consumer_sync();
}

// One attention item: kv head g, keys [lo, hi) of the token at position pos
// (32 keys per consumer warp per round).  Each consumer warp takes 32 keys:
// lane j scores key j against the G query heads (q staged in shared memory),
// the warp keeps an online softmax per head, and accumulates P.V with each
// lane owning D/32 consecutive output dims.  The warps' (m, l, acc) are
// merged in shared memory; with several splits the CTA writes a partial and
// the last split to finish merges them (log-sum-exp rescale).
template <int D, int GB>
__device__ void pk_attention(PkCtx& c, int l, int g, int split, int nsplit, int lo, int hi,
                             int pos, int seq, uint8_t* scratch) {
    const PersistArgs& a = *c.a;
    constexpr int H2 = D / 2;
    constexpr int DPL = D >= 32 ? D / 32 : 1;     // output dims per lane
    constexpr int C8 = D / 8;                     // 16-byte pieces of a row
    const int G = a.NH / a.NKV;
    const int tid = c.ctid, lane = c.lane, warp = c.cw;
    float* s_q = reinterpret_cast<float*>(scratch);                   // [PK_MAXG][D]
    float* s_kv = s_q + PK_MAXG * D;                                  // [2][D]
    float* s_wm = s_kv + 2 * D;                                       // [warps][PK_MAXG]
    float* s_wl = s_wm + PK_CONSUMERS * PK_MAXG;                      // [warps][PK_MAXG]
    float* s_wacc = s_wl + PK_CONSUMERS * PK_MAXG;                    // [warps][PK_MAXG][D]
    float* s_mrg = s_wacc + PK_CONSUMERS * PK_MAXG * D;               // [2][32][PK_MAXG]
    float* s_scale = s_mrg + 2 * PK_MAX_SPLITS * PK_MAXG;             // [PK_MAXG]
    int* s_last = reinterpret_cast<int*>(s_scale + PK_MAXG);

    const float* cs = a.cos_t + (size_t)pos * H2;
    const float* sn = a.sin_t + (size_t)pos * H2;
    const PersistLayer& Ly = a.layers[l];
    const size_t head_off = (((size_t)seq * a.L + l) * a.NKV + g) * (size_t)a.max_len * D;
    uint16_t* kc = a.kc + head_off;
    uint16_t* vc = a.vc + head_off;
    const float qscale = 1.4426950408889634f * rsqrtf((float)D);   // log2(e)/sqrt(D)

    // ---- q of the G heads and the new k, v: optional per-head RMSNorm, RoPE
    for (int e = tid; e < G * D; e += PK_CT) s_q[e] = __ldcg(a.qkv + (g * G) * D + e);
    for (int e = G * D + tid; e < GB * D; e += PK_CT) s_q[e] = 0.f;   // heads past G: inert
    for (int e = tid; e < 2 * D; e += PK_CT)
        s_kv[e] = __ldcg(a.qkv + a.NH * D + (e / D) * a.NKV * D + g * D + (e % D));
    consumer_sync();
    if (a.qk_norm) {   // PII-Tracer forward(): per-head RMSNorm before RoPE
        for (int h = warp; h < G + 1; h += PK_CONSUMERS) {
            float* v = h < G ? s_q + h * D : s_kv;
            const float* w = h < G ? Ly.q_norm : Ly.k_norm;
            float ss = 0.f;
            for (int d = lane; d < D; d += 32) ss += v[d] * v[d];
            ss = warp_sum(ss);
            const float ri = rsqrtf(ss / (float)D + a.eps);
            __syncwarp();
            for (int d = lane; d < D; d += 32) v[d] = v[d] * ri * w[d];
        }
        consumer_sync();
    }
    for (int e = tid; e < (G + 1) * H2; e += PK_CT) {
        const int h = e / H2, i = e % H2;
        float* v = h < G ? s_q + h * D : s_kv;
        float r0, r1;
        rope_pair(v[i], v[i + H2], cs[i], sn[i], r0, r1);
        const float f = h < G ? qscale : 1.f;
        v[i] = r0 * f;
        v[i + H2] = r1 * f;
    }
    consumer_sync();
    if (pos >= lo && pos < hi) {   // this split owns the new row
        for (int d = tid; d < D; d += PK_CT) {
            kc[(size_t)pos * D + d] = f32_to_bf16(s_kv[d]);
            vc[(size_t)pos * D + d] = f32_to_bf16(s_kv[D + d]);
        }
        __threadfence();
    }
    consumer_sync();

    // ---- warp-level online softmax over 32 keys per round
    float m[GB], lsum[GB], acc[GB][DPL];
#pragma unroll
    for (int h = 0; h < GB; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[h][t] = 0.f;
    }
    const int dl = lane * DPL;   // first output dim of this lane
    for (int base = lo + warp * 32; base < hi; base += 32 * PK_CONSUMERS) {
        const int j = base + lane;
        const bool valid = j < hi;
        // K row j in registers, V[base + jj][dl .. dl + DPL) for the warp's 32 keys
        uint4 kr[C8];
        const uint16_t* krow = kc + (size_t)(valid ? j : lo) * D;   // a valid row either way
#pragma unroll
        for (int q8 = 0; q8 < C8; ++q8) kr[q8] = ldcg_v4(krow + q8 * 8);
        float s[GB];
#pragma unroll
        for (int h = 0; h < GB; ++h) s[h] = 0.f;
        // all G heads advance together: G independent FMA chains per element
#pragma unroll
        for (int q8 = 0; q8 < C8; ++q8) {
            float kf[8];
            unpack8(kr[q8], kf);
#pragma unroll
            for (int h = 0; h < GB; ++h) {   // branch-free: heads past G have q = 0
                const float4 qa = reinterpret_cast<const float4*>(s_q + h * D)[2 * q8];
                const float4 qb = reinterpret_cast<const float4*>(s_q + h * D)[2 * q8 + 1];
                float d = s[h];
                d = fmaf(qa.x, kf[0], d); d = fmaf(qa.y, kf[1], d);
                d = fmaf(qa.z, kf[2], d); d = fmaf(qa.w, kf[3], d);
                d = fmaf(qb.x, kf[4], d); d = fmaf(qb.y, kf[5], d);
                d = fmaf(qb.z, kf[6], d); d = fmaf(qb.w, kf[7], d);
                s[h] = d;
            }
        }
#pragma unroll
        for (int h = 0; h < GB; ++h) s[h] = valid ? s[h] : -INFINITY;
        float p[GB];
#pragma unroll
        for (int h = 0; h < GB; ++h) {   // branch-free over GB heads
            const float mn = fmaxf(m[h], warp_max(s[h]));
            p[h] = exp2f(s[h] - mn);
            const float sc = exp2f(m[h] - mn);
            lsum[h] = lsum[h] * sc + warp_sum(p[h]);
            m[h] = mn;
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[h][t] *= sc;
        }
        // P.V: V values of this lane's dims for a batch of keys are loaded
        // before they are used (one round trip per batch, not per key).
        constexpr int KB = 16;
        const int nk = min(32, hi - base);
#pragma unroll
        for (int kb = 0; kb < 32; kb += KB) {
            // raw bf16 of this lane's DPL dims (2 per 32-bit word), rows clamped
            // into [lo, hi) so every address is valid; p = 0 masks the extras
            constexpr int WPL = DPL >= 2 ? DPL / 2 : 1;
            uint32_t vr[KB][WPL];
#pragma unroll
            for (int t = 0; t < KB; ++t) {
                const int jj = kb + t < nk ? kb + t : 0;
                const uint16_t* vrow = vc + (size_t)(base + jj) * D + (dl < D ? dl : 0);
                if (DPL == 1) {
                    vr[t][0] = ldcg_u32(reinterpret_cast<const uint16_t*>(
                        reinterpret_cast<uintptr_t>(vrow) & ~uintptr_t(3)));
                } else if (WPL == 1) {
                    vr[t][0] = ldcg_u32(vrow);
                } else {
                    const uint2 u2 = ldcg_v2(vrow);
                    vr[t][0] = u2.x;
                    vr[t][WPL - 1] = u2.y;
                }
            }
            float vv[KB][DPL];
#pragma unroll
            for (int t = 0; t < KB; ++t) {
                if (DPL == 1) {
                    vv[t][0] = (dl & 1) ? bf16_hi(vr[t][0]) : bf16_lo(vr[t][0]);
                } else {
#pragma unroll
                    for (int u = 0; u < DPL; u += 2) {
                        vv[t][u] = bf16_lo(vr[t][u / 2]);
                        vv[t][(u + 1) % DPL] = bf16_hi(vr[t][u / 2]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < KB; ++t) {
#pragma unroll
                for (int h = 0; h < GB; ++h) {
                    const float pj = __shfl_sync(FULL_MASK, p[h], kb + t);
#pragma unroll
                    for (int u = 0; u < DPL; ++u) acc[h][u] = fmaf(pj, vv[t][u], acc[h][u]);
                }
            }
        }
    }
    // ---- merge the consumer warps
#pragma unroll
    for (int h = 0; h < GB; ++h) {
        if (h < G) {
            if (lane == 0) {
                s_wm[warp * PK_MAXG + h] = m[h];
                s_wl[warp * PK_MAXG + h] = lsum[h];
            }
#pragma unroll
            for (int t = 0; t < DPL; ++t)
                if (dl + t < D) s_wacc[((size_t)warp * PK_MAXG + h) * D + dl + t] = acc[h][t];
        }
    }
    consumer_sync();
    float* att = a.att + (size_t)(g * G) * D;
    float* part = a.part + (((size_t)g * PK_MAX_SPLITS + split) * G) * (D + 2);
    for (int e = tid; e < G * D; e += PK_CT) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < PK_CONSUMERS; ++w)
            if (s_wl[w * PK_MAXG + h] > 0.f) M = fmaxf(M, s_wm[w * PK_MAXG + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < PK_CONSUMERS; ++w) {
            const float lw = s_wl[w * PK_MAXG + h];
            if (lw > 0.f) {
                const float f = exp2f(s_wm[w * PK_MAXG + h] - M);
                L += lw * f;
                O += s_wacc[((size_t)w * PK_MAXG + h) * D + d] * f;
            }
        }
        if (nsplit == 1) {
            att[e] = O / L;
        } else {
            part[(size_t)h * (D + 2) + 2 + d] = O;
            if (d == 0) {
                part[(size_t)h * (D + 2) + 0] = M;
                part[(size_t)h * (D + 2) + 1] = L;
            }
        }
    }
    if (nsplit == 1) return;
    __threadfence();
    consumer_sync();
    if (tid == 0) {
        const unsigned done = atomicAdd(&a.counters[g], 1u);
        *s_last = (done == (unsigned)(nsplit - 1));
    }
    consumer_sync();
    if (!*s_last) return;
    __threadfence();
    const float* pb = a.part + ((size_t)g * PK_MAX_SPLITS) * G * (D + 2);
    float* s_pm = s_mrg;
    float* s_pl = s_mrg + PK_MAX_SPLITS * PK_MAXG;
    for (int e = tid; e < nsplit * G; e += PK_CT) {
        s_pm[e] = __ldcg(pb + (size_t)e * (D + 2));
        s_pl[e] = __ldcg(pb + (size_t)e * (D + 2) + 1);
    }
    consumer_sync();
    if (tid < G) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < nsplit; ++s2)
            if (s_pl[s2 * G + tid] > 0.f) M = fmaxf(M, s_pm[s2 * G + tid]);
        float Lsum = 0.f;
        for (int s2 = 0; s2 < nsplit; ++s2) {
            const float lv = s_pl[s2 * G + tid];
            const float f = lv > 0.f ? exp2f(s_pm[s2 * G + tid] - M) : 0.f;   // empty: nothing
            s_pm[s2 * G + tid] = f;
            Lsum += lv * f;
        }
        s_scale[tid] = 1.f / Lsum;
    }
    consumer_sync();
    for (int e = tid; e < G * D; e += PK_CT) {
        const int h = e / D, d = e % D;
        float O = 0.f;
#pragma unroll 8
        for (int s2 = 0; s2 < nsplit; ++s2)
            O = fmaf(__ldcg(pb + ((size_t)s2 * G + h) * (D + 2) + 2 + d), s_pm[s2 * G + h], O);
        att[e] = O * s_scale[h];
    }
    if (tid == 0) a.counters[g] = 0u;
}

template <int D, int GB>
__global__ void __launch_bounds__(PK_THREADS, 1) k_decode_persist(PersistArgs a) {
    extern __shared__ uint8_t pk_raw[];
    uint8_t* sm =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pk_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = sm;
    uint8_t* scratch = ring + (size_t)a.ring_slots * a.chunk_bytes;   // xs / attention scratch
    uint64_t* full = reinterpret_cast<uint64_t*>(scratch + a.scratch_bytes);
    uint64_t* empty = full + a.ring_slots;
    float* red = reinterpret_cast<float*>(empty + a.ring_slots);    // [32]
    unsigned long long* s_best = reinterpret_cast<unsigned long long*>(red + 32);   // [8]
    float* s_rows = reinterpret_cast<float*>(s_best + 8);                            // [PK_MAX_ROWS]
    float* s_redrows = s_rows + PK_MAX_ROWS;                  // [PK_CONSUMERS][PK_SPLIT_ROWS]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.ring_slots; ++s) {
            pk_mbar_init(&full[s], 1);
            pk_mbar_init(&empty[s], PK_CONSUMERS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) pk_producer(a, ring, full, empty);
        return;
    }

    PkCtx c;
    c.a = &a;
    c.ring = ring;
    c.full = full;
    c.empty = empty;
    c.xs = reinterpret_cast<float*>(scratch);
    c.n = 0;
    c.ctid = threadIdx.x - 32;
    c.cw = warp - 1;
    c.lane = lane;
    c.ok = true;
    c.epoch = ld_relaxed(a.bar + 32 + blockIdx.x);   // every CTA ended the last step equal
    c.rows = s_rows;
    const int cta = blockIdx.x, ncta = gridDim.x;

    // ---- token checks (every CTA computes the same; CTA 0 reports) ----
    int id = a.ids[0];
    const int seq = a.seqs[0];
    bool ok = true;
    if (id < 0 || id >= a.V) {   // Falcon-H1 logits(): token outside vocabulary
        if (cta == 0 && c.ctid == 0) raise_status(a.status, EMBER_ERR_TOKEN);
        id = 0;
        ok = false;
    }
    int pos = 0;
    if (seq < 0 || seq >= a.max_seqs) {
        if (cta == 0 && c.ctid == 0) raise_status(a.status, EMBER_ERR_INVALID_ARG);
        ok = false;
    } else {
        const int cur = a.cursor[seq];
        pos = a.positions ? a.positions[0] : cur;
        if (pos < 0 || pos >= a.max_len) {
            if (cta == 0 && c.ctid == 0) raise_status(a.status, EMBER_ERR_CAPACITY);
            ok = false;
            pos = 0;
        } else if (pos != cur) {   // ember internals: explicit position == cursor
            if (cta == 0 && c.ctid == 0) raise_status(a.status, EMBER_ERR_STATE);
        }
    }
    const uint16_t* erow = a.embed + (size_t)id * a.H;

    for (int l = 0; l < a.L; ++l) {
        const PersistLayer& Ly = a.layers[l];
        // ---------------- QKV
        int q0, q1;
        pk_rows(a.qkv_n, cta, ncta, q0, q1);
        const float* bias = Ly.bqkv;
        if (l == 0) {
            // the residual stream starts as the embedding row; each CTA writes
            // the x rows it will own in the o_proj phase
            int o0, o1;
            pk_rows(a.H, cta, ncta, o0, o1);
            for (int k = o0 + c.ctid; k < o1; k += PK_CT) a.x[k] = bf16_to_f32(erow[k]);
            pk_stage(c, nullptr, erow, Ly.attn_norm, a.H, a.eps, red, bias, q0, q1);
        } else {
            pk_stage(c, a.x, nullptr, Ly.attn_norm, a.H, a.eps, red, bias, q0, q1);
        }
        pk_consume(c, PH_QKV, l, s_redrows, [&](int row, float v, float) {
            a.qkv[row] = bias ? v + c.rows[row - q0] : v;
        });
        grid_sync(a.bar, c.epoch, a.status);
        // ---------------- ATTN
        if (ok) {
            const int n_keys = pos + 1;
            int max_sp = ncta / a.NKV;
            max_sp = max_sp < 1 ? 1 : (max_sp > PK_MAX_SPLITS ? PK_MAX_SPLITS : max_sp);
            int per = (n_keys + max_sp - 1) / max_sp;
            per = per < 32 * PK_CONSUMERS ? 32 * PK_CONSUMERS : per;   // one full round at least
            const int nsplit = (n_keys + per - 1) / per;
            for (int item = cta; item < a.NKV * nsplit; item += ncta) {
                const int g = item / nsplit, s = item % nsplit;
                const int lo = s * per, hi = min(n_keys, lo + per);
                pk_attention<D, GB>(c, l, g, s, nsplit, lo, hi, pos, seq, scratch);
                consumer_sync();
            }
        }
        grid_sync(a.bar, c.epoch, a.status);
        // ---------------- O
        int h0, h1;
        pk_rows(a.H, cta, ncta, h0, h1);
        pk_stage(c, a.att, nullptr, nullptr, a.NH * a.D, a.eps, red, a.x, h0, h1);
        pk_consume(c, PH_O, l, s_redrows, [&](int row, float v, float) { a.x[row] = c.rows[row - h0] + v; });
        grid_sync(a.bar, c.epoch, a.status);
        // ---------------- GU
        pk_stage(c, a.x, nullptr, Ly.mlp_norm, a.H, a.eps, red);
        pk_consume(c, PH_GU, l, s_redrows, [&](int row, float g0, float u0) {
            a.act[row >> 1] = g0 / (1.f + __expf(-g0)) * u0;
        });
        grid_sync(a.bar, c.epoch, a.status);
        // ---------------- D
        pk_stage(c, a.act, nullptr, nullptr, a.F, a.eps, red, a.x, h0, h1);
        pk_consume(c, PH_D, l, s_redrows, [&](int row, float v, float) { a.x[row] = c.rows[row - h0] + v; });
        grid_sync(a.bar, c.epoch, a.status);
    }
    // ---------------- HEAD (tied: logits = E . RMSNorm(x)), greedy argmax
    if (c.ctid == 0) s_best[0] = 0ull;
    pk_stage(c, a.x, nullptr, a.final_norm, a.H, a.eps, red);   // ends with consumer_sync
    unsigned long long best = 0ull;
    pk_consume(c, PH_HEAD, 0, s_redrows, [&](int row, float v, float) {
        if (a.logits) a.logits[row] = v;
        const unsigned long long k = argmax_key(v, (uint32_t)row);
        best = k > best ? k : best;
    });
    // whichever thread ran the epilogue holds a running best: fold them all
    if (best) atomicMax(&s_best[0], best);
    consumer_sync();
    if (c.ctid == 0) atomicMax(a.keys, s_best[0]);
    grid_sync(a.bar, c.epoch, a.status);
    if (cta == 0 && c.ctid == 0) {
        const unsigned long long k = *(volatile unsigned long long*)a.keys;
        if (a.argmax) a.argmax[0] = argmax_key_index(k);
        *a.keys = 0ull;
        if (ok) a.cursor[seq] = pos + 1;
    }
}

typedef void (*PkKernel)(PersistArgs);

}  // namespace ember
