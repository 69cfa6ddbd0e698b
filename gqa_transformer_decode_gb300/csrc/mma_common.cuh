// mma_common.cuh -- warp-level tensor-core helpers shared by the decode
// attention kernels: ldmatrix loads, mma.m16n8k16 (f16 in, f32 accumulate),
// bf16 -> f16 pair conversion and the 128-byte-swizzled K/V tile addressing
// of the 64 x 128 TMA box.
#pragma once
#include "common.cuh"

namespace ember {

__device__ __forceinline__ uint32_t sa_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

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
// a bf16 pair -> the same pair as f16 (round to nearest)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t u) { return pack_f16x2(bf16_lo(u), bf16_hi(u)); }

// [16][D] f16 tile, 16-byte chunk c of row r XOR-swizzled by (r & 7)
template <int D>
__device__ __forceinline__ int q_off(int r, int c) {
    return r * (D * 2) + ((c ^ (r & 7)) << 4);
}
// K / V tile as written by the 128-byte-swizzled TMA box (64 elements x 128
// keys per box, D / 64 boxes side by side): chunk c (8 values) of key r
__device__ __forceinline__ int kv_off(int r, int c) {
    return (c >> 3) * (128 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

}  // namespace ember
