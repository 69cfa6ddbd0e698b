// decode_persistent.cu -- host side of the persistent batch-1 decode kernel
// (decode_persistent.cuh): shared-memory plan, occupancy check, cooperative
// launch.
#include "decode_persistent.cuh"

namespace ember {

// ------------------------------------------------------------------- host --
static size_t pk_attn_scratch(int D) {
    return (size_t)PK_MAXG * D * 4 + 2 * D * 4 + 2 * PK_CONSUMERS * PK_MAXG * 4 +
           (size_t)PK_CONSUMERS * PK_MAXG * D * 4 + 2 * PK_MAX_SPLITS * PK_MAXG * 4 +
           PK_MAXG * 4 + 16;
}

static bool pk_config(PersistArgs& a, int& smem_total) {
    const int max_smem = 227 * 1024;
    const int q = a.NH * a.D;
    int kmax = a.H > a.F ? a.H : a.F;
    kmax = kmax > q ? kmax : q;
    if (kmax > 8192) return false;
    if (a.NH / a.NKV > PK_MAXG) return false;
    // rows of the bias / residual phases one CTA owns must fit the row buffer
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if ((a.qkv_n + sms - 1) / sms + 1 > PK_MAX_ROWS || (a.H + sms - 1) / sms + 1 > PK_MAX_ROWS)
        return false;
    size_t scratch = (size_t)kmax * 4;
    const size_t att = pk_attn_scratch(a.D);
    scratch = scratch > att ? scratch : att;
    scratch = (scratch + 1023) / 1024 * 1024;
    const int chunk = 32 * 1024;
    const int tail = 1024 /*alignment slack*/ + 256 /*reductions*/ + PK_MAX_ROWS * 4 +
                     PK_CONSUMERS * PK_SPLIT_ROWS * 4;
    const int slots = (int)((max_smem - (int)scratch - tail - 2 * 16 * 8) / chunk);
    if (slots < 2) return false;
    // a chunk in split-K mode (fewer rows than consumer warps) holds at most
    // PK_SPLIT_ROWS rows: rows per chunk = chunk / (2K) >= PK_CONSUMERS or
    // <= PK_SPLIT_ROWS always holds since PK_SPLIT_ROWS >= PK_CONSUMERS
    a.ring_slots = slots > 16 ? 16 : slots;
    a.chunk_bytes = chunk;
    a.scratch_bytes = (int)scratch;
    smem_total = a.ring_slots * chunk + (int)scratch + tail + 2 * a.ring_slots * 8;
    return smem_total <= max_smem;
}

// instantiated per head_dim in decode_persistent_d*.cu (compiled in parallel)
PkKernel pk_kernel_d16(int G);
PkKernel pk_kernel_d32(int G);
PkKernel pk_kernel_d64(int G);
PkKernel pk_kernel_d128(int G);

static PkKernel pk_kernel(const PersistArgs& a) {
    const int G = a.NH / a.NKV;
    switch (a.D) {
        case 16: return pk_kernel_d16(G);
        case 32: return pk_kernel_d32(G);
        case 64: return pk_kernel_d64(G);
        case 128: return pk_kernel_d128(G);
        default: return nullptr;
    }
}

bool persist_prepare(PersistArgs& a, int& grid, int& smem) {
    PkKernel k = pk_kernel(a);
    if (!k || !pk_config(a, smem)) return false;
    // a per-function limit shared by all models: set it to the device maximum
    int cur_dev = 0, optin = 0;
    cudaFuncAttributes fa{};
    if (cudaGetDevice(&cur_dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, cur_dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, k) != cudaSuccess || smem > optin - (int)fa.sharedSizeBytes ||
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, PK_THREADS, smem) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        return false;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    grid = sms > PK_MAX_CTAS ? PK_MAX_CTAS : sms;
    return true;
}

cudaError_t launch_persist(const PersistArgs& a, int grid, int smem, cudaStream_t s) {
    PkKernel k = pk_kernel(a);
    if (!k) return cudaErrorInvalidValue;
    count_launches(1);
    trace_launch(reinterpret_cast<const void*>(k), s);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace ember
