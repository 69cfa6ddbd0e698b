// kernels.h -- launch interfaces of the ember kernels (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ember {

// Host-side count of kernel launches (every launch_* call adds its kernels).
void count_launches(long long n);
// Records an event before the launch of kernel fn when the calling thread
// traces a decode step (ember_decode_step_traced); otherwise does nothing.
void trace_launch(const void* fn, cudaStream_t s);
unsigned long long launches_so_far();

// Launch with the programmatic-stream-serialization attribute (PDL) unless
// disabled (EMBER_NO_PDL=1): the kernel may start while its predecessor in
// the stream finishes, and must pdl_wait() before reading its outputs.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args&&... args) {
    count_launches(1);
    trace_launch(reinterpret_cast<const void*>(kern), s);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- embedding --
// x[t] = f32(E[ids[t]]) and the per-token argument checks of a decode step
// (seq in range, position == cursor, position < max_len, id < vocab) or of a
// prefill (start position == cursor).
struct EmbedArgs {
    const uint16_t* E;
    int V, H;
    const int32_t* ids;
    int n;
    float* x;                    // [n][H]
    int* status;
    // decode-step checks (seqs == nullptr for prefill / encode)
    const int32_t* seqs;
    const int32_t* positions;
    const int32_t* cursor;
    int max_seqs, max_len;
    int* tok_ok;                 // [n] 1 = token may touch the cache
    int32_t* tok_pos;            // [n] resolved position (positions[t] or the cursor)
    // prefill check (pf_seq < 0: none)
    int pf_seq, pf_start;
    float* zero0;                // [n][zlen] set to 0 when non-null (residual accumulators)
    float* zero1;
    int zlen;                    // floats per token zeroed in zero0 / zero1 (0: H)
};
void launch_embed(const EmbedArgs& a, cudaStream_t s);

// --------------------------------------------------------------------- GEMV --
// Batch-1..8 decode projections: y[b][n] = rinv_b * sum_k W[n][k] x[b][k] w_k
// with the RMSNorm of x fused into the prologue when norm_w != nullptr.
struct GemvArgs {
    const uint16_t* W;           // [N][K] bf16, or f16 when w_f16 (unused when Wq is set)
    int N, K;
    int w_f16;
    const int8_t* Wq;            // q8_0 weights: codes [N][K] (K % 32 == 0), or nullptr
    const uint16_t* Wd;          // q8_0 scales [N][K/32] (f16 bits)
    const float* x;              // [nb][ldx] f32
    int ldx;
    const float* norm_w;         // [K] f32 or nullptr
    float eps;
    const float* bias;           // [N] f32 or nullptr (EPI_STORE)
    float* out;                  // mode-dependent, row stride ldo
    int ldo;
    int nb;
    int mode;                    // EpiMode
    unsigned long long* keys;    // [nb] argmax keys (EPI_ARGMAX)
    int* status;
    int w_exp;                   // W stored scaled by 2^-w_exp: products multiplied by 2^w_exp
    const float* x_add;          // [x_add_slots][K] summed into x (split-K accumulator copies;
                                 // nb == 1, bf16 W), or nullptr
    int x_add_slots;
};
// Returns the launch's own error (not the thread's pending last error).
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s, int num_sms);

// ------------------------------------------------------- decode attention --
// Split-KV flash decoding: one CTA per (token, kv head, split), all G query
// heads of the kv head together; the last CTA of a (token, kv head) merges the
// splits.  Also applies q/k norm + RoPE and writes the token's K/V row.
struct AttnDecodeArgs {
    const float* qkv;            // [nb][ld_qkv] pre-RoPE q | k | v (biased)
    int ld_qkv;
    int nb, NH, NKV, D, L, layer;
    const int32_t* seqs;
    const int32_t* positions;    // resolved positions (the embed kernel's tok_pos)
    const int* tok_ok;
    uint16_t* kc;                // K cache base [S][L][NKV][max_len][D]
    uint16_t* vc;
    int max_len;
    const float* cos_t;          // [max_len][D/2]
    const float* sin_t;
    const float* q_norm;         // [D] or nullptr
    const float* k_norm;
    float eps;
    float* att;                  // [nb][NH*D] f32 (used when att_b == nullptr)
    uint16_t* att_b;             // [nb][NH*D] f16 GEMM operand, or nullptr
    float* part;                 // split partials
    unsigned* counters;          // [nb*NKV], zero between launches
    int splits;
    int* status;
    const void* k_map;           // host copies of the caches' 3-D TMA maps, or nullptr
    const void* v_map;           // (read by the launcher only)
};
void launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t s);
// The same on the warp tensor cores (decode_attn_mma.cu): head_dim 64 / 128,
// at most 16 query heads per kv head, K/V through the TMA maps.
// launch_attn_decode picks it when the maps are given.
bool attn_decode_mma_supported(int D, int G);
void launch_attn_decode_mma(const AttnDecodeArgs& a, cudaStream_t s);

// Greedy argmax write-back and cursor advance at the end of a step.
struct FinishArgs {
    int nb;
    unsigned long long* keys;    // reset to 0 here
    int32_t* argmax;             // [nb] or nullptr
    // decode: cursor[seqs[b]] = positions[b] + 1 for ok tokens
    const int32_t* seqs;
    const int32_t* positions;
    const int* tok_ok;
    int32_t* cursor;
    // prefill: cursor[pf_seq] = pf_end (pf_seq >= 0)
    int pf_seq, pf_end;
};
void launch_finish(const FinishArgs& a, cudaStream_t s);
void launch_set_cursor(int32_t* cursor, int seq, int pos, cudaStream_t s);

// ------------------------------------------------------------- prefill side --
// xb[t] = f16(RMSNorm(x[t]) * w)   (A operand of the tensor-core GEMMs);
// with zero set, also zero[t][0, zlen) = 0 (the next GEMM's split-K output)
void launch_rmsnorm_h(const float* x, const float* w, float eps, int n, int H, uint16_t* xb,
                      int* status, cudaStream_t s, float* zero = nullptr, int zlen = 0);
// xb[t] = bf16(RMSNorm(x[t]) * w)   (A operand of the tied-head GEMM)
void launch_rmsnorm_bf16(const float* x, const float* w, float eps, int n, int H, uint16_t* xb,
                         cudaStream_t s);
// h[t] = RMSNorm(x[t]) * w  in f32
void launch_rmsnorm_f32(const float* x, const float* w, float eps, int n, int H, float* h,
                        cudaStream_t s);

// q/k norm + RoPE of n tokens; q -> bf16 [n][NH*D]; K, V rows -> bf16 cache.
// Token t of sequence z = t / T_per_seq goes to position pos0 + t % T_per_seq
// of cache rows k + z*seq_stride + g*head_stride + pos*D.
struct RopeKVArgs {
    const float* qkv;
    int ld_qkv;
    int n, NH, NKV, D;
    int T_per_seq, pos0;
    const float* cos_t;
    const float* sin_t;
    const float* q_norm;
    const float* k_norm;
    float eps;
    uint16_t* q_out;             // [n][NH*D] f16 (the attention MMA operand)
    uint16_t* kc;
    uint16_t* vc;
    long long seq_stride, head_stride;
    // nullable: the f16 copy of each new K row (the value the bf16 cache
    // holds) also goes to kh[(z * NKV + g) * kh_pad + pos][D], the tensor-core
    // attention's K operand
    uint16_t* kh;
    int kh_pad;
};
void launch_rope_kv(const RopeKVArgs& a, cudaStream_t s);

// Whole-prompt attention reading K/V rows from the cache layout above.
// Query row t of sequence z sits at position pos0 + t; keys [0, pos0+t] are
// visible when causal, [0, T_per_seq + pos0) otherwise.
struct AttnPrefillArgs {
    const uint16_t* q;           // [n][NH*D] f16, RoPE'd
    int n, NH, NKV, D;
    int T_per_seq, pos0, causal;
    const uint16_t* kc;
    const uint16_t* vc;
    long long seq_stride, head_stride;
    uint16_t* att;               // [n][NH*D] f16 (GEMM operand)
    int* status;
};
void launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t s);

// out[t][j] = sum_k h[t][k] W[j][k] + b[j]  (label head, f32 h)
void launch_cls_head(const float* h, int n, int H, const uint16_t* W, const float* b, int labels,
                     float* out, cudaStream_t s);

// out[b][j] = mean_t h[b*T + t] . W[j] + bias[j] (mean-pooled head; bf16 W, bias)
cudaError_t launch_pooled_head(const float* h, int B, int T, int H, const uint16_t* W, const uint16_t* b,
                               int n_out, float* out, cudaStream_t s);
// dst[0..n) = src[0..n) (f32), ordered after the previous kernel
void launch_copy_f32(float* dst, const float* src, int n, cudaStream_t s);

// Standalone RoPE + bf16 store (kernel-level parity entry point).
void launch_rope_store(const float* x, int n_tok, int n_heads, int D, const float* cos_t,
                       const float* sin_t, uint16_t* out, cudaStream_t s);

// bf16 [n] -> f32 [n] (weight repack of norms / biases)
void launch_bf16_to_f32(const uint16_t* in, float* out, long long n, cudaStream_t s);
// bf16 bits -> f16 bits in place (weight repack of the layer matrices)
// q8_0 quantization of n bf16 values at p (n % 32 == 0): codes q[n], f16
// scales d[n/32]; f16_out (nullable, may be p) receives the f16 of the
// decoded values times 2^-f16_exp.
void launch_q8_0_quantize(const uint16_t* p, long long n, int8_t* q, uint16_t* d, uint16_t* f16_out,
                          int f16_exp, cudaStream_t s);
void launch_bf16_to_f16_inplace(uint16_t* p, long long n, int exp, cudaStream_t s);
// *out = max(*out, max |p[i]|) as f32 bits, over n bf16 values (NaN skipped)
void launch_absmax_bf16(const uint16_t* p, long long n, unsigned* out, cudaStream_t s);

// ----------------------------------------------------------- tcgen05 GEMM --
// D[M,N] = A[M,K] . B[N,K]^T (bf16 in, f32 accumulate in TMEM) with a fused
// epilogue.  A and B are described by TMA tensor maps made by make_gemm_plan.
struct GemmEpilogue {
    int mode;                    // EpiMode (EPI_STORE, EPI_RESID, EPI_SWIGLU, EPI_ARGMAX)
    float* out_f32;              // EPI_STORE / EPI_RESID: [M][ldo]; EPI_ARGMAX: logits or nullptr
    uint16_t* out_h;             // EPI_SWIGLU: [M][ldo] f16 (N/2 columns)
    int ldo;
    const float* bias;           // EPI_STORE, nullable
    unsigned long long* keys;    // EPI_ARGMAX: [M] argmax keys (start at 0)
    int ksplit;                  // set by launch_gemm: K split over grid.z (red.add outputs)
    int w_exp;                   // B is stored scaled by 2^-w_exp: products are multiplied by 2^w_exp
    int zeroed;                  // EPI_STORE: out_f32 is zero, so K may be split
    // Host pointer to a tensor map over the output (make_out_map), or null.
    // The many-row GEMM then writes its EPI_STORE / EPI_RESID / EPI_SWIGLU
    // tiles through shared memory with TMA (EPI_RESID as an f32 reduce-add);
    // the map's rows bound the rows written.
    const void* out_map;
};
// Tensor map over an output [rows][ld] (cols <= ld) for GemmEpilogue.out_map:
// f32 with 32 x 128 boxes, or f16 (the SwiGLU output) with 64 x 128 boxes,
// 128-byte swizzle.  False if the driver rejects it.
bool make_out_map(void* out, const void* ptr, int rows, int cols, int ld, bool f16);

struct GemmPlan {
    alignas(64) unsigned char tmA[128];
    alignas(64) unsigned char tmB[128];
    alignas(64) unsigned char tmB64[128];   // B with a 64-row box (few-row A, split-K)
    int M, N, K;
    int bn;                      // N tile (64, 128 or 256)
    int sms;                     // SMs of the device the plan was made on
    bool f16;                    // operands f16 (else bf16)
    bool ok;
};
// A rows = M (activations), B rows = N (weights); both row-major with K
// contiguous and 16-byte aligned rows.  Returns false if the driver rejects
// the tensor maps.
bool make_gemm_plan(GemmPlan& p, const uint16_t* A, int M, int lda, const uint16_t* B, int N,
                    int ldb, int K, bool f16);
// For m_rows <= 128 (one row tile) the GEMM runs with 64-column tiles and,
// for EPI_STORE / EPI_RESID, splits K across CTAs until about one CTA per SM;
// the partial sums are added with red.global.add, so EPI_STORE then needs a
// zeroed output.  gemm_splits() returns the split launch_gemm will use.
int gemm_splits(const GemmPlan& p, int m_rows, int mode);
// Persistent tiles for m_rows > 128 (gemm_persistent.cu); launch_gemm picks it.
void launch_gemm_persistent(const void* tmA, const void* tmB, int bn, int m_rows, int N, int K,
                            uint32_t idesc, const GemmEpilogue& e, int* status, int sms,
                            cudaStream_t s);
// Encode a bf16 TMA tensor map (rank 2..4, 128-byte swizzle, zero fill out
// of bounds).  dims[0] is the contiguous dimension; strides (rank-1 entries)
// are in bytes.  False if the driver rejects it.
bool encode_map_bf16(void* out, const void* ptr, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);

// m_rows: rows of A actually valid (<= p.M); the rest is ignored.
void launch_gemm(const GemmPlan& p, int m_rows, const GemmEpilogue& e, int* status,
                 cudaStream_t s);

// ------------------------------------------------ tensor-core attention --
// Whole-prompt GQA attention on tcgen05 (head_dim 64 or 128).  Maps: Q over
// the f16 queries [rows][NH*D] (box 64 x 128); K over the f16 copy of the K
// rows Kh [z][keys_pad][D] (3-D, box 64 x 128 x 1); Vt over transposed f16 V
// [z][D][keys_pad] (3-D, box 64 x D x 1).  Query row t of sequence z
// (t < T_per_seq) sits at position pos0 + t; it reads Kh and Vt at z index
// z*NKV + g.
struct AttnTcArgs {
    int T_per_seq, pos0, causal, n_keys;
    int NH, NKV, G;
    uint16_t* att;               // [rows][ld_att] f16 (GEMM operand)
    int ld_att;
    int* status;
};
bool attn_tc_supported(int D);
void launch_attn_tc(const void* map_q, const void* map_k, const void* map_vt, const AttnTcArgs& a,
                    int nseq, int D, cudaStream_t s);
// head_dim 64 / 128, two query tiles per CTA in ping-pong (attn_tc2.cu)
void launch_attn_tc2(const void* map_q, const void* map_k, const void* map_vt, const AttnTcArgs& a,
                     int nseq, int D, cudaStream_t s);

// Vt[z][d][key] = f16(V[z][key][d]) and Kh[z][key][d] = f16(K[z][key][d]) for
// keys < n_keys, 0 for keys in [n_keys, keys_pad): V (and K) rows of index
// z = (z / nkv, z % nkv) start at v + (z/nkv)*v_z_stride + (z%nkv)*v_h_stride
// (the same offsets from k).  kh may be null; Kh rows in [kh_from, n_keys)
// are left alone (the RoPE kernel wrote them).
struct VtArgs {
    const uint16_t *v, *k;
    long long v_z_stride, v_h_stride;
    int nkv, D, n_keys, keys_pad;
    uint16_t *vt, *kh;
    int kh_from;
};
void launch_vt(const VtArgs& a, int zs, cudaStream_t s);

// ------------------------------------------- fused batch-1 decode layer --
// Two kernels per decoder layer (decode_fused.cu).  Residual stream of kernel
// n: x_n = x_in + z_in; the kernel writes x_out = x_n, zeroes z_zero and adds
// its output into z_acc (three rotating accumulators, two x buffers).
// The batch-1 decode's split-K accumulators have ZSLOTS copies of the
// hidden vector: a CTA adds into copy (CTA index % ZSLOTS) and a reader sums
// the copies, so that ZSLOTS times fewer atomic additions meet at one address.
constexpr int ZSLOTS = 8;

struct FusedPlan {
    int C = 0;           // CTAs per cluster (one cluster per kv head)
    int nr = 0, no = 0;  // q/k/v rows and o_proj rows per CTA
    int smem_attn = 0, smem_mlp = 0;
    int ns = 0;          // weight ring stages of the MLP kernel
    int fc = 0;          // intermediate features per MLP chunk (4, 8 or 16)
    int xi = 0;          // 16-byte input chunks per lane in the row dots (4: inputs <= 1024, 8: <= 2048)
    int mlp_grid = 0;
    bool resident = false;   // every MLP CTA's chunks fit its shared memory (ns = chunks per CTA)
    bool part = false;       // partitioned: attention and MLP blocks on disjoint SMs, all weights resident
    int zs = ZSLOTS;         // copies of the MLP block's split-K accumulator (1..ZSLOTS)
    int mlp_delay_ns = 0;    // partitioned: MLP weight copies start this long after the CTA arrives
    int pf_late = 0;         // MLP CTAs that start after the attention (their chunks are prefetched to L2)
    bool ok = false;
    const char* why = "not planned";   // reason when !ok
};
bool fused_decode_plan(FusedPlan& p, int H, int NH, int NKV, int D, int F, int num_sms);

struct FusedAttnArgs {
    const uint16_t* wqkv;        // f16 [q rows | k rows | v rows][H]
    const float* bqkv;           // or nullptr
    const float* norm_w;
    float eps;
    const float* q_norm;         // [D] or nullptr (then k_norm unused)
    const float* k_norm;
    const uint16_t* wo;          // f16 o_proj grouped by kv head: [NKV][H][G*D]
    int H, NH, NKV, D, L, layer;
    const float* x_in;
    const float* z_in;
    float* x_out;
    float* z_zero;
    float* z_acc;
    uint16_t* kc;                // K / V cache [seq][layer][kv head][max_len][D] bf16
    uint16_t* vc;
    int max_len, max_seqs;
    const int32_t* seqs;
    const int32_t* tok_pos;
    const int* tok_ok;
    const int32_t* positions;    // the step's explicit positions (nullptr: the cursor)
    const int32_t* cursor;       // [max_seqs] the cache's cursors
    int resident;                // resident plan: o_proj rows and two K/V tiles loaded before the wait
    int qkv_exp, o_exp;          // storage scales of wqkv / wo (2^-e), undone on the products
    int zs;                      // accumulator copies the MLP block before this one added into
    const float* cos_t;
    const float* sin_t;
    int* status;
    int C, nr, no;
};
// k_map / v_map: 3-D TMA maps (D, max_len, seqs*layers*kv heads), box 64 x 128 x 1
void launch_fused_attn(const void* k_map, const void* v_map, const FusedAttnArgs& a, int xi, int smem,
                       cudaStream_t s);

struct FusedMlpArgs {
    const uint16_t* wgu;         // f16 [2F][H], row 2f gate_f, row 2f+1 up_f
    const uint16_t* wdT;         // f16 [F][H] (down_proj transposed)
    const float* norm_w;
    float eps;
    int H, F;
    const float* x_in;
    const float* z_in;
    float* x_out;
    float* z_zero;
    float* z_acc;
    int* status;
    int ns;
    int pf_late;                 // the last pf_late CTAs start late: the others prefetch their chunks to L2
    int load_delay_ns;           // partitioned plan: delay of the weight copies after the CTA arrives
    int gu_exp, d_exp;           // storage scales of wgu / wdT (2^-e), undone on the products
    int zs;                      // accumulator copies to add into (CTA index % zs)
};
void launch_fused_mlp(const FusedMlpArgs& a, int fc, int xi, int grid, int smem, cudaStream_t s);
// One bounded mbarrier wait that nothing completes (which: 0 the CTA wait,
// 1 the cluster-scope wait), raising EMBER_ERR_TIMEOUT into status.
void launch_wait_probe(int which, long long budget, int* status, cudaStream_t s);
// The partitioned plan's MLP block: grid CTAs of 512 threads on their own SMs.
void launch_fused_mlp_res(const FusedMlpArgs& a, int xi, int grid, int smem, cudaStream_t s);

// ---------------------------------------------------------------- sampler --
// One token per row of logits [B][ldl] (V used): temperature t (t <= 0:
// greedy), top-k (0 < k < V), top-p (0 < p < 1), softmax, inverse-CDF draw
// with r[b] in [0, 1).  sampler.cu.
struct SampleArgs {
    const float* logits;
    int B, V;
    long long ldl;
    float t;
    int k;
    float p;
    const float* r;
    int32_t* out;
};
cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s);

// out[c][r] = in[r][c] for 16-bit elements
void launch_transpose16(const uint16_t* in, uint16_t* out, int rows, int cols, cudaStream_t s);

}  // namespace ember
