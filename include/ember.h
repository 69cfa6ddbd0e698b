/*
 * ember.h -- C ABI of the GB300 (sm_103a) decoder forward library.
 *
 * One forward pass of a Llama/Qwen2-style decoder-only transformer: embedding
 * gather; per layer RMSNorm, q/k/v projections (optional biases, optional
 * per-head q/k RMSNorm), rotate-half RoPE (plain or llama3-scaled),
 * grouped-query attention over a causal bf16 KV cache (or unmasked, for the
 * bidirectional encoder variant), o_proj and a SwiGLU MLP; then a final
 * RMSNorm, a tied LM head (or a linear label head) and greedy argmax.  It runs
 * as one prefill followed by one cached decode step per new token.
 *
 * Where each operation is defined (page title, section / function):
 *   ember, scripts/reference_forward.py: forward() -- rmsnorm, q/k/v + bias,
 *     rope() rotate-half, KV append, per-head GQA loop, o_proj, SwiGLU, tied
 *     head; main() -- the greedy loop; load_safetensors() -- bf16 decode.
 *   LowLlamaBasic, reference.py: predict() -- rotary_cos_sin() with llama3
 *     scaling, self_attn() causal whole-sequence attention.
 *   PII-Tracer-vLLM, serving/reference_forward.py: forward() -- per-head q/k
 *     RMSNorm before RoPE, bidirectional attention, token_cls_head (+ bias).
 *   Falcon-H1-0.5B-Rust, src/lib.rs: Config::validate and logits()/generate()
 *     -- the argument errors mirrored by EMBER_ERR_INVALID_ARG / _TOKEN.
 *   ember internals: "ForwardModel trait" -- create_cache(max_seq_len) and
 *     forward_with_cache(ids, cache, start_pos), the shape of this ABI;
 *     "kv cache" -- one contiguous block per layer, a cursor that advances once
 *     per token after all layers, explicit positions (the prefill bug);
 *     "qk_scratch" -- no allocation on the hot path.
 *
 * Conventions for every call:
 *   - Pointers named ids / seqs / positions / logits / argmax / hidden / out and
 *     every weight pointer are DEVICE pointers (cudaMalloc'd or equivalent);
 *     every other pointer is a host pointer.
 *   - Calls that take a stream are asynchronous on it: the library enqueues
 *     kernels and returns.  Argument errors detectable on the host return at
 *     once; errors that depend on device data (a token id >= vocab, a position
 *     that disagrees with the cache cursor) raise a device-side status that
 *     ember_sync_status() reports.  The kernels never read or write outside
 *     their buffers on such errors: the offending token is skipped.
 *   - Nothing allocates device memory after ember_model_create / ember_kv_alloc
 *     except the first decode call of a new (batch, pointer) signature, which
 *     instantiates a CUDA graph for it.
 *   - ember_last_error() returns a thread-local message for the last failure.
 *   - Only one stream may use a given model at a time: the model owns one
 *     activation workspace.
 */
#ifndef EMBER_H
#define EMBER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *ember_stream_t;

typedef enum ember_status {
    EMBER_OK = 0,
    EMBER_ERR_INVALID_ARG = 1, /* bad dims, null pointer, n == 0, bad seq index       */
    EMBER_ERR_CAPACITY = 2,    /* start_pos + n > max_len, n > max_tokens, batch too big */
    EMBER_ERR_STATE = 3,       /* a position disagrees with the sequence's cursor        */
    EMBER_ERR_TOKEN = 4,       /* a token id outside [0, vocab) (found on the device)    */
    EMBER_ERR_TIMEOUT = 5,     /* a bounded device wait gave up                          */
    EMBER_ERR_CUDA = 6,        /* a CUDA runtime / driver call failed                    */
    EMBER_ERR_OOM = 7,         /* device allocation failed                               */
    EMBER_ERR_UNSUPPORTED = 8, /* a valid request this build does not serve              */
    EMBER_ERR_RANGE = 9        /* an activation outside the f16 range of the tensor-core
                                  operands (|v| > 65504 or NaN; found on the device)     */
} ember_status;

/* Model hyper-parameters.  Field names follow the HuggingFace config.json
 * fields the pages read (ember reference_forward.py main(); LowLlamaBasic
 * predict(); PII-Tracer forward(): head_dim is explicit, not hidden/heads).
 * Validation (Falcon-H1 Config::validate): every dimension > 0,
 * n_heads % n_kv_heads == 0, head_dim even; this build additionally needs
 * hidden and ff to be multiples of 8 (16-byte weight rows), head_dim one of
 * 16, 32, 64, 128, n_heads/n_kv_heads <= 16, hidden <= 8192, ff <= 16384. */
typedef struct ember_config {
    int32_t vocab, hidden, layers, n_heads, n_kv_heads, head_dim, ff;
    double rope_theta;       /* RoPE base                                         */
    double rms_eps;          /* RMSNorm epsilon                                   */
    int32_t rope_llama3;     /* 1: llama3 frequency scaling (LowLlamaBasic)       */
    double rs_factor, rs_low, rs_high; /* llama3 factor, low/high freq factors   */
    int32_t rs_orig_max_pos; /* llama3 original_max_position_embeddings           */
    int32_t qkv_bias;        /* 1: q/k/v projections carry biases (Qwen2)         */
    int32_t qk_norm;         /* 1: per-head RMSNorm of q and k before RoPE (Qwen3)*/
    int32_t causal;          /* 1: causal decoder; 0: bidirectional encoder       */
    int32_t n_labels;        /* 0: tied LM head over vocab; >0: linear head       */
    int32_t max_tokens;      /* capacity of one prefill / encode / decode call in
                                tokens (0 -> 4096); sizes the workspace           */
    int32_t max_positions;   /* RoPE table length for encode (0 -> max_tokens)    */
    int32_t weights_q8;      /* 1: the layer matrices (q/k/v, o, gate/up, down)
                                are quantized to q8_0 blocks at model creation
                                (ember internals, q8_0: 32 int8 codes per f16
                                scale d, value = code * d; codes = the nearest
                                integer to w / (amax/127), d = f16(amax/127)) and
                                every later product uses the decoded values, not
                                the bf16 inputs.  Needs hidden, ff and
                                n_heads*head_dim to be multiples of 32 and every
                                |w| / 127 within the f16 range (else
                                UNSUPPORTED).  Embedding, head and norms stay as
                                given.                                           */
} ember_config;

/* One layer's weights: device pointers to bf16 bit patterns, HuggingFace
 * [out_features, in_features] row-major.  Biases / q_norm / k_norm may be NULL
 * when the config disables them. */
typedef struct ember_layer_weights {
    const uint16_t *attn_norm;          /* [hidden]                          */
    const uint16_t *wq, *wk, *wv;       /* [NH*D, hidden], [NKV*D, hidden] x2 */
    const uint16_t *bq, *bk, *bv;       /* [NH*D], [NKV*D], [NKV*D]          */
    const uint16_t *q_norm, *k_norm;    /* [head_dim]                        */
    const uint16_t *wo;                 /* [hidden, NH*D]                    */
    const uint16_t *mlp_norm;           /* [hidden]                          */
    const uint16_t *w_gate, *w_up;      /* [ff, hidden]                      */
    const uint16_t *w_down;             /* [hidden, ff]                      */
} ember_layer_weights;

typedef struct ember_weights {
    const uint16_t *embed;              /* [vocab, hidden]; tied LM head     */
    const uint16_t *final_norm;         /* [hidden]                          */
    const uint16_t *cls_w, *cls_b;      /* [n_labels, hidden], [n_labels]    */
    const ember_layer_weights *layers;  /* HOST array of `layers` entries    */
} ember_weights;

typedef struct ember_model ember_model;
typedef struct ember_kv ember_kv;

/* Validate the config, repack the weights into the library's device layout
 * (fused [q;k;v] rows, interleaved gate/up rows, f32 norms and biases) and
 * allocate the activation workspace for cfg->max_tokens tokens.  The caller
 * keeps ownership of its weight buffers and may free them once this returns
 * (the call synchronises the device).  Errors: INVALID_ARG, OOM, CUDA. */
ember_status ember_model_create(const ember_config *cfg, const ember_weights *w,
                                ember_model **out);
void ember_model_destroy(ember_model *m);

/* Bytes of one bf16 KV cache for max_seqs sequences of max_len positions:
 * layers * 2 (K and V) * n_kv_heads * max_len * head_dim * 2 bytes * max_seqs
 * (ember internals, "kv cache": one contiguous block per layer). */
size_t ember_kv_bytes(const ember_config *cfg, int32_t max_seqs, int32_t max_len);

/* Allocate a zeroed bf16 KV cache ([seq][layer][kv_head][pos][head_dim] for
 * K and for V) and zeroed cursors, plus the RoPE tables for max_len
 * positions.  Errors: INVALID_ARG (max_seqs or max_len <= 0, encoder model),
 * OOM, CUDA. */
ember_status ember_kv_alloc(ember_model *m, int32_t max_seqs, int32_t max_len, ember_kv **out);
/* Synchronises the device, frees the cache and drops the decode graphs
 * captured against it.  A cache may outlive its model (it is then only good
 * for ember_kv_free; ember_kv_layout returns STATE). */
void ember_kv_free(ember_kv *kv);

/* Set sequence seq's cursor to 0 (its rows are left as they are and are
 * overwritten by the next prefill).  Asynchronous on stream. */
ember_status ember_kv_reset(ember_kv *kv, int32_t seq, ember_stream_t stream);

/* Set sequence seq's cursor to pos (0 <= pos <= max_len): rewinds a sequence
 * to an earlier length, keeping rows [0, pos).  Asynchronous on stream.
 * Errors: INVALID_ARG (seq out of range), CAPACITY (pos out of range). */
ember_status ember_kv_set_cursor(ember_kv *kv, int32_t seq, int32_t pos, ember_stream_t stream);

/* Read-only view of the cache for inspection: device base pointers of K and
 * V (bf16 bits) and the element strides of [seq, layer, kv_head, pos]; the
 * head_dim stride is 1. */
ember_status ember_kv_layout(const ember_kv *kv, const uint16_t **k_base,
                             const uint16_t **v_base, int64_t strides[4]);

/* Prefill: run n tokens ids[0..n) of sequence seq at positions
 * start_pos .. start_pos+n-1 through every layer, appending their K/V rows,
 * then advance the cursor to start_pos + n (ember internals, ForwardModel
 * forward_with_cache(ids, cache, start_pos)).
 *   logits  [vocab]   f32, logits of the last position (nullable)
 *   argmax  [1]       int32, greedy token of the last position, lowest index
 *                     among equal maxima (nullable)
 *   hidden  [n,hidden] f32, final-RMSNorm'd states of every position (nullable)
 * Host errors: INVALID_ARG (n <= 0, seq out of range, null ids), CAPACITY
 * (start_pos + n > max_len or n > max_tokens).  Device status: STATE when
 * start_pos != the cursor, TOKEN for an id >= vocab. */
ember_status ember_prefill(ember_model *m, ember_kv *kv, int32_t seq, const int32_t *ids,
                           int32_t n, int32_t start_pos, float *logits, int32_t *argmax,
                           float *hidden, ember_stream_t stream);

/* One cached decode step for `batch` sequences: token ids[b] of sequence
 * seqs[b] at position positions[b] (ember reference_forward.py forward(tok,
 * pos)); afterwards the cursor of seqs[b] is positions[b] + 1.  All arrays are
 * device arrays of `batch` entries; the sequences must be distinct.
 * positions may be NULL: each token then goes at its sequence's cursor, so
 * repeated calls with the same buffers (argmax fed back as ids) replay one
 * CUDA graph.
 *   logits [batch, vocab] f32 (nullable); argmax [batch] int32 (nullable).
 * argmax may be the next call's ids, so a greedy loop needs no host sync.
 * Host errors: INVALID_ARG, CAPACITY (batch > max_tokens or > max_seqs).
 * Device status: STATE (position != cursor), CAPACITY (position >= max_len),
 * INVALID_ARG (seq out of range), TOKEN. */
ember_status ember_decode_step(ember_model *m, ember_kv *kv, int32_t batch, const int32_t *seqs,
                               const int32_t *ids, const int32_t *positions, float *logits,
                               int32_t *argmax, ember_stream_t stream);

/* One decode step exactly as ember_decode_step computes it, run for
 * profiling: each kernel starts only after the previous one has finished (no
 * programmatic launch overlap), with a CUDA event recorded on `stream` before
 * every launch and after the last; the sequence runs as a one-off CUDA graph
 * so that host launch latency leaves no gaps.  Waits for the stream.
 *   launch_us [cap]  device time of launch i (its event to the next event)
 *   names     [cap]  launch i's kernel name as the CUDA runtime reports it
 *                    (mangled; static strings owned by the runtime)
 *   n                the step's number of launches (may exceed cap; entries
 *                    i >= cap are not written)
 * The times are those of serialised launches (each kernel's weight loads no
 * longer overlap its predecessor), an upper bound on a launch's share of a
 * graph-replayed step.  Errors as ember_decode_step, plus INVALID_ARG for a
 * stream that is being captured or NULL trace buffers with cap > 0, and CUDA
 * when an event cannot be created or timed. */
ember_status ember_decode_step_traced(ember_model *m, ember_kv *kv, int32_t batch, const int32_t *seqs,
                                      const int32_t *ids, const int32_t *positions, float *logits,
                                      int32_t *argmax, ember_stream_t stream, float *launch_us,
                                      const char **names, int32_t cap, int32_t *n);

/* Bidirectional (or causal, per the config) forward of B independent
 * sequences of T tokens each, positions restarting at 0 per sequence, no KV
 * cache (PII-Tracer forward()).
 *   out    [B*T, n_labels] f32 label logits (n_labels > 0), or
 *          [B*T, vocab] f32 tied-head logits (n_labels == 0)   (nullable)
 *   hidden [B*T, hidden] f32 final-RMSNorm'd states              (nullable)
 * Host errors: INVALID_ARG, CAPACITY (B*T > max_tokens, T > max_positions). */
ember_status ember_encode(ember_model *m, const int32_t *ids, int32_t B, int32_t T, float *out,
                          float *hidden, ember_stream_t stream);

/* ember_prefill that also records, after every decoder block, the residual
 * stream at the last of the n positions ("ember internals" ForwardModel
 * forward_with_activations: hidden states after each transformer block at
 * the last token, the input of the probe mode).
 *   acts [layers, hidden] f32 (device, required); logits / argmax as in
 *   ember_prefill (nullable).  The cache and its cursor advance as in
 *   ember_prefill.  Errors as ember_prefill, plus INVALID_ARG for NULL acts. */
ember_status ember_prefill_activations(ember_model *m, ember_kv *kv, int32_t seq, const int32_t *ids,
                                       int32_t n, int32_t start_pos, float *acts, float *logits,
                                       int32_t *argmax, ember_stream_t stream);

/* The mean-pooled sensitivity head of the bidirectional encoder
 * (PII-Tracer-vLLM serving/reference_forward.py forward(): the mean over
 * positions of the final-normed states, times the head's weight, plus its
 * bias): out[b][j] = (1/T sum_t hidden[b*T + t]) . w[j] + bias[j].
 *   hidden [B*T, H] f32 (device): the `hidden` output of ember_encode
 *   w      [n_out, H] bf16 bits, bias [n_out] bf16 bits or NULL (device;
 *          the caller's, not copied)
 *   out    [B, n_out] f32 (device)
 * Each column's sum runs in position order.  H <= 12288.  Asynchronous on
 * `stream`.  Errors: INVALID_ARG, CUDA. */
ember_status ember_mean_pooled_head(const float *hidden, int32_t B, int32_t T, int32_t H,
                                    const uint16_t *w, const uint16_t *bias, int32_t n_out,
                                    float *out, ember_stream_t stream);

/* Synchronise the stream, read and clear the device status word.  Returns
 * the first device-side error raised since the last call, else EMBER_OK. */
ember_status ember_sync_status(ember_model *m, ember_stream_t stream);

const char *ember_last_error(void);

/* ---- token sampler ------------------------------------------------------- */

/* One token per row of logits, the five stages of "ember internals" §sampler
 * in order: (1) temperature -- x = logit / temperature when temperature > 0;
 * temperature <= 0 is greedy and returns the first maximal logit (NaN counts
 * as maximal); (2) top-k -- for 0 < top_k < V every x below the top_k-th
 * largest is masked (ties with it are kept; 0 or >= V: no-op); (3) top-p --
 * for 0 < top_p < 1 the x whose softmax probability lies below the smallest
 * probability of the shortest most-probable set holding more than top_p of
 * the mass are masked (otherwise no-op); (4) softmax over the survivors
 * (uniform when every logit is -inf); (5) the first index whose running sum
 * of probabilities, in index order, exceeds r[b] (the last maximal index
 * when rounding leaves r[b] above the total).
 *   logits [B, ldl] f32, the first V columns used      (device)
 *   r      [B] f32 draws in [0, 1), one per row         (device; unused and
 *                                                        nullable when greedy)
 *   out    [B] int32 token ids                          (device)
 * Arithmetic: the division of stage 1 is IEEE f32; stages 2-3 select by exact
 * comparisons of x; the masses of stages 3-5 are exp(x - max) in f32 rounded
 * to multiples of 2^-40 and summed exactly (64-bit integers), so a call is
 * deterministic and its decisions differ from exact arithmetic only for draws
 * (or top_p) within ~1e-6 of a boundary.  Asynchronous on `stream`; reads
 * nothing else and allocates nothing.  Errors: INVALID_ARG (NULL pointers,
 * B or V <= 0, ldl < V, top_k < 0, NaN temperature or top_p), CUDA. */
ember_status ember_sample(const float *logits, int32_t B, int32_t V, int32_t ldl, float temperature,
                          int32_t top_k, float top_p, const float *r, int32_t *out,
                          ember_stream_t stream);

/* ---- kernel-level entry points used by the parity tests ------------------ */

/* The RoPE-and-store step of the K cache write, alone: for each of n_tok rows
 * of n_heads*head_dim f32 values x (already q/k-normed where the model does
 * so), rotate-half by the f32 tables cos_t/sin_t [n_tok, head_dim/2] and
 * round to bf16 (nearest even) into out [n_tok, n_heads*head_dim].  It is the
 * same device code the fused cache write runs; every product and sum is
 * rounded separately, so identical f32 inputs give identical bits on any
 * correct f32 implementation (ember reference_forward.py rope()). */
ember_status ember_rope_store(const float *x, int32_t n_tok, int32_t n_heads, int32_t head_dim,
                              const float *cos_t, const float *sin_t, uint16_t *out,
                              ember_stream_t stream);

/* D[M,N] = A[M,K] . B[N,K]^T with bf16 A, B and f32 D (row-major, K
 * contiguous), on the tcgen05 tensor-core GEMM the projections use.  K and
 * the row strides must be multiples of 8 elements.  Errors: INVALID_ARG. */
ember_status ember_gemm_bf16(const uint16_t *A, const uint16_t *B, float *D, int32_t M,
                             int32_t N, int32_t K, ember_stream_t stream);

/* y[b][n] = sum_k W[n][k] * x[b][k] for b < nb (nb <= 8), on the split GEMV
 * the batch-1..8 decode projections run (W bf16 [N][K], x and y f32, row
 * strides K and N; K a multiple of 8, K <= 16384).  The projections of
 * ember reference_forward.py forward() (q = Wq xb, ...) without their fused
 * prologue / epilogue.  Errors: INVALID_ARG. */
ember_status ember_gemv_bf16(const uint16_t *W, int32_t N, int32_t K, const float *x, int32_t nb,
                             float *y, ember_stream_t stream);

/* q8_0 block quantization (ember internals, q8_0 block format; the encoder
 * the pages leave implicit, read as: per block of 32 values amax = max |w|,
 * codes = w / (amax / 127) in f32 rounded to the nearest integer, ties to
 * even, clamped to [-127, 127], zero for a zero block; scale = amax / 127
 * rounded to f16, nearest even) of n bf16 values w (n a positive multiple of
 * 32).  Writes the int8 codes q[n] and the f16 scales d[n/32] (bit patterns):
 * the planar form of the pages' 34-byte blocks (scale, then 32 codes), which
 * this library keeps as two arrays so that the codes stay 8-byte aligned.
 * It is the quantizer ember_model_create runs for weights_q8.  All pointers
 * are device pointers owned by the caller.  Errors: INVALID_ARG. */
ember_status ember_q8_0_quantize(const uint16_t *w, int64_t n, int8_t *q, uint16_t *d,
                                 ember_stream_t stream);

/* y[b][n] = sum_k (q[n][k] * d[n][k/32]) * x[b][k] for b < nb (nb <= 8): the
 * split GEMV of ember_gemv_bf16 reading q8_0 weights (codes q int8 [N][K],
 * f16 scales d [N][K/32] as ember_q8_0_quantize writes them), the decode
 * projections of a weights_q8 model.  K a multiple of 32, K <= 16384; q
 * 8-byte and x 16-byte aligned.  Errors: INVALID_ARG. */
ember_status ember_gemv_q8_0(const int8_t *q, const uint16_t *d, int32_t N, int32_t K,
                             const float *x, int32_t nb, float *y, ember_stream_t stream);

/* ---- greedy LM head with no allocation ----------------------------------- */

/* The method this library implements has no counterpart to this entry point;
 * it serves callers that may not allocate device memory at all -- a serving
 * loop whose HBM is already handed out (to a KV pool, say), or a latency path
 * that cannot take the device-wide stall a cudaMalloc / cudaFree can cause.
 *
 * argmax[b] = the first index n of the largest y[b][n] = sum_k W[n][k] x[b][k]
 * for b < nb: the split GEMV of ember_gemv_bf16 (same arguments, same
 * arithmetic, bf16 W [N][K], f32 x [nb][K]; K a multiple of 8, K <= 16384, W
 * and x 16-byte aligned) with its argmax epilogue, the greedy step of the tied
 * LM head.  y (f32 [nb][N]) receives the logits when non-NULL.  argmax is a
 * device int32 [nb].  All pointers are the caller's; nothing is kept.
 *
 * Scratch: the per-row argmax keys sit in a fixed device array inside the
 * library (EMBER_NOALLOC_MAX_ROWS u64 keys, 64 bytes per device); no call
 * allocates, frees or calls an allocating library routine.  The keys must be
 * zero when a call starts: the set-up clears them once and each call clears
 * them again after use, in its second kernel.
 *
 * Set-up: the first call on each device (with that device current) resolves
 * the array's address and clears it on the given stream.  Make that first
 * call before any stream capture begins on the device.
 *
 * Concurrency: every call on one device shares that one array.  Two calls
 * whose kernels may overlap (different streams without an ordering between
 * them, or different host threads) race on it and may return wrong indices:
 * order them on one stream or with events.
 *
 * Errors: CAPACITY when nb > EMBER_NOALLOC_MAX_ROWS; INVALID_ARG for NULL or
 * misaligned pointers and bad sizes; UNSUPPORTED for device ordinals >= 64;
 * CUDA for a failed set-up or launch.  Returns once the two kernels are
 * queued on `stream`. */
#define EMBER_NOALLOC_MAX_ROWS 8
ember_status ember_gemv_argmax_noalloc(const uint16_t *W, int32_t N, int32_t K, const float *x,
                                       int32_t nb, float *y, int32_t *argmax,
                                       ember_stream_t stream);

/* Test-only (failure detection): runs one of the library's bounded device
 * waits -- which = 0 the shared-memory mbarrier wait of the TMA / tensor-core
 * kernels, 1 the cluster-scope wait of the fused batch-1 decode -- on an
 * mbarrier that nothing completes, with a budget of budget_cycles SM cycles
 * (<= 2e8) instead of the kernels' ~1 s.  The wait gives up and the kernel
 * raises EMBER_ERR_TIMEOUT in m's status word, which the next
 * ember_sync_status returns (and clears); nothing else is touched.  The
 * method this library implements has no counterpart to it. */
ember_status ember_test_bounded_wait(ember_model *m, int32_t which, int64_t budget_cycles,
                                     ember_stream_t stream);

/* Number of kernels this library has launched in this process so far (a
 * CUDA-graph replay counts each kernel node it runs).  For accounting. */
uint64_t ember_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* EMBER_H */
