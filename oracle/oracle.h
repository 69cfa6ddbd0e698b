/*
 * oracle.h -- plain, slow CPU oracle of the Llama/Qwen2-style decoder forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  It shares
 * no code, header, table or constant generator with the CUDA library: the two
 * meet only at the seeded input generator (gqa_transformer_decode_gb300/synth.py),
 * which holds none of the method's arithmetic.
 *
 * Arithmetic: every activation, dot product, norm, softmax and logit is held in
 * IEEE double.  Weights arrive as f32 (the exact decode of the bf16 bit
 * patterns, see orc_bf16_decode) and are widened to double exactly.  The pages
 * compute in f32 (NumPy / fp32 torch); double keeps the oracle's own rounding
 * error near 1e-16 so the whole tolerance budget belongs to the GPU.
 *
 * Threading: OpenMP over output rows / heads / vocabulary entries only.  Each
 * output scalar is accumulated by one thread in index order, so results are
 * bit-identical at every thread count.
 *
 * Pages followed (by page title, section / function):
 *   [RF]  ember, scripts/reference_forward.py  -- forward(), rmsnorm(), rope(),
 *         load_safetensors() bf16 decode, the greedy loop in main()
 *   [LL]  LowLlamaBasic, reference.py          -- predict(): rotary_cos_sin()
 *         with llama3 scaling, self_attn() causal einsum
 *   [FH]  Falcon-H1-0.5B-Rust, src/lib.rs      -- Config::validate, generate()
 *   [PII] PII-Tracer-vLLM, serving/reference_forward.py -- q/k per-head
 *         RMSNorm before RoPE, bidirectional attention, token_cls_head
 *   [EI]  ember internals                      -- kv cache cursor semantics,
 *         softmax fully-masked fallback, GQA head mapping
 *
 * Parity pins: see tests/test_oracle_*.py.  Every function here is pinned by at
 * least one closed form, invariant or library-routine special case there;
 * none is "parity unpinned" except the real-checkpoint goldens the pages print
 * (which need checkpoints absent here and are not reproduced).
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Model hyper-parameters ([RF] main(): config.json fields; [LL] predict();
 * [PII] forward(): head_dim is explicit). */
typedef struct {
    int vocab, hidden, layers, n_heads, n_kv_heads, head_dim, ff;
    double rope_theta, rms_eps;
    int rope_llama3;                 /* [LL] rotary_cos_sin(): llama3 scaling */
    double rs_factor, rs_low, rs_high;
    int rs_orig_max_pos;
    int qkv_bias;                    /* [RF] q/k/v biases (Qwen2)              */
    int qk_norm;                     /* [PII] per-head q/k RMSNorm             */
    int causal;                      /* 1 = causal mask, 0 = bidirectional     */
    int n_labels;                    /* 0 = tied LM head, >0 = linear head     */
} orc_config;

/* One decoder layer's weights, f32, HF [out, in] row-major. */
typedef struct {
    const float *attn_norm;                  /* [H]                     */
    const float *wq, *wk, *wv;               /* [NH*D,H] [NKV*D,H] x2   */
    const float *bq, *bk, *bv;               /* biases or NULL          */
    const float *q_norm, *k_norm;            /* [D] or NULL             */
    const float *wo;                         /* [H, NH*D]               */
    const float *mlp_norm;                   /* [H]                     */
    const float *w_gate, *w_up;              /* [F, H]                  */
    const float *w_down;                     /* [H, F]                  */
} orc_layer;

typedef struct {
    orc_config cfg;
    const float *embed;        /* [V, H]; also the tied LM head          */
    const float *final_norm;   /* [H]                                    */
    const float *cls_w;        /* [n_labels, H] or NULL                  */
    const float *cls_b;        /* [n_labels] or NULL                     */
    const orc_layer *layers;   /* [L]                                    */
} orc_model;

/* KV cache: one contiguous block per layer, [L][NKV][max_len][D] doubles,
 * with a cursor that advances once per token after all layers ([EI] kv cache,
 * cursor semantics).  kv_bf16 != 0 rounds K (after RoPE) and V to bf16
 * (round-to-nearest-even) on write. */
typedef struct {
    int layers, n_kv_heads, head_dim, max_len, len, kv_bf16;
    double *k, *v;
} orc_cache;

/* ---- primitives (exported so the tests can pin each one) ---------------- */
void   orc_bf16_decode(const uint16_t *in, float *out, size_t n);
uint16_t orc_bf16_round(double x);
void   orc_rmsnorm(const double *x, const float *w, int n, double eps, double *y);
void   orc_rope_inv_freq(const orc_config *cfg, double *inv_freq /*[D/2]*/);
void   orc_rope_apply(double *v, int head_dim, const double *inv_freq, long pos);
void   orc_softmax(double *s, int n);
double orc_silu(double g);
long   orc_argmax(const double *v, long n);
void   orc_attention(const double *q /*[NH*D]*/, const double *kc, const double *vc,
                     int n_heads, int n_kv_heads, int head_dim, long kv_stride_head,
                     long n_keys, double *out /*[NH*D]*/);
/* cos/sin of pos * inv_freq_i computed in double, rounded to f32, for
 * positions pos0 .. pos0+npos-1: the f32 table an f32 engine would use. */
void   orc_rope_table_f32(const orc_config *cfg, long pos0, int npos, float *cos_t,
                          float *sin_t /*[npos][D/2]*/);
/* f32 rotate-half + bf16 store of a cache row, for the bit-exact KV check:
 * identical f32 inputs and tables must give identical bf16 bits. */
void   orc_rope_store_bf16_f32(const float *x /*[n_heads*D]*/, int n_heads, int head_dim,
                               const float *cos_t, const float *sin_t /*[D/2] at pos*/,
                               uint16_t *out);

/* f16 (IEEE half) bits of an f32 value, nearest even; the f32 value of f16 bits. */
uint16_t orc_f16_round(float x);
float    orc_f16_decode(uint16_t h);
/* [EI] q8_0: 34-byte blocks (little-endian f16 scale d, 32 int8 codes q),
 * value q * d.  quantize: d = amax / 127 (f32) stored as f16, q = nearest
 * integer (ties even) of x / d in f32, clamped to +-127; n a multiple of 32. */
void     orc_q8_0_dequant(const uint8_t *src, long n_blocks, float *dst);
void     orc_q8_0_quantize(const float *x, long n, uint8_t *dst);

/* ---- whole forward ------------------------------------------------------ */
int  orc_validate(const orc_config *cfg);      /* 0 ok, <0 error ([FH] validate) */

/* Whole-sequence forward without a cache ([LL] predict, [PII] forward).
 * hidden: [T,H] final-normed states (nullable); logits: [T,V] (nullable,
 * tied head); cls: [T,n_labels] (nullable, linear head). */
int  orc_forward_full(const orc_model *m, const int32_t *ids, int T,
                      double *hidden, double *logits, double *cls);

/* [EI] ForwardModel forward_with_activations(): the same whole-sequence
 * forward, collecting the residual stream at the last position after every
 * decoder block, acts [L, H]; logits: [V] at the last position (nullable). */
int  orc_forward_activations(const orc_model *m, const int32_t *ids, int T, double *acts,
                             double *logits);

/* [PII] forward() sensitivity head: out[j] = mean_t(hidden[t]) . w[j] + b[j]
 * over hidden [T, H] (the final-normed states), w [n_out, H], b [n_out] or NULL. */
void orc_mean_pooled_head(const double *hidden, int T, int H, const float *w, const float *b,
                          int n_out, double *out);

orc_cache *orc_cache_new(const orc_config *cfg, int max_len, int kv_bf16);
void       orc_cache_free(orc_cache *c);

/* Cached forward of n new tokens at positions start_pos..start_pos+n-1
 * ([RF] forward(tok,pos) with the KV append; [EI] explicit pos = cursor +
 * token index).  Returns -3 if start_pos != cache->len, -2 on capacity. */
int  orc_forward_cached(const orc_model *m, orc_cache *c, const int32_t *ids, int n,
                        int start_pos, double *hidden, double *logits);

/* [RF] greedy loop: prefill the prompt, tokens[0] = argmax of the last prompt
 * position, then n_steps cached forwards each fed the previous token.
 * tokens: [n_steps+1]; logits: [(n_steps+1), V] nullable; hidden likewise.
 * forced: if non-NULL, the token fed at step i is forced[i-1] instead of the
 * argmax (teacher forcing), tokens[] still records the argmax. */
int  orc_greedy(const orc_model *m, orc_cache *c, const int32_t *prompt, int n_prompt,
                int n_steps, const int32_t *forced, int32_t *tokens, double *logits,
                double *hidden);

int  orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
