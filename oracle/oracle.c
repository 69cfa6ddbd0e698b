/*
 * oracle.c -- plain, slow CPU oracle of the decoder forward pass.
 * TEST INFRASTRUCTURE ONLY (see oracle.h for who may load it, the arithmetic
 * reading and the page key [RF] [LL] [FH] [PII] [EI]).
 *
 * Build: gcc -O2 -ffp-contract=off [-fopenmp] -shared -fPIC oracle.c -lm
 * (-ffp-contract=off keeps every product and sum separately rounded, which
 * orc_rope_store_bf16_f32 relies on; the double paths do not care).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ECAP (-2)
#define ORC_ESTATE (-3)
#define ORC_ETOKEN (-4)

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* [RF] load_safetensors(): a bf16 weight is the high half of an f32, so the
 * decode widens the 16 bits to 32 and shifts them left by 16 (exact). */
void orc_bf16_decode(const uint16_t *in, float *out, size_t n) {
    for (size_t i = 0; i < n; ++i) {
        uint32_t u = ((uint32_t)in[i]) << 16;
        memcpy(&out[i], &u, sizeof u);
    }
}

/* Round a double to the nearest bf16 (8 significant bits, f32 exponent
 * range), ties to even; the inverse direction of orc_bf16_decode.  Used for
 * the bf16 KV cache option and the bit-exact KV check. */
uint16_t orc_bf16_round(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);             /* a in [2^(e-1), 2^e) */
    int qexp = e - 8;               /* weight of the last kept bit */
    if (qexp < -133) qexp = -133;   /* bf16 subnormal spacing 2^-133 */
    double r = rint(ldexp(a, -qexp));   /* default mode: nearest, ties even */
    double y = ldexp(r, qexp);
    if (y >= 0x1p128) return sign | 0x7F80;
    float f = (float)y;             /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* [RF] rmsnorm(), [LL] rms_norm(), [PII] rms_norm(): scale by the reciprocal
 * root-mean-square (no mean subtraction), then by the weight. */
void orc_rmsnorm(const double *x, const float *w, int n, double eps, double *y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * (double)w[i];
}

/* [RF] main(): inv_freq_i = theta^(-2i/D) for i < D/2.
 * [LL] rotary_cos_sin(): with llama3 scaling, z = (orig * f / 2pi - low) /
 * (high - low) and f is multiplied by lerp(1/factor, 1, clip(z, 0, 1)). */
void orc_rope_inv_freq(const orc_config *cfg, double *inv_freq) {
    int D = cfg->head_dim, half = D / 2;
    for (int i = 0; i < half; ++i) {
        double f = pow(cfg->rope_theta, -(2.0 * (double)i) / (double)D);
        if (cfg->rope_llama3) {
            double z = ((double)cfg->rs_orig_max_pos * f / (2.0 * M_PI) - cfg->rs_low) /
                       (cfg->rs_high - cfg->rs_low);
            if (z < 0.0) z = 0.0;
            if (z > 1.0) z = 1.0;
            double lo = 1.0 / cfg->rs_factor;
            f *= lo + z * (1.0 - lo);
        }
        inv_freq[i] = f;
    }
}

/* [RF] rope(), [PII] apply_rope(): HuggingFace rotate-half.  Element i pairs
 * with element i + D/2; the angle of pair i at position pos is pos*inv_freq_i. */
void orc_rope_apply(double *v, int head_dim, const double *inv_freq, long pos) {
    int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        double ang = (double)pos * inv_freq[i];
        double c = cos(ang), s = sin(ang);
        double x0 = v[i], x1 = v[i + half];
        v[i] = x0 * c - x1 * s;
        v[i + half] = x1 * c + x0 * s;
    }
}

void orc_rope_table_f32(const orc_config *cfg, long pos0, int npos, float *cos_t,
                        float *sin_t) {
    int half = cfg->head_dim / 2;
    double *inv = malloc(sizeof(double) * (half > 0 ? half : 1));
    orc_rope_inv_freq(cfg, inv);
    for (int p = 0; p < npos; ++p)
        for (int i = 0; i < half; ++i) {
            double ang = (double)(pos0 + p) * inv[i];
            cos_t[(size_t)p * half + i] = (float)cos(ang);
            sin_t[(size_t)p * half + i] = (float)sin(ang);
        }
    free(inv);
}

/* f32 variant of the same rotation followed by the bf16 store, evaluated the
 * way an f32 engine does it: each product rounded to f32, then the sum. */
void orc_rope_store_bf16_f32(const float *x, int n_heads, int head_dim,
                             const float *cos_t, const float *sin_t, uint16_t *out) {
    int half = head_dim / 2;
    for (int h = 0; h < n_heads; ++h) {
        const float *xh = x + (size_t)h * head_dim;
        uint16_t *oh = out + (size_t)h * head_dim;
        for (int i = 0; i < half; ++i) {
            float x0 = xh[i], x1 = xh[i + half], c = cos_t[i], s = sin_t[i];
            float p0 = x0 * c, p1 = x1 * s, p2 = x1 * c, p3 = x0 * s;
            float r0 = p0 - p1, r1 = p2 + p3;
            oh[i] = orc_bf16_round((double)r0);
            oh[i + half] = orc_bf16_round((double)r1);
        }
    }
}

/* IEEE half (f16) bits of an f32 value, nearest even, with subnormals and
 * overflow to infinity; and the exact f32 value of an f16 bit pattern. */
uint16_t orc_f16_round(float x) {
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);             /* a in [2^(e-1), 2^e) */
    int qexp = e - 11;              /* weight of the last kept bit (11 significant bits) */
    if (qexp < -24) qexp = -24;     /* f16 subnormal spacing 2^-24 */
    double r = rint(ldexp(a, -qexp));
    double y = ldexp(r, qexp);
    if (y >= 65520.0) return sign | 0x7C00;   /* rounds past 65504 */
    if (y == 0.0) return sign;
    int ye;
    double m = frexp(y, &ye);       /* y = m * 2^ye, m in [0.5, 1) */
    if (ye - 1 < -14)               /* subnormal: y = k * 2^-24 */
        return sign | (uint16_t)ldexp(y, 24);
    return sign | (uint16_t)(((ye - 1 + 15) << 10) | ((uint16_t)ldexp(m * 2.0 - 1.0, 10) & 0x3FF));
}

float orc_f16_decode(uint16_t h) {
    int s = h >> 15, ex = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (ex == 0) v = ldexp((double)m, -24);
    else if (ex == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1.0 + m / 1024.0, ex - 15);
    return (float)(s ? -v : v);
}

/* [EI] q8_0 block quantization: a block encodes 32 values in 34 bytes -- a
 * little-endian f16 scale d, then 32 signed int8 codes q; value j is q_j * d
 * (the pages' decoding loop). */
void orc_q8_0_dequant(const uint8_t *src, long n_blocks, float *dst) {
    for (long i = 0; i < n_blocks; ++i) {
        const uint8_t *b = src + i * 34;
        const float d = orc_f16_decode((uint16_t)(b[0] | (b[1] << 8)));
        for (int j = 0; j < 32; ++j) dst[i * 32 + j] = (float)(int8_t)b[2 + j] * d;
    }
}

/* The encoder, which the pages do not print (their weights arrive quantized):
 * per block, amax = max |x|, d = amax / 127 in f32, stored as f16 (nearest
 * even); q_j = x_j / d in f32 rounded to the nearest integer (ties to even),
 * clamped to [-127, 127]; a block of zeros has d = 0 and q = 0. */
void orc_q8_0_quantize(const float *x, long n, uint8_t *dst) {
    for (long i = 0; i < n / 32; ++i) {
        const float *xb = x + i * 32;
        float amax = 0.f;
        for (int j = 0; j < 32; ++j) {
            const float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        const float d = amax / 127.0f;
        const uint16_t dh = orc_f16_round(d);
        uint8_t *b = dst + i * 34;
        b[0] = (uint8_t)(dh & 0xFF);
        b[1] = (uint8_t)(dh >> 8);
        for (int j = 0; j < 32; ++j) {
            float q = d > 0.f ? rintf(xb[j] / d) : 0.f;
            if (q > 127.f) q = 127.f;
            if (q < -127.f) q = -127.f;
            b[2 + j] = (uint8_t)(int8_t)q;
        }
    }
}

/* [EI] softmax: subtract the row maximum before exponentiating; a row whose
 * maximum is -inf (every entry masked) becomes the uniform distribution. */
void orc_softmax(double *s, int n) {
    if (n <= 0) return;
    double mx = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (s[i] > mx) mx = s[i];
    if (mx == -INFINITY) {
        for (int i = 0; i < n; ++i) s[i] = 1.0 / (double)n;
        return;
    }
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
        s[i] = exp(s[i] - mx);
        sum += s[i];
    }
    for (int i = 0; i < n; ++i) s[i] /= sum;
}

/* [RF] forward(): act = gate / (1 + exp(-gate)). */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* [RF] np.argmax semantics: the first index of the maximum; a NaN counts as
 * larger than every number and the first NaN wins. */
long orc_argmax(const double *v, long n) {
    long best = 0;
    for (long i = 0; i < n; ++i) {
        if (isnan(v[i])) return i;
        if (v[i] > v[best]) best = i;
    }
    return best;
}

/* [RF] forward() per-head loop and [EI] GQA: query head h reads kv head
 * h / (NH/NKV); scores q.k_j / sqrt(D) over the n_keys visible keys, softmax,
 * then the probability-weighted sum of the value rows.
 * kc/vc: [NKV][kv_stride_head] with row j of head g at g*kv_stride_head + j*D. */
void orc_attention(const double *q, const double *kc, const double *vc, int n_heads,
                   int n_kv_heads, int head_dim, long kv_stride_head, long n_keys,
                   double *out) {
    int G = n_heads / n_kv_heads;
    double scale = 1.0 / sqrt((double)head_dim);
    double *sc = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    for (int h = 0; h < n_heads; ++h) {
        int g = h / G;
        const double *qh = q + (size_t)h * head_dim;
        const double *kg = kc + (size_t)g * kv_stride_head;
        const double *vg = vc + (size_t)g * kv_stride_head;
        for (long j = 0; j < n_keys; ++j) {
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d) dot += qh[d] * kg[j * head_dim + d];
            sc[j] = dot * scale;
        }
        orc_softmax(sc, (int)n_keys);
        double *oh = out + (size_t)h * head_dim;
        for (int d = 0; d < head_dim; ++d) {
            double acc = 0.0;
            for (long j = 0; j < n_keys; ++j) acc += sc[j] * vg[j * head_dim + d];
            oh[d] = acc;
        }
    }
    free(sc);
}

/* [FH] Config::validate: no zero dimension, whole GQA groups, even head_dim. */
int orc_validate(const orc_config *c) {
    if (c->vocab <= 0 || c->hidden <= 0 || c->layers <= 0 || c->n_heads <= 0 ||
        c->n_kv_heads <= 0 || c->head_dim <= 0 || c->ff <= 0)
        return ORC_EINVAL;
    if (c->n_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0) return ORC_EINVAL;
    if (!(c->rms_eps >= 0.0) || !(c->rope_theta > 0.0)) return ORC_EINVAL;
    if (c->rope_llama3 && (!(c->rs_factor > 0.0) || !(c->rs_high != c->rs_low)))
        return ORC_EINVAL;
    return ORC_OK;
}

/* y[t][r] = sum_i W[r][i] * x[t][i] (+ b[r]) for t < T; W is [rows, in]. */
static void linear(const float *W, const float *b, const double *x, int T, int rows, int in,
                   double *y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const float *w = W + (size_t)r * in;
        for (int t = 0; t < T; ++t) {
            const double *xt = x + (size_t)t * in;
            double acc = 0.0;
            for (int i = 0; i < in; ++i) acc += (double)w[i] * xt[i];
            if (b) acc += (double)b[r];
            y[(size_t)t * rows + r] = acc;
        }
    }
}

static int check_ids(const orc_config *c, const int32_t *ids, int n) {
    for (int t = 0; t < n; ++t)
        if (ids[t] < 0 || ids[t] >= c->vocab) return ORC_ETOKEN;   /* [FH] logits() */
    return ORC_OK;
}

/* Per-layer scratch shared by both forwards. */
typedef struct {
    double *xb, *q, *k, *v, *att, *tmp, *gate, *up;
} scratch;

static int scratch_new(scratch *s, const orc_config *c, int T) {
    size_t H = c->hidden, QD = (size_t)c->n_heads * c->head_dim,
           KD = (size_t)c->n_kv_heads * c->head_dim, F = c->ff;
    s->xb = malloc(sizeof(double) * T * H);
    s->q = malloc(sizeof(double) * T * QD);
    s->k = malloc(sizeof(double) * T * KD);
    s->v = malloc(sizeof(double) * T * KD);
    s->att = malloc(sizeof(double) * T * QD);
    s->tmp = malloc(sizeof(double) * T * H);
    s->gate = malloc(sizeof(double) * T * F);
    s->up = malloc(sizeof(double) * T * F);
    return (s->xb && s->q && s->k && s->v && s->att && s->tmp && s->gate && s->up) ? 0 : -1;
}

static void scratch_free(scratch *s) {
    free(s->xb); free(s->q); free(s->k); free(s->v);
    free(s->att); free(s->tmp); free(s->gate); free(s->up);
}

/* Steps common to both forwards before attention: RMSNorm, q/k/v (+bias),
 * optional per-head q/k RMSNorm ([PII] before RoPE), RoPE at pos0 + t. */
static void qkv_rope(const orc_model *m, const orc_layer *ly, const double *x, int T, long pos0,
                     const double *inv_freq, scratch *s) {
    const orc_config *c = &m->cfg;
    int H = c->hidden, D = c->head_dim, NH = c->n_heads, NKV = c->n_kv_heads;
    for (int t = 0; t < T; ++t)
        orc_rmsnorm(x + (size_t)t * H, ly->attn_norm, H, c->rms_eps, s->xb + (size_t)t * H);
    linear(ly->wq, c->qkv_bias ? ly->bq : NULL, s->xb, T, NH * D, H, s->q);
    linear(ly->wk, c->qkv_bias ? ly->bk : NULL, s->xb, T, NKV * D, H, s->k);
    linear(ly->wv, c->qkv_bias ? ly->bv : NULL, s->xb, T, NKV * D, H, s->v);
    double *tmp = malloc(sizeof(double) * D);
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < NH; ++h) {
            double *qh = s->q + ((size_t)t * NH + h) * D;
            if (c->qk_norm) {
                orc_rmsnorm(qh, ly->q_norm, D, c->rms_eps, tmp);
                memcpy(qh, tmp, sizeof(double) * D);
            }
            orc_rope_apply(qh, D, inv_freq, pos0 + t);
        }
        for (int g = 0; g < NKV; ++g) {
            double *kh = s->k + ((size_t)t * NKV + g) * D;
            if (c->qk_norm) {
                orc_rmsnorm(kh, ly->k_norm, D, c->rms_eps, tmp);
                memcpy(kh, tmp, sizeof(double) * D);
            }
            orc_rope_apply(kh, D, inv_freq, pos0 + t);
        }
    }
    free(tmp);
}

/* Steps after attention: x += Wo att; x += Wd (silu(Wg xb) * Wu xb). */
static void oproj_mlp(const orc_model *m, const orc_layer *ly, double *x, int T, scratch *s) {
    const orc_config *c = &m->cfg;
    int H = c->hidden, QD = c->n_heads * c->head_dim, F = c->ff;
    linear(ly->wo, NULL, s->att, T, H, QD, s->tmp);
    for (size_t i = 0; i < (size_t)T * H; ++i) x[i] += s->tmp[i];
    for (int t = 0; t < T; ++t)
        orc_rmsnorm(x + (size_t)t * H, ly->mlp_norm, H, c->rms_eps, s->xb + (size_t)t * H);
    linear(ly->w_gate, NULL, s->xb, T, F, H, s->gate);
    linear(ly->w_up, NULL, s->xb, T, F, H, s->up);
    for (size_t i = 0; i < (size_t)T * F; ++i) s->gate[i] = orc_silu(s->gate[i]) * s->up[i];
    linear(ly->w_down, NULL, s->gate, T, H, F, s->tmp);
    for (size_t i = 0; i < (size_t)T * H; ++i) x[i] += s->tmp[i];
}

/* Final RMSNorm and heads ([RF] tied head embed @ x; [PII] token_cls_head).
 * Logits are written for the last logits_rows positions only. */
static void final_heads(const orc_model *m, const double *x, int T, double *hidden,
                        double *logits, int logits_rows, double *cls) {
    const orc_config *c = &m->cfg;
    int H = c->hidden, V = c->vocab;
    double *h = malloc(sizeof(double) * (size_t)T * H);
    for (int t = 0; t < T; ++t)
        orc_rmsnorm(x + (size_t)t * H, m->final_norm, H, c->rms_eps, h + (size_t)t * H);
    if (hidden) memcpy(hidden, h, sizeof(double) * (size_t)T * H);
    if (logits && logits_rows > 0) {
        int t0 = T - logits_rows;
        linear(m->embed, NULL, h + (size_t)t0 * H, logits_rows, V, H, logits);
    }
    if (cls && c->n_labels > 0) linear(m->cls_w, m->cls_b, h, T, c->n_labels, H, cls);
    free(h);
}

/* The whole-sequence forward; acts (nullable) collects the residual stream at
 * the last position after every block ([EI] forward_with_activations). */
static int forward_full(const orc_model *m, const int32_t *ids, int T, double *hidden,
                        double *logits, int logits_rows, double *cls, double *acts) {
    const orc_config *c = &m->cfg;
    if (orc_validate(c) || T <= 0) return ORC_EINVAL;
    if (check_ids(c, ids, T)) return ORC_ETOKEN;
    int H = c->hidden, D = c->head_dim, NH = c->n_heads, NKV = c->n_kv_heads;
    double *x = malloc(sizeof(double) * (size_t)T * H);
    double *inv = malloc(sizeof(double) * (D / 2));
    /* K/V of every position for the current layer, [NKV][T][D]. */
    double *K = malloc(sizeof(double) * (size_t)NKV * T * D);
    double *V = malloc(sizeof(double) * (size_t)NKV * T * D);
    scratch s;
    if (!x || !inv || !K || !V || scratch_new(&s, c, T)) return ORC_EINVAL;
    orc_rope_inv_freq(c, inv);
    for (int t = 0; t < T; ++t)             /* [RF] x = embed[tok] */
        for (int i = 0; i < H; ++i) x[(size_t)t * H + i] = m->embed[(size_t)ids[t] * H + i];
    for (int l = 0; l < c->layers; ++l) {
        const orc_layer *ly = &m->layers[l];
        qkv_rope(m, ly, x, T, 0, inv, &s);
        for (int t = 0; t < T; ++t)
            for (int g = 0; g < NKV; ++g)
                for (int d = 0; d < D; ++d) {
                    K[((size_t)g * T + t) * D + d] = s.k[((size_t)t * NKV + g) * D + d];
                    V[((size_t)g * T + t) * D + d] = s.v[((size_t)t * NKV + g) * D + d];
                }
        /* [LL] self_attn(): key s visible to query t iff s <= t (causal);
         * [PII]: every key visible (bidirectional). */
#pragma omp parallel for schedule(dynamic, 1)
        for (int t = 0; t < T; ++t) {
            long n_keys = c->causal ? (long)t + 1 : (long)T;
            orc_attention(s.q + (size_t)t * NH * D, K, V, NH, NKV, D, (long)T * D, n_keys,
                          s.att + (size_t)t * NH * D);
        }
        oproj_mlp(m, ly, x, T, &s);
        if (acts) memcpy(acts + (size_t)l * H, x + (size_t)(T - 1) * H, sizeof(double) * H);
    }
    final_heads(m, x, T, hidden, logits, logits_rows, cls);
    scratch_free(&s);
    free(x); free(inv); free(K); free(V);
    return ORC_OK;
}

int orc_forward_full(const orc_model *m, const int32_t *ids, int T, double *hidden,
                     double *logits, double *cls) {
    return forward_full(m, ids, T, hidden, logits, logits ? T : 0, cls, NULL);
}

int orc_forward_activations(const orc_model *m, const int32_t *ids, int T, double *acts,
                            double *logits) {
    if (!acts) return ORC_EINVAL;
    return forward_full(m, ids, T, NULL, logits, logits ? 1 : 0, NULL, acts);
}

/* [PII] forward(): the sensitivity head reads the mean over positions of the
 * final-normed states, sens_j = mean_t(h[t]) . w[j] + b[j]. */
void orc_mean_pooled_head(const double *hidden, int T, int H, const float *w, const float *b,
                          int n_out, double *out) {
    double *mean = calloc((size_t)H, sizeof(double));
    if (!mean) return;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < H; ++i) mean[i] += hidden[(size_t)t * H + i];
    for (int i = 0; i < H; ++i) mean[i] /= (double)T;
    for (int j = 0; j < n_out; ++j) {
        double acc = 0.0;
        for (int i = 0; i < H; ++i) acc += mean[i] * (double)w[(size_t)j * H + i];
        out[j] = acc + (b ? (double)b[j] : 0.0);
    }
    free(mean);
}

orc_cache *orc_cache_new(const orc_config *cfg, int max_len, int kv_bf16) {
    if (orc_validate(cfg) || max_len <= 0) return NULL;
    orc_cache *c = calloc(1, sizeof *c);
    if (!c) return NULL;
    c->layers = cfg->layers;
    c->n_kv_heads = cfg->n_kv_heads;
    c->head_dim = cfg->head_dim;
    c->max_len = max_len;
    c->len = 0;
    c->kv_bf16 = kv_bf16;
    size_t n = (size_t)cfg->layers * cfg->n_kv_heads * max_len * cfg->head_dim;
    c->k = calloc(n, sizeof(double));
    c->v = calloc(n, sizeof(double));
    if (!c->k || !c->v) {
        orc_cache_free(c);
        return NULL;
    }
    return c;
}

void orc_cache_free(orc_cache *c) {
    if (!c) return;
    free(c->k);
    free(c->v);
    free(c);
}

static double kv_store_value(const orc_cache *c, double x) {
    if (!c->kv_bf16) return x;
    uint16_t b = orc_bf16_round(x);
    float f;
    orc_bf16_decode(&b, &f, 1);
    return (double)f;
}

int orc_forward_cached(const orc_model *m, orc_cache *cache, const int32_t *ids, int n,
                       int start_pos, double *hidden, double *logits) {
    const orc_config *c = &m->cfg;
    if (orc_validate(c) || n <= 0 || !cache || !c->causal) return ORC_EINVAL;
    if (cache->layers != c->layers || cache->n_kv_heads != c->n_kv_heads ||
        cache->head_dim != c->head_dim)
        return ORC_EINVAL;
    if (start_pos != cache->len) return ORC_ESTATE;   /* [EI] bug #5: explicit pos */
    if ((long)start_pos + n > cache->max_len) return ORC_ECAP;
    if (check_ids(c, ids, n)) return ORC_ETOKEN;
    int H = c->hidden, D = c->head_dim, NH = c->n_heads, NKV = c->n_kv_heads;
    size_t layer_stride = (size_t)NKV * cache->max_len * D;
    double *x = malloc(sizeof(double) * (size_t)n * H);
    double *inv = malloc(sizeof(double) * (D / 2));
    scratch s;
    if (!x || !inv || scratch_new(&s, c, n)) return ORC_EINVAL;
    orc_rope_inv_freq(c, inv);
    for (int t = 0; t < n; ++t)
        for (int i = 0; i < H; ++i) x[(size_t)t * H + i] = m->embed[(size_t)ids[t] * H + i];
    for (int l = 0; l < c->layers; ++l) {
        const orc_layer *ly = &m->layers[l];
        double *Kl = cache->k + (size_t)l * layer_stride;
        double *Vl = cache->v + (size_t)l * layer_stride;
        qkv_rope(m, ly, x, n, start_pos, inv, &s);
        /* append: token t goes to position cursor + t ([EI] the fix for bug #5) */
        for (int t = 0; t < n; ++t)
            for (int g = 0; g < NKV; ++g)
                for (int d = 0; d < D; ++d) {
                    size_t dst = ((size_t)g * cache->max_len + start_pos + t) * D + d;
                    Kl[dst] = kv_store_value(cache, s.k[((size_t)t * NKV + g) * D + d]);
                    Vl[dst] = kv_store_value(cache, s.v[((size_t)t * NKV + g) * D + d]);
                }
#pragma omp parallel for schedule(dynamic, 1)
        for (int t = 0; t < n; ++t)
            orc_attention(s.q + (size_t)t * NH * D, Kl, Vl, NH, NKV, D,
                          (long)cache->max_len * D, (long)start_pos + t + 1,
                          s.att + (size_t)t * NH * D);
        oproj_mlp(m, ly, x, n, &s);
    }
    /* [EI] cursor semantics: the cursor advances once all layers have stored. */
    cache->len += n;
    final_heads(m, x, n, hidden, logits, logits ? 1 : 0, NULL);
    scratch_free(&s);
    free(x); free(inv);
    return ORC_OK;
}

int orc_greedy(const orc_model *m, orc_cache *cache, const int32_t *prompt, int n_prompt,
               int n_steps, const int32_t *forced, int32_t *tokens, double *logits,
               double *hidden) {
    const orc_config *c = &m->cfg;
    int V = c->vocab, H = c->hidden;
    if (n_steps < 0 || !tokens) return ORC_EINVAL;
    double *lg = malloc(sizeof(double) * V);
    double *hp = malloc(sizeof(double) * (size_t)n_prompt * H);
    if (!lg || !hp) return ORC_EINVAL;
    int rc = orc_forward_cached(m, cache, prompt, n_prompt, cache->len, hp, lg);
    if (rc) goto done;
    if (hidden) memcpy(hidden, hp + (size_t)(n_prompt - 1) * H, sizeof(double) * H);
    if (logits) memcpy(logits, lg, sizeof(double) * V);
    tokens[0] = (int32_t)orc_argmax(lg, V);
    for (int i = 1; i <= n_steps; ++i) {
        int32_t feed = forced ? forced[i - 1] : tokens[i - 1];
        rc = orc_forward_cached(m, cache, &feed, 1, cache->len,
                                hidden ? hidden + (size_t)i * H : NULL, lg);
        if (rc) goto done;
        if (logits) memcpy(logits + (size_t)i * V, lg, sizeof(double) * V);
        tokens[i] = (int32_t)orc_argmax(lg, V);
    }
done:
    free(lg);
    free(hp);
    return rc;
}
