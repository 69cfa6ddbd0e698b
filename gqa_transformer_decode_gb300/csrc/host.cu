// host.cu -- the C ABI of include/ember.h: configuration checks, weight
// repack into the device layout, workspace and KV-cache ownership, and the
// launch sequences of prefill, decode and encode.
//
// Shape of the interface: ember internals, "ForwardModel trait"
// (create_cache(max_seq_len); forward_with_cache(ids, cache, start_pos)) and
// "kv cache" (one block per layer, cursor advanced after all layers, explicit
// positions); argument errors after Falcon-H1-0.5B-Rust Config::validate,
// logits() and generate().
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"

using namespace ember;

namespace {

thread_local std::string g_err;

ember_status fail(ember_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

#define CK(call)                                                                          \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess)                                                            \
            return fail(EMBER_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                              \
    } while (0)

constexpr int MAX_DECODE_BATCH = 64;   // tokens of one decode step
constexpr int GEMV_MAX_BATCH = 8;      // above this the step runs on the GEMM path
constexpr int MAX_SPLITS = 32;         // split-KV partials per (token, kv head)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over one cudaMalloc'd block, 256-byte aligned pieces.
struct Arena {
    size_t off = 0;
    std::vector<std::pair<void**, size_t>> items;
    template <class T>
    void add(T** p, size_t count) {
        items.push_back({reinterpret_cast<void**>(p), count * sizeof(T)});
    }
    cudaError_t commit(void** base) {
        size_t total = 0;
        for (auto& it : items) total = align_up(total, 256) + it.second;
        total = align_up(total, 256);
        cudaError_t e = cudaMalloc(base, total ? total : 256);
        if (e != cudaSuccess) return e;
        size_t o = 0;
        for (auto& it : items) {
            o = align_up(o, 256);
            *it.first = static_cast<char*>(*base) + o;
            o += it.second;
        }
        return cudaSuccess;
    }
};

// RoPE tables: inv_freq_i = theta^(-2i/D) in double, llama3 scaling per
// LowLlamaBasic rotary_cos_sin(), then cos/sin of pos*inv_freq_i rounded to f32.
void rope_tables(const ember_config& c, int npos, std::vector<float>& cs, std::vector<float>& sn) {
    const int half = c.head_dim / 2;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) {
        double f = std::pow(c.rope_theta, -(2.0 * i) / (double)c.head_dim);
        if (c.rope_llama3) {
            const double pi = 3.14159265358979323846;
            double z = ((double)c.rs_orig_max_pos * f / (2.0 * pi) - c.rs_low) / (c.rs_high - c.rs_low);
            z = z < 0.0 ? 0.0 : (z > 1.0 ? 1.0 : z);
            const double lo = 1.0 / c.rs_factor;
            f *= lo + z * (1.0 - lo);
        }
        inv[i] = f;
    }
    cs.resize((size_t)npos * half);
    sn.resize((size_t)npos * half);
    for (int p = 0; p < npos; ++p)
        for (int i = 0; i < half; ++i) {
            const double a = (double)p * inv[i];
            cs[(size_t)p * half + i] = (float)std::cos(a);
            sn[(size_t)p * half + i] = (float)std::sin(a);
        }
}

struct LayerDev {
    uint16_t *wqkv, *wo, *wgu, *wd;
    uint16_t* wdT = nullptr;   // f16 [F][H] down_proj transposed (fused batch-1 decode)
    uint16_t* woG = nullptr;   // f16 [NKV][H][G*D] o_proj grouped by kv head (fused decode)
    float *attn_norm, *mlp_norm, *bqkv, *q_norm, *k_norm;
    GemmPlan p_qkv, p_o, p_gu, p_d;
    // storage scales 2^-e of wqkv, wo, wgu, wd: e > 0 only for a matrix whose
    // bf16 values exceed the f16 range (its products are multiplied by 2^e)
    int e_qkv = 0, e_o = 0, e_gu = 0, e_d = 0;
    // q8_0 copies (weights_q8): codes [N][K] and f16 scales [N][K/32] of the
    // same four matrices, read by the decode GEMVs
    int8_t *q_qkv = nullptr, *q_o = nullptr, *q_gu = nullptr, *q_d = nullptr;
    uint16_t *d_qkv = nullptr, *d_o = nullptr, *d_gu = nullptr, *d_d = nullptr;
};

struct GraphEntry {
    unsigned long long kv_gen;   // the KV cache the graph was captured against
    int batch;
    const void *seqs, *ids, *pos, *logits, *argmax;
    cudaGraphExec_t exec;
    long long kernels;   // kernel nodes, counted once per replay
};

std::atomic<long long> g_launches{0};
std::atomic<unsigned long long> g_kv_gen{0};   // a unique id per KV cache ever allocated

}  // namespace

namespace ember {
// Launch trace of ember_decode_step_traced: an event before every kernel
// launch of the calling thread (and one after the last), with the kernel.
struct LaunchTrace {
    std::vector<cudaEvent_t> ev;
    std::vector<const void*> fn;
    cudaError_t err = cudaSuccess;
};
thread_local LaunchTrace* g_trace = nullptr;
void trace_launch(const void* fn, cudaStream_t s) {
    if (!g_trace) return;
    cudaEvent_t e = nullptr;
    cudaError_t r = cudaEventCreate(&e);
    // External: under stream capture the record becomes an event node of the graph
    if (r == cudaSuccess) r = cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
    if (r != cudaSuccess) {
        if (g_trace->err == cudaSuccess) g_trace->err = r;
        if (e) cudaEventDestroy(e);
        return;
    }
    g_trace->ev.push_back(e);
    g_trace->fn.push_back(fn);
}
bool pdl_enabled() {
    static const bool on = !(getenv("EMBER_NO_PDL") && atoi(getenv("EMBER_NO_PDL")));
    return on && !g_trace;   // traced launches run one after another
}
void count_launches(long long n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
unsigned long long launches_so_far() { return (unsigned long long)g_launches.load(); }
}  // namespace ember

struct ember_model {
    ember_config c;
    int q, kv, qkv_n, G, T, sms;
    void* wblock = nullptr;
    void* ablock = nullptr;
    uint16_t* embed = nullptr;
    uint16_t* cls_w = nullptr;
    float *final_norm = nullptr, *cls_b = nullptr;
    std::vector<LayerDev> layers;
    // workspace
    float *x, *qkv, *att_f, *act_f, *hbuf, *part;
    uint16_t *xb, *qr, *att_b, *act_b, *enc_k, *enc_v, *hb;
    unsigned* counters;
    unsigned long long* keys;
    int *tok_ok, *status;
    int32_t* tok_pos;
    float *enc_cos = nullptr, *enc_sin = nullptr;
    uint16_t* enc_vt = nullptr;          // transposed V of the encoder batch
    uint16_t* enc_kh = nullptr;          // f16 K of the encoder batch
    alignas(64) unsigned char q_map[128];   // TMA map over the RoPE'd bf16 queries
    bool q_map_ok = false;
    int enc_positions = 0;
    GemmPlan p_head;   // tied head on bf16 final states (encode without labels)
    // TMA maps over the many-row GEMM outputs: q/k/v (f32), the residual
    // stream (f32, reduce-add) and the SwiGLU output (f16)
    alignas(64) unsigned char omap_qkv[128];
    alignas(64) unsigned char omap_x[128];
    alignas(64) unsigned char omap_act[128];
    // fused batch-1 decode (two kernels per layer)
    FusedPlan fp;
    float* fx[2] = {nullptr, nullptr};             // residual stream copies [H]
    float* fz[3] = {nullptr, nullptr, nullptr};    // split-K accumulators [H]
    std::vector<GraphEntry> graphs;
    std::vector<ember_kv*> kvs;   // live caches (detached when the model goes first)
    bool use_graphs = true;
    std::mutex mu;
};

struct ember_kv {
    ember_model* m;
    int max_seqs, max_len;
    uint16_t *k = nullptr, *v = nullptr;
    int32_t* cursor = nullptr;
    float *cos_t = nullptr, *sin_t = nullptr;
    uint16_t* vt = nullptr;              // transposed V of one layer's kv heads (prefill)
    uint16_t* kh = nullptr;              // f16 K of one layer's kv heads (prefill)
    alignas(64) unsigned char k_map[128];   // TMA map over the whole K cache, 3-D
    bool k_map_ok = false;
    alignas(64) unsigned char v_map[128];   // the same over the V cache
    bool v_map_ok = false;
    unsigned long long gen = 0;             // never reused, unlike the host address
};

static ember_status validate(const ember_config* c) {
    if (!c) return fail(EMBER_ERR_INVALID_ARG, "config is NULL");
    if (c->vocab <= 0 || c->hidden <= 0 || c->layers <= 0 || c->n_heads <= 0 ||
        c->n_kv_heads <= 0 || c->head_dim <= 0 || c->ff <= 0)
        return fail(EMBER_ERR_INVALID_ARG, "zero dimension");
    if (c->n_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0)
        return fail(EMBER_ERR_INVALID_ARG, "invalid GQA/RoPE shape: heads %% kv_heads or odd head_dim");
    if (c->head_dim != 16 && c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
        return fail(EMBER_ERR_UNSUPPORTED, "head_dim must be 16, 32, 64 or 128");
    if (c->n_heads / c->n_kv_heads > 16) return fail(EMBER_ERR_UNSUPPORTED, "GQA group > 16");
    if (c->hidden % 8 || c->ff % 8) return fail(EMBER_ERR_UNSUPPORTED, "hidden and ff must be multiples of 8");
    if (c->hidden > 8192 || c->ff > 16384 || c->n_heads * c->head_dim > 16384)
        return fail(EMBER_ERR_UNSUPPORTED, "hidden > 8192, ff > 16384 or heads*head_dim > 16384");
    if (!(c->rope_theta > 0.0) || !(c->rms_eps >= 0.0))
        return fail(EMBER_ERR_INVALID_ARG, "rope_theta must be > 0 and rms_eps >= 0");
    if (c->rope_llama3 && (!(c->rs_factor > 0.0) || c->rs_high == c->rs_low || c->rs_orig_max_pos <= 0))
        return fail(EMBER_ERR_INVALID_ARG, "invalid llama3 rope scaling");
    if (c->n_labels < 0 || c->max_tokens < 0 || c->max_positions < 0)
        return fail(EMBER_ERR_INVALID_ARG, "negative n_labels / max_tokens / max_positions");
    if (c->weights_q8 != 0 && c->weights_q8 != 1) return fail(EMBER_ERR_INVALID_ARG, "weights_q8 must be 0 or 1");
    if (c->weights_q8 && (c->hidden % 32 || c->ff % 32 || (c->n_heads * c->head_dim) % 32))
        return fail(EMBER_ERR_UNSUPPORTED, "weights_q8 needs hidden, ff and n_heads*head_dim to be multiples of 32");
    return EMBER_OK;
}

extern "C" {

const char* ember_last_error(void) { return g_err.c_str(); }

size_t ember_kv_bytes(const ember_config* c, int32_t max_seqs, int32_t max_len) {
    if (!c || max_seqs <= 0 || max_len <= 0) return 0;
    return (size_t)c->layers * 2 * c->n_kv_heads * (size_t)max_len * c->head_dim * 2 *
           (size_t)max_seqs;
}

ember_status ember_model_create(const ember_config* cfg, const ember_weights* w, ember_model** out) {
    if (!out) return fail(EMBER_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    ember_status st = validate(cfg);
    if (st != EMBER_OK) return st;
    if (!w || !w->embed || !w->final_norm || !w->layers)
        return fail(EMBER_ERR_INVALID_ARG, "missing weight: embed, final_norm or layers");
    const ember_config& c = *cfg;
    if (c.n_labels > 0 && !w->cls_w) return fail(EMBER_ERR_INVALID_ARG, "missing weight: cls_w");
    for (int l = 0; l < c.layers; ++l) {
        const ember_layer_weights& L = w->layers[l];
        if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.mlp_norm || !L.w_gate ||
            !L.w_up || !L.w_down)
            return fail(EMBER_ERR_INVALID_ARG, "missing weight in layer %d", l);
        if (c.qkv_bias && (!L.bq || !L.bk || !L.bv))
            return fail(EMBER_ERR_INVALID_ARG, "missing q/k/v bias in layer %d", l);
        if (c.qk_norm && (!L.q_norm || !L.k_norm))
            return fail(EMBER_ERR_INVALID_ARG, "missing q/k norm in layer %d", l);
    }

    ember_model* m = new ember_model();
    m->c = c;
    if (m->c.max_tokens == 0) m->c.max_tokens = 4096;
    if (m->c.max_positions == 0) m->c.max_positions = m->c.max_tokens;
    const int H = c.hidden, D = c.head_dim, F = c.ff, V = c.vocab, NKV = c.n_kv_heads;
    m->q = c.n_heads * D;
    m->kv = NKV * D;
    m->qkv_n = m->q + 2 * m->kv;
    m->G = c.n_heads / NKV;
    m->T = m->c.max_tokens;
    m->use_graphs = !(getenv("EMBER_NO_GRAPH") && atoi(getenv("EMBER_NO_GRAPH")));
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&m->sms, cudaDevAttrMultiProcessorCount, dev);
    m->layers.resize(c.layers);
    // the fused batch-1 kernels stream f16 weights only: q8_0 models decode
    // batch 1 through the q8_0 GEMVs
    if (c.causal && !c.weights_q8 && !(getenv("EMBER_NO_FUSED") && atoi(getenv("EMBER_NO_FUSED"))))
        fused_decode_plan(m->fp, H, c.n_heads, NKV, D, F, m->sms);
    if (getenv("EMBER_VERBOSE") && atoi(getenv("EMBER_VERBOSE")))
        fprintf(stderr, "ember: fused batch-1 decode %s%s (%s, clusters of %d, attention smem %d, MLP grid %d smem %d fc %d ns %d)\n",
                m->fp.ok ? "on" : "off: ", m->fp.ok ? "" : m->fp.why,
                m->fp.part ? "partitioned" : (m->fp.resident ? "resident MLP" : "MLP ring"), m->fp.C, m->fp.smem_attn,
                m->fp.mlp_grid, m->fp.smem_mlp, m->fp.fc, m->fp.ns);

    // ---- weights ----
    Arena wa;
    wa.add(&m->embed, (size_t)V * H);
    wa.add(&m->final_norm, H);
    if (c.n_labels > 0) {
        wa.add(&m->cls_w, (size_t)c.n_labels * H);
        wa.add(&m->cls_b, c.n_labels);
    }
    for (auto& L : m->layers) {
        wa.add(&L.wqkv, (size_t)m->qkv_n * H);
        wa.add(&L.wo, (size_t)H * m->q);
        wa.add(&L.wgu, (size_t)2 * F * H);
        wa.add(&L.wd, (size_t)H * F);
        if (m->fp.ok) {
            wa.add(&L.wdT, (size_t)F * H);
            wa.add(&L.woG, (size_t)H * m->q);
        }
        if (c.weights_q8) {
            wa.add(&L.q_qkv, (size_t)m->qkv_n * H);
            wa.add(&L.q_o, (size_t)H * m->q);
            wa.add(&L.q_gu, (size_t)2 * F * H);
            wa.add(&L.q_d, (size_t)H * F);
            wa.add(&L.d_qkv, (size_t)m->qkv_n * H / 32);
            wa.add(&L.d_o, (size_t)H * m->q / 32);
            wa.add(&L.d_gu, (size_t)2 * F * H / 32);
            wa.add(&L.d_d, (size_t)H * F / 32);
        }
        wa.add(&L.attn_norm, H);
        wa.add(&L.mlp_norm, H);
        wa.add(&L.bqkv, m->qkv_n);
        wa.add(&L.q_norm, D);
        wa.add(&L.k_norm, D);
    }
    // ---- workspace ----
    const int T = m->T, B = MAX_DECODE_BATCH;
    Arena aa;
    aa.add(&m->x, (size_t)T * H);
    aa.add(&m->xb, (size_t)T * H);
    aa.add(&m->qkv, (size_t)T * m->qkv_n);
    aa.add(&m->qr, (size_t)T * m->q);
    aa.add(&m->att_b, (size_t)T * m->q);
    aa.add(&m->act_b, (size_t)T * F);
    aa.add(&m->hbuf, (size_t)T * H);
    aa.add(&m->hb, (size_t)T * H);
    aa.add(&m->att_f, (size_t)B * m->q);
    aa.add(&m->act_f, (size_t)GEMV_MAX_BATCH * F);
    aa.add(&m->part, (size_t)B * NKV * MAX_SPLITS * m->G * (D + 2));
    aa.add(&m->counters, (size_t)B * NKV);
    aa.add(&m->keys, (size_t)B);
    aa.add(&m->tok_ok, (size_t)B);
    aa.add(&m->tok_pos, (size_t)B);
    aa.add(&m->status, 1);
    if (m->fp.ok) {
        for (auto& p : m->fx) aa.add(&p, (size_t)H);
        for (auto& p : m->fz) aa.add(&p, (size_t)H * ZSLOTS);
    }
    if (!c.causal) {
        aa.add(&m->enc_k, (size_t)T * m->kv);
        aa.add(&m->enc_v, (size_t)T * m->kv);
        aa.add(&m->enc_vt, (size_t)8 * T * m->kv);   // B * round8(T) <= 8 * B * T keys
        aa.add(&m->enc_kh, (size_t)8 * T * m->kv);
        aa.add(&m->enc_cos, (size_t)m->c.max_positions * (D / 2));
        aa.add(&m->enc_sin, (size_t)m->c.max_positions * (D / 2));
    }

    auto cleanup = [&](ember_status s) {
        if (m->wblock) cudaFree(m->wblock);
        if (m->ablock) cudaFree(m->ablock);
        delete m;
        return s;
    };
    if (wa.commit(&m->wblock) != cudaSuccess) {
        cudaGetLastError();
        return cleanup(fail(EMBER_ERR_OOM, "weight allocation failed"));
    }
    if (aa.commit(&m->ablock) != cudaSuccess) {
        cudaGetLastError();
        return cleanup(fail(EMBER_ERR_OOM, "workspace allocation failed"));
    }

    cudaStream_t s = nullptr;
    const auto D2D = cudaMemcpyDeviceToDevice;
    cudaError_t e = cudaSuccess;
    auto cp = [&](void* dst, const void* src, size_t bytes) {
        if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, D2D, s);
    };
    cp(m->embed, w->embed, (size_t)V * H * 2);
    launch_bf16_to_f32(w->final_norm, m->final_norm, H, s);
    if (c.n_labels > 0) {
        cp(m->cls_w, w->cls_w, (size_t)c.n_labels * H * 2);
        if (w->cls_b) launch_bf16_to_f32(w->cls_b, m->cls_b, c.n_labels, s);
        else if (e == cudaSuccess) e = cudaMemsetAsync(m->cls_b, 0, c.n_labels * 4, s);
    }
    for (int l = 0; l < c.layers; ++l) {
        const ember_layer_weights& W = w->layers[l];
        LayerDev& L = m->layers[l];
        // fused [q; k; v] rows
        cp(L.wqkv, W.wq, (size_t)m->q * H * 2);
        cp(L.wqkv + (size_t)m->q * H, W.wk, (size_t)m->kv * H * 2);
        cp(L.wqkv + (size_t)(m->q + m->kv) * H, W.wv, (size_t)m->kv * H * 2);
        cp(L.wo, W.wo, (size_t)H * m->q * 2);
        // gate / up interleaved by row: row 2i = gate_i, row 2i+1 = up_i
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(L.wgu, (size_t)4 * H, W.w_gate, (size_t)2 * H, (size_t)2 * H, F,
                                  D2D, s);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(L.wgu + H, (size_t)4 * H, W.w_up, (size_t)2 * H, (size_t)2 * H, F,
                                  D2D, s);
        cp(L.wd, W.w_down, (size_t)H * F * 2);
    }
    // The layer matrices run as f16 (more mantissa for the f16 activations
    // they meet in the tensor-core GEMMs); embedding / head stay bf16.  A
    // matrix whose largest |w| exceeds the f16 range (65504) is stored as
    // f16(W * 2^-e), the smallest such e, and every product with it is
    // multiplied by 2^e: the rescaling is exact, so a bf16 checkpoint with
    // large weights keeps its values.
    unsigned* d_max = nullptr;
    std::vector<unsigned> h_max((size_t)4 * c.layers, 0u);
    if (e == cudaSuccess) e = cudaMalloc(&d_max, h_max.size() * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemsetAsync(d_max, 0, h_max.size() * sizeof(unsigned), s);
    for (int l = 0; l < c.layers && e == cudaSuccess; ++l) {
        LayerDev& L = m->layers[l];
        launch_absmax_bf16(L.wqkv, (long long)m->qkv_n * H, d_max + 4 * l + 0, s);
        launch_absmax_bf16(L.wo, (long long)H * m->q, d_max + 4 * l + 1, s);
        launch_absmax_bf16(L.wgu, (long long)2 * F * H, d_max + 4 * l + 2, s);
        launch_absmax_bf16(L.wd, (long long)H * F, d_max + 4 * l + 3, s);
    }
    if (e == cudaSuccess) e = cudaMemcpy(h_max.data(), d_max, h_max.size() * sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (d_max) cudaFree(d_max);
    // q8_0: the decoded values reach 127 * f16(amax / 127) <= amax * (1 + 2^-11)
    const float grow = c.weights_q8 ? 1.f + 1.f / 1024.f : 1.f;
    if (c.weights_q8) {
        for (unsigned bits : h_max) {
            float v;
            std::memcpy(&v, &bits, 4);
            if (!(v / 127.f <= 65504.f))
                return cleanup(fail(EMBER_ERR_UNSUPPORTED,
                                    "weights_q8: a layer weight of magnitude %g has a q8_0 scale beyond f16", v));
        }
    }
    auto exp_for = [grow](unsigned bits) {
        float v;
        std::memcpy(&v, &bits, 4);
        v *= grow;
        int ex = 0;
        while (v > 65504.f && ex < 126) {
            v *= 0.5f;
            ++ex;
        }
        return ex;
    };
    for (int l = 0; l < c.layers; ++l) {
        const ember_layer_weights& W = w->layers[l];
        LayerDev& L = m->layers[l];
        L.e_qkv = exp_for(h_max[4 * l + 0]);
        L.e_o = exp_for(h_max[4 * l + 1]);
        L.e_gu = exp_for(h_max[4 * l + 2]);
        L.e_d = exp_for(h_max[4 * l + 3]);
        if (e == cudaSuccess && c.weights_q8) {   // codes + scales, and f16 of the decoded values
            launch_q8_0_quantize(L.wqkv, (long long)m->qkv_n * H, L.q_qkv, L.d_qkv, L.wqkv, L.e_qkv, s);
            launch_q8_0_quantize(L.wo, (long long)H * m->q, L.q_o, L.d_o, L.wo, L.e_o, s);
            launch_q8_0_quantize(L.wgu, (long long)2 * F * H, L.q_gu, L.d_gu, L.wgu, L.e_gu, s);
            launch_q8_0_quantize(L.wd, (long long)H * F, L.q_d, L.d_d, L.wd, L.e_d, s);
        } else if (e == cudaSuccess) {
            launch_bf16_to_f16_inplace(L.wqkv, (long long)m->qkv_n * H, L.e_qkv, s);
            launch_bf16_to_f16_inplace(L.wo, (long long)H * m->q, L.e_o, s);
            launch_bf16_to_f16_inplace(L.wgu, (long long)2 * F * H, L.e_gu, s);
            launch_bf16_to_f16_inplace(L.wd, (long long)H * F, L.e_d, s);
        }
        if (e == cudaSuccess) {
            if (L.wdT) launch_transpose16(L.wd, L.wdT, H, F, s);
            if (L.woG) {   // group g's o_proj columns as one [H][G*D] block
                const size_t gd = (size_t)m->G * D;
                for (int g = 0; g < NKV && e == cudaSuccess; ++g)
                    e = cudaMemcpy2DAsync(L.woG + (size_t)g * H * gd, gd * 2, L.wo + (size_t)g * gd,
                                          (size_t)m->q * 2, gd * 2, H, D2D, s);
            }
        }
        launch_bf16_to_f32(W.attn_norm, L.attn_norm, H, s);
        launch_bf16_to_f32(W.mlp_norm, L.mlp_norm, H, s);
        if (c.qkv_bias) {
            launch_bf16_to_f32(W.bq, L.bqkv, m->q, s);
            launch_bf16_to_f32(W.bk, L.bqkv + m->q, m->kv, s);
            launch_bf16_to_f32(W.bv, L.bqkv + m->q + m->kv, m->kv, s);
        } else if (e == cudaSuccess) {
            e = cudaMemsetAsync(L.bqkv, 0, (size_t)m->qkv_n * 4, s);
        }
        if (c.qk_norm) {
            launch_bf16_to_f32(W.q_norm, L.q_norm, D, s);
            launch_bf16_to_f32(W.k_norm, L.k_norm, D, s);
        }
        // tensor-core plans of the whole-prompt projections
        bool ok = make_gemm_plan(L.p_qkv, m->xb, T, H, L.wqkv, m->qkv_n, H, H, true) &&
                  make_gemm_plan(L.p_o, m->att_b, T, m->q, L.wo, H, m->q, m->q, true) &&
                  make_gemm_plan(L.p_gu, m->xb, T, H, L.wgu, 2 * F, H, H, true) &&
                  make_gemm_plan(L.p_d, m->act_b, T, F, L.wd, H, F, F, true);
        if (!ok) return cleanup(fail(EMBER_ERR_CUDA, "TMA tensor map encoding failed (layer %d)", l));
    }
    if (!make_gemm_plan(m->p_head, m->hb, T, H, m->embed, V, H, H, false))
        return cleanup(fail(EMBER_ERR_CUDA, "TMA tensor map encoding failed (head)"));
    if (!make_out_map(m->omap_qkv, m->qkv, T, m->qkv_n, m->qkv_n, false) ||
        !make_out_map(m->omap_x, m->x, T, H, H, false) || !make_out_map(m->omap_act, m->act_b, T, F, F, true))
        return cleanup(fail(EMBER_ERR_CUDA, "TMA tensor map encoding failed (GEMM outputs)"));
    if (attn_tc_supported(D)) {
        const uint64_t qd[2] = {(uint64_t)m->q, (uint64_t)T};
        const uint64_t qs[1] = {(uint64_t)m->q * 2};
        const uint32_t qb[2] = {64, 128};
        m->q_map_ok = encode_map_bf16(m->q_map, m->qr, 2, qd, qs, qb);
        if (!m->q_map_ok) return cleanup(fail(EMBER_ERR_CUDA, "TMA tensor map encoding failed (q)"));
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(m->counters, 0, (size_t)B * NKV * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->keys, 0, (size_t)B * 8, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->status, 0, 4, s);
    if (e == cudaSuccess && !c.causal) {
        std::vector<float> cs, sn;
        rope_tables(m->c, m->c.max_positions, cs, sn);
        e = cudaMemcpy(m->enc_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
        if (e == cudaSuccess)
            e = cudaMemcpy(m->enc_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cleanup(fail(EMBER_ERR_CUDA, "weight repack failed: %s", cudaGetErrorString(e)));
    *out = m;
    return EMBER_OK;
}

void ember_model_destroy(ember_model* m) {
    if (!m) return;
    cudaDeviceSynchronize();
    for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
    for (ember_kv* kv : m->kvs) kv->m = nullptr;
    if (m->wblock) cudaFree(m->wblock);
    if (m->ablock) cudaFree(m->ablock);
    delete m;
}

ember_status ember_kv_alloc(ember_model* m, int32_t max_seqs, int32_t max_len, ember_kv** out) {
    if (!m || !out) return fail(EMBER_ERR_INVALID_ARG, "model or out is NULL");
    *out = nullptr;
    if (max_seqs <= 0 || max_len <= 0) return fail(EMBER_ERR_INVALID_ARG, "max_seqs and max_len must be > 0");
    if (!m->c.causal) return fail(EMBER_ERR_INVALID_ARG, "a bidirectional encoder has no KV cache");
    const size_t half = ember_kv_bytes(&m->c, max_seqs, max_len) / 2;
    ember_kv* kv = new ember_kv();
    kv->gen = ++g_kv_gen;
    kv->m = m;
    kv->max_seqs = max_seqs;
    kv->max_len = max_len;
    const int h2 = m->c.head_dim / 2;
    cudaError_t e = cudaMalloc(&kv->k, half);
    if (e == cudaSuccess) e = cudaMalloc(&kv->v, half);
    if (e == cudaSuccess) e = cudaMalloc(&kv->cursor, (size_t)max_seqs * 4);
    if (e == cudaSuccess) e = cudaMalloc(&kv->cos_t, (size_t)max_len * h2 * 4);
    if (e == cudaSuccess) e = cudaMalloc(&kv->sin_t, (size_t)max_len * h2 * 4);
    const int keys_cap = (max_len + 7) / 8 * 8;
    if (e == cudaSuccess && attn_tc_supported(m->c.head_dim))
        e = cudaMalloc(&kv->vt, (size_t)m->c.n_kv_heads * m->c.head_dim * keys_cap * 2);
    if (e == cudaSuccess && attn_tc_supported(m->c.head_dim))
        e = cudaMalloc(&kv->kh, (size_t)m->c.n_kv_heads * m->c.head_dim * keys_cap * 2);
    if (e != cudaSuccess) {
        cudaGetLastError();
        ember_kv_free(kv);
        return fail(EMBER_ERR_OOM, "KV cache allocation of %zu bytes failed", 2 * half);
    }
    std::vector<float> cs, sn;
    rope_tables(m->c, max_len, cs, sn);
    e = cudaMemset(kv->k, 0, half);
    if (e == cudaSuccess) e = cudaMemset(kv->v, 0, half);
    if (e == cudaSuccess) e = cudaMemset(kv->cursor, 0, (size_t)max_seqs * 4);
    if (e == cudaSuccess) e = cudaMemcpy(kv->cos_t, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(kv->sin_t, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        ember_kv_free(kv);
        return fail(EMBER_ERR_CUDA, "KV cache init failed: %s", cudaGetErrorString(e));
    }
    if (attn_tc_supported(m->c.head_dim)) {
        // K cache [seq][layer][kv head][pos][D] as one 3-D tensor: (D, pos, seq*layer*head)
        const ember_config& c = m->c;
        const uint64_t kd[3] = {(uint64_t)c.head_dim, (uint64_t)max_len,
                                (uint64_t)max_seqs * c.layers * c.n_kv_heads};
        const uint64_t ks[2] = {(uint64_t)c.head_dim * 2, (uint64_t)max_len * c.head_dim * 2};
        const uint32_t kb[3] = {64, 128, 1};
        kv->k_map_ok = encode_map_bf16(kv->k_map, kv->k, 3, kd, ks, kb);
        kv->v_map_ok = encode_map_bf16(kv->v_map, kv->v, 3, kd, ks, kb);
        if (!kv->k_map_ok || !kv->v_map_ok) {
            ember_kv_free(kv);
            return fail(EMBER_ERR_CUDA, "TMA tensor map encoding failed (KV cache)");
        }
    }
    {
        std::lock_guard<std::mutex> lk(m->mu);
        m->kvs.push_back(kv);
    }
    *out = kv;
    return EMBER_OK;
}

void ember_kv_free(ember_kv* kv) {
    if (!kv) return;
    cudaDeviceSynchronize();
    if (kv->m) {   // decode graphs captured against this cache point at its memory
        std::lock_guard<std::mutex> lk(kv->m->mu);
        auto& ks = kv->m->kvs;
        for (auto it = ks.begin(); it != ks.end(); ++it)
            if (*it == kv) {
                ks.erase(it);
                break;
            }
        auto& gs = kv->m->graphs;
        for (auto it = gs.begin(); it != gs.end();) {
            if (it->kv_gen == kv->gen) {
                cudaGraphExecDestroy(it->exec);
                it = gs.erase(it);
            } else {
                ++it;
            }
        }
    }
    cudaFree(kv->k);
    cudaFree(kv->v);
    cudaFree(kv->cursor);
    cudaFree(kv->cos_t);
    cudaFree(kv->sin_t);
    cudaFree(kv->vt);
    cudaFree(kv->kh);
    delete kv;
}

ember_status ember_kv_reset(ember_kv* kv, int32_t seq, ember_stream_t stream) {
    if (!kv) return fail(EMBER_ERR_INVALID_ARG, "kv is NULL");
    if (seq < 0 || seq >= kv->max_seqs) return fail(EMBER_ERR_INVALID_ARG, "seq %d out of range", seq);
    CK(cudaMemsetAsync(kv->cursor + seq, 0, 4, (cudaStream_t)stream));
    return EMBER_OK;
}

ember_status ember_kv_set_cursor(ember_kv* kv, int32_t seq, int32_t pos, ember_stream_t stream) {
    if (!kv) return fail(EMBER_ERR_INVALID_ARG, "kv is NULL");
    if (seq < 0 || seq >= kv->max_seqs) return fail(EMBER_ERR_INVALID_ARG, "seq %d out of range", seq);
    if (pos < 0 || pos > kv->max_len) return fail(EMBER_ERR_CAPACITY, "pos %d outside [0, %d]", pos, kv->max_len);
    launch_set_cursor(kv->cursor, seq, pos, (cudaStream_t)stream);
    CK(cudaGetLastError());
    return EMBER_OK;
}

ember_status ember_kv_layout(const ember_kv* kv, const uint16_t** k_base, const uint16_t** v_base,
                             int64_t strides[4]) {
    if (!kv || !k_base || !v_base || !strides) return fail(EMBER_ERR_INVALID_ARG, "NULL argument");
    if (!kv->m) return fail(EMBER_ERR_STATE, "the model of this cache was destroyed");
    const ember_config& c = kv->m->c;
    *k_base = kv->k;
    *v_base = kv->v;
    strides[2] = (int64_t)kv->max_len * c.head_dim;
    strides[1] = strides[2] * c.n_kv_heads;
    strides[0] = strides[1] * c.layers;
    strides[3] = c.head_dim;
    return EMBER_OK;
}

ember_status ember_sync_status(ember_model* m, ember_stream_t stream) {
    if (!m) return fail(EMBER_ERR_INVALID_ARG, "model is NULL");
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    CK(cudaGetLastError());
    int st = 0;
    CK(cudaMemcpy(&st, m->status, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemset(m->status, 0, 4));
    if (st != 0) return fail((ember_status)st, "device reported status %d", st);
    return EMBER_OK;
}

}  // extern "C"

// ----------------------------------------------------------- launch sequences --
// One decoder layer over n tokens already embedded in m->x, on the
// tensor-core path (whole-prompt prefill, encode, and decode batches > 8).
struct CacheView {
    uint16_t *k, *v;              // base of sequence z = 0, layer 0 handled by caller
    long long seq_stride, head_stride;
    int T_per_seq, pos0, causal;
    const float *cos_t, *sin_t;
    // tensor-core attention (head_dim 64 / 128): the f16 K and transposed-V
    // staging buffers and their maps (keys_pad keys per kv head)
    uint16_t* kh = nullptr;
    const void* kh_map = nullptr;
    uint16_t* vt = nullptr;
    const void* vt_map = nullptr;
    int keys_pad = 0;
};

// Map over a transposed-V buffer [zs][D][keys_pad].
static bool make_vt_map(void* out, const uint16_t* vt, int keys_pad, int D, int zs) {
    const uint64_t d[3] = {(uint64_t)keys_pad, (uint64_t)D, (uint64_t)zs};
    const uint64_t st[2] = {(uint64_t)keys_pad * 2, (uint64_t)keys_pad * D * 2};
    const uint32_t b[3] = {64, (uint32_t)D, 1};
    return encode_map_bf16(out, vt, 3, d, st, b);
}

// Map over an f16 K buffer [zs][keys_pad][D].
static bool make_kh_map(void* out, const uint16_t* kh, int keys_pad, int D, int zs) {
    const uint64_t d[3] = {(uint64_t)D, (uint64_t)keys_pad, (uint64_t)zs};
    const uint64_t st[2] = {(uint64_t)D * 2, (uint64_t)keys_pad * D * 2};
    const uint32_t b[3] = {64, 128, 1};
    return encode_map_bf16(out, kh, 3, d, st, b);
}

static void layer_tc(ember_model* m, int l, int n, const CacheView& cv, cudaStream_t s) {
    const ember_config& c = m->c;
    LayerDev& L = m->layers[l];
    const float eps = (float)c.rms_eps;
    launch_rmsnorm_h(m->x, L.attn_norm, eps, n, c.hidden, m->xb, m->status, s);
    GemmEpilogue e{};
    e.mode = EPI_STORE;
    e.out_f32 = m->qkv;
    e.ldo = m->qkv_n;
    e.bias = c.qkv_bias ? L.bqkv : nullptr;
    e.w_exp = L.e_qkv;
    e.out_map = m->omap_qkv;
    launch_gemm(L.p_qkv, n, e, m->status, s);
    RopeKVArgs r{};
    r.qkv = m->qkv;
    r.ld_qkv = m->qkv_n;
    r.n = n;
    r.NH = c.n_heads;
    r.NKV = c.n_kv_heads;
    r.D = c.head_dim;
    r.T_per_seq = cv.T_per_seq;
    r.pos0 = cv.pos0;
    r.cos_t = cv.cos_t;
    r.sin_t = cv.sin_t;
    r.q_norm = c.qk_norm ? L.q_norm : nullptr;
    r.k_norm = c.qk_norm ? L.k_norm : nullptr;
    r.eps = eps;
    r.q_out = m->qr;
    r.kc = cv.k;
    r.vc = cv.v;
    r.seq_stride = cv.seq_stride;
    r.head_stride = cv.head_stride;
    if (cv.kh_map && cv.vt_map) {   // the attention's f16 K rows of the new tokens
        r.kh = cv.kh;
        r.kh_pad = cv.keys_pad;
    }
    launch_rope_kv(r, s);
    if (cv.kh_map && cv.vt_map) {   // tensor-core attention
        const int nseq = n / cv.T_per_seq;
        const int n_keys = cv.pos0 + cv.T_per_seq;
        VtArgs va{};
        va.v = cv.v;
        va.k = cv.k;
        va.kh = cv.kh;
        va.v_z_stride = cv.seq_stride;
        va.v_h_stride = cv.head_stride;
        va.nkv = c.n_kv_heads;
        va.D = c.head_dim;
        va.n_keys = n_keys;
        va.keys_pad = cv.keys_pad;
        va.vt = cv.vt;
        va.kh_from = cv.pos0;   // Kh of the new tokens came with the RoPE kernel
        launch_vt(va, nseq * c.n_kv_heads, s);
        AttnTcArgs ta{};
        ta.T_per_seq = cv.T_per_seq;
        ta.pos0 = cv.pos0;
        ta.causal = cv.causal;
        ta.n_keys = n_keys;
        ta.NH = c.n_heads;
        ta.NKV = c.n_kv_heads;
        ta.G = c.n_heads / c.n_kv_heads;
        ta.att = m->att_b;
        ta.ld_att = m->q;
        ta.status = m->status;
        launch_attn_tc(m->q_map, cv.kh_map, cv.vt_map, ta, nseq, c.head_dim, s);
    } else {
    AttnPrefillArgs a{};
    a.q = m->qr;
    a.n = n;
    a.NH = c.n_heads;
    a.NKV = c.n_kv_heads;
    a.D = c.head_dim;
    a.T_per_seq = cv.T_per_seq;
    a.pos0 = cv.pos0;
    a.causal = cv.causal;
    a.kc = cv.k;
    a.vc = cv.v;
    a.seq_stride = cv.seq_stride;
    a.head_stride = cv.head_stride;
    a.att = m->att_b;
    a.status = m->status;
    launch_attn_prefill(a, s);
    }
    e = GemmEpilogue{};
    e.mode = EPI_RESID;
    e.out_f32 = m->x;
    e.ldo = c.hidden;
    e.w_exp = L.e_o;
    e.out_map = m->omap_x;
    launch_gemm(L.p_o, n, e, m->status, s);
    launch_rmsnorm_h(m->x, L.mlp_norm, eps, n, c.hidden, m->xb, m->status, s);
    e = GemmEpilogue{};
    e.mode = EPI_SWIGLU;
    e.out_h = m->act_b;
    e.ldo = c.ff;
    e.w_exp = L.e_gu;
    e.out_map = m->omap_act;
    launch_gemm(L.p_gu, n, e, m->status, s);
    e = GemmEpilogue{};
    e.mode = EPI_RESID;
    e.out_f32 = m->x;
    e.ldo = c.hidden;
    e.w_exp = L.e_d;
    e.out_map = m->omap_x;
    launch_gemm(L.p_d, n, e, m->status, s);
}

static ember_status prefill_impl(ember_model* m, ember_kv* kv, int32_t seq, const int32_t* ids,
                                 int32_t n, int32_t start_pos, float* logits, int32_t* argmax,
                                 float* hidden, float* acts, ember_stream_t stream) {
    if (!m || !kv || !ids) return fail(EMBER_ERR_INVALID_ARG, "NULL model, kv or ids");
    if (kv->m != m) return fail(EMBER_ERR_INVALID_ARG, "kv belongs to another model");
    if (n <= 0) return fail(EMBER_ERR_INVALID_ARG, "input_ids must not be empty");
    if (seq < 0 || seq >= kv->max_seqs) return fail(EMBER_ERR_INVALID_ARG, "seq %d out of range", seq);
    if (start_pos < 0) return fail(EMBER_ERR_INVALID_ARG, "negative start_pos");
    if (n > m->T) return fail(EMBER_ERR_CAPACITY, "n = %d > max_tokens = %d", n, m->T);
    if ((long long)start_pos + n > kv->max_len)
        return fail(EMBER_ERR_CAPACITY, "sequence too long: %d + %d > max_len %d", start_pos, n, kv->max_len);
    std::lock_guard<std::mutex> lock(m->mu);
    cudaStream_t s = (cudaStream_t)stream;
    const ember_config& c = m->c;
    EmbedArgs ea{};
    ea.E = m->embed;
    ea.V = c.vocab;
    ea.H = c.hidden;
    ea.ids = ids;
    ea.n = n;
    ea.x = m->x;
    ea.status = m->status;
    ea.pf_seq = seq;
    ea.pf_start = start_pos;
    ea.cursor = kv->cursor;
    launch_embed(ea, s);
    const long long head_stride = (long long)kv->max_len * c.head_dim;
    alignas(64) unsigned char vt_map[128], kh_map[128];
    const int keys_pad = (start_pos + n + 7) / 8 * 8;
    const bool tc = m->q_map_ok && kv->vt && kv->kh &&
                    make_vt_map(vt_map, kv->vt, keys_pad, c.head_dim, c.n_kv_heads) &&
                    make_kh_map(kh_map, kv->kh, keys_pad, c.head_dim, c.n_kv_heads);
    for (int l = 0; l < c.layers; ++l) {
        CacheView cv{};
        if (tc) {
            cv.kh = kv->kh;
            cv.kh_map = kh_map;
            cv.vt = kv->vt;
            cv.vt_map = vt_map;
            cv.keys_pad = keys_pad;
        }
        const long long off = (((long long)seq * c.layers + l) * c.n_kv_heads) * head_stride;
        cv.k = kv->k + off;
        cv.v = kv->v + off;
        cv.seq_stride = 0;
        cv.head_stride = head_stride;
        cv.T_per_seq = n;
        cv.pos0 = start_pos;
        cv.causal = 1;
        cv.cos_t = kv->cos_t;
        cv.sin_t = kv->sin_t;
        layer_tc(m, l, n, cv, s);
        if (acts)   // the residual stream after block l, at the last position
            launch_copy_f32(acts + (size_t)l * c.hidden, m->x + (size_t)(n - 1) * c.hidden, c.hidden, s);
    }
    if (hidden) launch_rmsnorm_f32(m->x, m->final_norm, (float)c.rms_eps, n, c.hidden, hidden, s);
    GemvArgs g{};
    g.W = m->embed;
    g.N = c.vocab;
    g.K = c.hidden;
    g.x = m->x + (size_t)(n - 1) * c.hidden;
    g.ldx = c.hidden;
    g.norm_w = m->final_norm;
    g.eps = (float)c.rms_eps;
    g.out = logits;
    g.ldo = c.vocab;
    g.nb = 1;
    g.mode = EPI_ARGMAX;
    g.keys = m->keys;
    g.status = m->status;
    launch_gemv(g, s, m->sms);
    FinishArgs f{};
    f.nb = 1;
    f.keys = m->keys;
    f.argmax = argmax;
    f.cursor = kv->cursor;
    f.pf_seq = seq;
    f.pf_end = start_pos + n;
    launch_finish(f, s);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_prefill(ember_model* m, ember_kv* kv, int32_t seq, const int32_t* ids,
                                      int32_t n, int32_t start_pos, float* logits, int32_t* argmax,
                                      float* hidden, ember_stream_t stream) {
    return prefill_impl(m, kv, seq, ids, n, start_pos, logits, argmax, hidden, nullptr, stream);
}

extern "C" ember_status ember_prefill_activations(ember_model* m, ember_kv* kv, int32_t seq,
                                                  const int32_t* ids, int32_t n, int32_t start_pos,
                                                  float* acts, float* logits, int32_t* argmax,
                                                  ember_stream_t stream) {
    if (!acts) return fail(EMBER_ERR_INVALID_ARG, "NULL acts");
    return prefill_impl(m, kv, seq, ids, n, start_pos, logits, argmax, nullptr, acts, stream);
}

extern "C" ember_status ember_mean_pooled_head(const float* hidden, int32_t B, int32_t T, int32_t H,
                                               const uint16_t* w, const uint16_t* b, int32_t n_out,
                                               float* out, ember_stream_t stream) {
    if (!hidden || !w || !out) return fail(EMBER_ERR_INVALID_ARG, "NULL hidden, w or out");
    if (B <= 0 || T <= 0 || H <= 0 || n_out <= 0) return fail(EMBER_ERR_INVALID_ARG, "bad sizes");
    if (H > 12288) return fail(EMBER_ERR_INVALID_ARG, "hidden > 12288");
    const cudaError_t e = launch_pooled_head(hidden, B, T, H, w, b, n_out, out, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(EMBER_ERR_CUDA, "pooled head launch failed: %s", cudaGetErrorString(e));
    return EMBER_OK;
}

// Kernel sequence of one decode step (captured into a graph when possible).
static void decode_enqueue(ember_model* m, ember_kv* kv, int B, const int32_t* seqs,
                           const int32_t* ids, const int32_t* positions, float* logits,
                           int32_t* argmax, cudaStream_t s) {
    const ember_config& c = m->c;
    const float eps = (float)c.rms_eps;
    EmbedArgs ea{};
    ea.E = m->embed;
    ea.V = c.vocab;
    ea.H = c.hidden;
    ea.ids = ids;
    ea.n = B;
    ea.x = m->x;
    ea.status = m->status;
    ea.seqs = seqs;
    ea.positions = positions;
    ea.cursor = kv->cursor;
    ea.max_seqs = kv->max_seqs;
    ea.max_len = kv->max_len;
    ea.tok_ok = m->tok_ok;
    ea.tok_pos = m->tok_pos;
    ea.pf_seq = -1;
    if (B == 1 && m->fp.ok && kv->k_map_ok && kv->v_map_ok) {
        // two kernels per layer; kernel n reads fx[(n-1)%2] + fz[(n-1)%3], writes
        // fx[n%2], zeroes fz[(n-2)%3] and accumulates into fz[n%3] (embed: n = 0)
        ea.x = m->fx[0];
        ea.zero0 = m->fz[0];
        ea.zero1 = m->fz[1];
        ea.zlen = c.hidden * ZSLOTS;
        launch_embed(ea, s);
        const FusedPlan& fp = m->fp;
        int n = 1;
        auto io = [&](const float*& xi, const float*& zi, float*& xo, float*& zz, float*& za) {
            xi = m->fx[(n - 1) % 2];
            zi = m->fz[(n - 1) % 3];
            xo = m->fx[n % 2];
            zz = m->fz[(n + 1) % 3];   // (n - 2) mod 3
            za = m->fz[n % 3];
            ++n;
        };
        for (int l = 0; l < c.layers; ++l) {
            LayerDev& L = m->layers[l];
            FusedAttnArgs a{};
            a.wqkv = L.wqkv;
            a.bqkv = c.qkv_bias ? L.bqkv : nullptr;
            a.norm_w = L.attn_norm;
            a.eps = eps;
            a.q_norm = c.qk_norm ? L.q_norm : nullptr;
            a.k_norm = c.qk_norm ? L.k_norm : nullptr;
            a.wo = L.woG;
            a.qkv_exp = L.e_qkv;
            a.zs = fp.zs;
            a.o_exp = L.e_o;
            a.H = c.hidden;
            a.NH = c.n_heads;
            a.NKV = c.n_kv_heads;
            a.D = c.head_dim;
            a.L = c.layers;
            a.layer = l;
            io(a.x_in, a.z_in, a.x_out, a.z_zero, a.z_acc);
            a.kc = kv->k;
            a.vc = kv->v;
            a.max_len = kv->max_len;
            a.max_seqs = kv->max_seqs;
            a.positions = positions;
            a.cursor = kv->cursor;
            a.resident = fp.part ? 1 : 0;
            a.seqs = seqs;
            a.tok_pos = m->tok_pos;
            a.tok_ok = m->tok_ok;
            a.cos_t = kv->cos_t;
            a.sin_t = kv->sin_t;
            a.status = m->status;
            a.C = fp.C;
            a.nr = fp.nr;
            a.no = fp.no;
            launch_fused_attn(kv->k_map, kv->v_map, a, fp.xi, fp.smem_attn, s);
            FusedMlpArgs f{};
            f.wgu = L.wgu;
            f.gu_exp = L.e_gu;
            f.zs = fp.zs;
            f.d_exp = L.e_d;
            f.wdT = L.wdT;
            f.norm_w = L.mlp_norm;
            f.eps = eps;
            f.H = c.hidden;
            f.F = c.ff;
            io(f.x_in, f.z_in, f.x_out, f.z_zero, f.z_acc);
            f.status = m->status;
            f.ns = fp.ns;
            f.pf_late = fp.pf_late;
            f.load_delay_ns = pdl_enabled() ? fp.mlp_delay_ns : 0;
            if (fp.part) launch_fused_mlp_res(f, fp.xi, fp.mlp_grid, fp.smem_mlp, s);
            else launch_fused_mlp(f, fp.fc, fp.xi, fp.mlp_grid, fp.smem_mlp, s);
        }
        GemvArgs g{};
        g.W = m->embed;
        g.N = c.vocab;
        g.K = c.hidden;
        g.x = m->fx[(n - 1) % 2];
        g.x_add = m->fz[(n - 1) % 3];
        g.x_add_slots = m->fp.zs;
        g.ldx = c.hidden;
        g.norm_w = m->final_norm;
        g.eps = eps;
        g.out = logits;
        g.ldo = c.vocab;
        g.nb = 1;
        g.mode = EPI_ARGMAX;
        g.keys = m->keys;
        g.status = m->status;
        launch_gemv(g, s, m->sms);
        FinishArgs f{};
        f.nb = 1;
        f.keys = m->keys;
        f.argmax = argmax;
        f.seqs = seqs;
        f.positions = m->tok_pos;
        f.tok_ok = m->tok_ok;
        f.cursor = kv->cursor;
        f.pf_seq = -1;
        launch_finish(f, s);
        return;
    }
    launch_embed(ea, s);
    const bool gemv = B <= GEMV_MAX_BATCH;
    // a q8_0 model's GEMVs read its codes and scales (the decoded values,
    // unscaled) instead of the f16 copy
    auto q8 = [](GemvArgs& g, const int8_t* q, const uint16_t* d) {
        if (!q) return;
        g.Wq = q;
        g.Wd = d;
        g.w_exp = 0;
    };
    // key splits per (token, kv head): the SIMT kernel wants ~8 CTAs per SM;
    // the tensor-core kernel streams best as one wave of long-lived CTAs at
    // 2 per SM (each with a deep copy ring), so it takes the most splits
    // that still fit in that wave
    const bool mma_attn = kv->k_map_ok && kv->v_map_ok &&
                          attn_decode_mma_supported(c.head_dim, c.n_heads / c.n_kv_heads);
    const int units = B * c.n_kv_heads;
    int splits = mma_attn ? (2 * m->sms) / units : (8 * m->sms + units - 1) / units;
    splits = splits < 1 ? 1 : (splits > MAX_SPLITS ? MAX_SPLITS : splits);
    for (int l = 0; l < c.layers; ++l) {
        LayerDev& L = m->layers[l];
        if (gemv) {
            GemvArgs g{};
            g.W = L.wqkv; g.w_f16 = 1;
            g.w_exp = L.e_qkv;
            q8(g, L.q_qkv, L.d_qkv);
            g.N = m->qkv_n;
            g.K = c.hidden;
            g.x = m->x;
            g.ldx = c.hidden;
            g.norm_w = L.attn_norm;
            g.eps = eps;
            g.bias = c.qkv_bias ? L.bqkv : nullptr;
            g.out = m->qkv;
            g.ldo = m->qkv_n;
            g.nb = B;
            g.mode = EPI_STORE;
            g.status = m->status;
            launch_gemv(g, s, m->sms);
        } else {
            // split K adds into a zeroed output: the norm kernel clears it
            const bool qsplit = gemm_splits(L.p_qkv, B, EPI_STORE) > 1;
            launch_rmsnorm_h(m->x, L.attn_norm, eps, B, c.hidden, m->xb, m->status, s,
                             qsplit ? m->qkv : nullptr, m->qkv_n);
            GemmEpilogue e{};
            e.mode = EPI_STORE;
            e.out_f32 = m->qkv;
            e.ldo = m->qkv_n;
            e.bias = c.qkv_bias ? L.bqkv : nullptr;
            e.zeroed = qsplit ? 1 : 0;
            e.w_exp = L.e_qkv;
            launch_gemm(L.p_qkv, B, e, m->status, s);
        }
        AttnDecodeArgs a{};
        a.qkv = m->qkv;
        a.ld_qkv = m->qkv_n;
        a.nb = B;
        a.NH = c.n_heads;
        a.NKV = c.n_kv_heads;
        a.D = c.head_dim;
        a.L = c.layers;
        a.layer = l;
        a.seqs = seqs;
        a.positions = m->tok_pos;
        a.tok_ok = m->tok_ok;
        a.kc = kv->k;
        a.vc = kv->v;
        a.max_len = kv->max_len;
        a.cos_t = kv->cos_t;
        a.sin_t = kv->sin_t;
        a.q_norm = c.qk_norm ? L.q_norm : nullptr;
        a.k_norm = c.qk_norm ? L.k_norm : nullptr;
        a.eps = eps;
        a.att = m->att_f;
        a.att_b = gemv ? nullptr : m->att_b;
        a.part = m->part;
        a.counters = m->counters;
        a.splits = splits;
        a.status = m->status;
        a.k_map = mma_attn ? kv->k_map : nullptr;
        a.v_map = mma_attn ? kv->v_map : nullptr;
        launch_attn_decode(a, s);
        if (gemv) {
            GemvArgs g{};
            g.W = L.wo; g.w_f16 = 1;
            g.w_exp = L.e_o;
            q8(g, L.q_o, L.d_o);
            g.N = c.hidden;
            g.K = m->q;
            g.x = m->att_f;
            g.ldx = m->q;
            g.out = m->x;
            g.ldo = c.hidden;
            g.nb = B;
            g.mode = EPI_RESID;
            g.status = m->status;
            launch_gemv(g, s, m->sms);
            g = GemvArgs{};
            g.W = L.wgu; g.w_f16 = 1;
            g.w_exp = L.e_gu;
            q8(g, L.q_gu, L.d_gu);
            g.N = 2 * c.ff;
            g.K = c.hidden;
            g.x = m->x;
            g.ldx = c.hidden;
            g.norm_w = L.mlp_norm;
            g.eps = eps;
            g.out = m->act_f;
            g.ldo = c.ff;
            g.nb = B;
            g.mode = EPI_SWIGLU;
            g.status = m->status;
            launch_gemv(g, s, m->sms);
            g = GemvArgs{};
            g.W = L.wd; g.w_f16 = 1;
            g.w_exp = L.e_d;
            q8(g, L.q_d, L.d_d);
            g.N = c.hidden;
            g.K = c.ff;
            g.x = m->act_f;
            g.ldx = c.ff;
            g.out = m->x;
            g.ldo = c.hidden;
            g.nb = B;
            g.mode = EPI_RESID;
            g.status = m->status;
            launch_gemv(g, s, m->sms);
        } else {
            // the attention kernel wrote its output as the f16 GEMM operand att_b
            GemmEpilogue e{};
            e.mode = EPI_RESID;
            e.out_f32 = m->x;
            e.ldo = c.hidden;
            e.w_exp = L.e_o;
            launch_gemm(L.p_o, B, e, m->status, s);
            launch_rmsnorm_h(m->x, L.mlp_norm, eps, B, c.hidden, m->xb, m->status, s);
            e = GemmEpilogue{};
            e.mode = EPI_SWIGLU;
            e.out_h = m->act_b;
            e.ldo = c.ff;
            e.w_exp = L.e_gu;
            launch_gemm(L.p_gu, B, e, m->status, s);
            e = GemmEpilogue{};
            e.mode = EPI_RESID;
            e.out_f32 = m->x;
            e.ldo = c.hidden;
            e.w_exp = L.e_d;
            launch_gemm(L.p_d, B, e, m->status, s);
        }
    }
    // LM head + argmax: the split GEMV for up to GEMV_MAX_BATCH tokens, else one
    // tensor-core GEMM over the bf16 final states (the vocabulary is read once)
    if (!gemv) {
        launch_rmsnorm_bf16(m->x, m->final_norm, eps, B, c.hidden, m->hb, s);
        GemmEpilogue e{};
        e.mode = EPI_ARGMAX;
        e.out_f32 = logits;
        e.ldo = c.vocab;
        e.keys = m->keys;
        launch_gemm(m->p_head, B, e, m->status, s);
    }
    for (int b0 = 0; gemv && b0 < B; b0 += GEMV_MAX_BATCH) {
        GemvArgs g{};
        g.W = m->embed;
        g.N = c.vocab;
        g.K = c.hidden;
        g.x = m->x + (size_t)b0 * c.hidden;
        g.ldx = c.hidden;
        g.norm_w = m->final_norm;
        g.eps = eps;
        g.out = logits ? logits + (size_t)b0 * c.vocab : nullptr;
        g.ldo = c.vocab;
        g.nb = (B - b0) < GEMV_MAX_BATCH ? (B - b0) : GEMV_MAX_BATCH;
        g.mode = EPI_ARGMAX;
        g.keys = m->keys + b0;
        g.status = m->status;
        launch_gemv(g, s, m->sms);
    }
    FinishArgs f{};
    f.nb = B;
    f.keys = m->keys;
    f.argmax = argmax;
    f.seqs = seqs;
    f.positions = m->tok_pos;
    f.tok_ok = m->tok_ok;
    f.cursor = kv->cursor;
    f.pf_seq = -1;
    launch_finish(f, s);
}

extern "C" ember_status ember_decode_step(ember_model* m, ember_kv* kv, int32_t batch,
                                          const int32_t* seqs, const int32_t* ids,
                                          const int32_t* positions, float* logits, int32_t* argmax,
                                          ember_stream_t stream) {
    if (!m || !kv || !seqs || !ids)
        return fail(EMBER_ERR_INVALID_ARG, "NULL model, kv, seqs or ids");
    if (kv->m != m) return fail(EMBER_ERR_INVALID_ARG, "kv belongs to another model");
    if (batch <= 0) return fail(EMBER_ERR_INVALID_ARG, "batch must be > 0");
    if (batch > MAX_DECODE_BATCH || batch > m->T || batch > kv->max_seqs)
        return fail(EMBER_ERR_CAPACITY, "batch %d exceeds the decode capacity", batch);
    std::lock_guard<std::mutex> lock(m->mu);
    cudaStream_t s = (cudaStream_t)stream;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    CK(cudaStreamIsCapturing(s, &cap));
    if (!m->use_graphs || s == nullptr || cap != cudaStreamCaptureStatusNone) {
        decode_enqueue(m, kv, batch, seqs, ids, positions, logits, argmax, s);
        CK(cudaGetLastError());
        return EMBER_OK;
    }
    for (auto& g : m->graphs) {
        if (g.kv_gen == kv->gen && g.batch == batch && g.seqs == seqs && g.ids == ids && g.pos == positions &&
            g.logits == logits && g.argmax == argmax) {
            CK(cudaGraphLaunch(g.exec, s));
            count_launches(g.kernels);
            return EMBER_OK;
        }
    }
    cudaGraph_t graph = nullptr;
    CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    const long long before = (long long)launches_so_far();
    decode_enqueue(m, kv, batch, seqs, ids, positions, logits, argmax, s);
    const long long kernels = (long long)launches_so_far() - before;
    count_launches(-kernels);   // captured, not run
    const cudaError_t le = cudaGetLastError();   // a launch the capture rejected
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (e != cudaSuccess)
        return fail(EMBER_ERR_CUDA, "graph capture failed: %s (launch error: %s)", cudaGetErrorString(e),
                    cudaGetErrorString(le));
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(EMBER_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
    if (m->graphs.size() >= 16) {
        cudaGraphExecDestroy(m->graphs.front().exec);
        m->graphs.erase(m->graphs.begin());
    }
    m->graphs.push_back({kv->gen, batch, seqs, ids, positions, logits, argmax, exec, kernels});
    CK(cudaGraphLaunch(exec, s));
    count_launches(kernels);
    return EMBER_OK;
}

extern "C" ember_status ember_decode_step_traced(ember_model* m, ember_kv* kv, int32_t batch,
                                                 const int32_t* seqs, const int32_t* ids,
                                                 const int32_t* positions, float* logits, int32_t* argmax,
                                                 ember_stream_t stream, float* launch_us, const char** names,
                                                 int32_t cap, int32_t* n) {
    if (!m || !kv || !seqs || !ids || !n || cap < 0 || (cap > 0 && (!launch_us || !names)))
        return fail(EMBER_ERR_INVALID_ARG, "NULL model, kv, seqs, ids, n, or trace buffers");
    if (kv->m != m) return fail(EMBER_ERR_INVALID_ARG, "kv belongs to another model");
    if (batch <= 0) return fail(EMBER_ERR_INVALID_ARG, "batch must be > 0");
    if (batch > MAX_DECODE_BATCH || batch > m->T || batch > kv->max_seqs)
        return fail(EMBER_ERR_CAPACITY, "batch %d exceeds the decode capacity", batch);
    std::lock_guard<std::mutex> lock(m->mu);
    cudaStream_t s = (cudaStream_t)stream;
    cudaStreamCaptureStatus capst = cudaStreamCaptureStatusNone;
    CK(cudaStreamIsCapturing(s, &capst));
    if (capst != cudaStreamCaptureStatusNone)
        return fail(EMBER_ERR_INVALID_ARG, "a traced step cannot be captured");
    // captured into a one-off graph (event-record nodes between the kernel
    // nodes), so that host launch latency adds no gaps between launches
    LaunchTrace tr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        g_trace = &tr;
        decode_enqueue(m, kv, batch, seqs, ids, positions, logits, argmax, s);
        trace_launch(nullptr, s);   // the end of the last launch
        g_trace = nullptr;
        const cudaError_t le = cudaGetLastError();
        e = cudaStreamEndCapture(s, &graph);
        if (e == cudaSuccess) e = le;
        if (e == cudaSuccess) e = tr.err;
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
    if (e == cudaSuccess) e = cudaGraphLaunch(exec, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    const int k = (int)tr.ev.size() - 1;
    *n = k < 0 ? 0 : k;
    for (int i = 0; e == cudaSuccess && i < k && i < cap; ++i) {
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, tr.ev[i], tr.ev[i + 1]);
        launch_us[i] = ms * 1e3f;
        const char* nm = nullptr;
        names[i] = cudaFuncGetName(&nm, tr.fn[i]) == cudaSuccess && nm ? nm : "?";
    }
    for (cudaEvent_t ev : tr.ev) cudaEventDestroy(ev);
    if (e != cudaSuccess) return fail(EMBER_ERR_CUDA, "traced decode step: %s", cudaGetErrorString(e));
    return EMBER_OK;
}

extern "C" ember_status ember_encode(ember_model* m, const int32_t* ids, int32_t B, int32_t T,
                                     float* out, float* hidden, ember_stream_t stream) {
    if (!m || !ids) return fail(EMBER_ERR_INVALID_ARG, "NULL model or ids");
    if (B <= 0 || T <= 0) return fail(EMBER_ERR_INVALID_ARG, "input_ids must not be empty");
    if ((long long)B * T > m->T) return fail(EMBER_ERR_CAPACITY, "B*T = %lld > max_tokens %d", (long long)B * T, m->T);
    if (m->c.causal) return fail(EMBER_ERR_UNSUPPORTED, "encode of a causal model is not built yet");
    if (T > m->c.max_positions) return fail(EMBER_ERR_CAPACITY, "T = %d > max_positions %d", T, m->c.max_positions);
    std::lock_guard<std::mutex> lock(m->mu);
    cudaStream_t s = (cudaStream_t)stream;
    const ember_config& c = m->c;
    const int n = B * T;
    EmbedArgs ea{};
    ea.E = m->embed;
    ea.V = c.vocab;
    ea.H = c.hidden;
    ea.ids = ids;
    ea.n = n;
    ea.x = m->x;
    ea.status = m->status;
    ea.pf_seq = -1;
    launch_embed(ea, s);
    alignas(64) unsigned char kh_map[128], vt_map[128];
    const int keys_pad = (T + 7) / 8 * 8;
    const bool tc = m->q_map_ok &&
                    make_kh_map(kh_map, m->enc_kh, keys_pad, c.head_dim, B * c.n_kv_heads) &&
                    make_vt_map(vt_map, m->enc_vt, keys_pad, c.head_dim, B * c.n_kv_heads);
    for (int l = 0; l < c.layers; ++l) {
        CacheView cv{};
        if (tc) {
            cv.kh = m->enc_kh;
            cv.kh_map = kh_map;
            cv.vt = m->enc_vt;
            cv.vt_map = vt_map;
            cv.keys_pad = keys_pad;
        }
        cv.k = m->enc_k;
        cv.v = m->enc_v;
        cv.head_stride = (long long)T * c.head_dim;
        cv.seq_stride = cv.head_stride * c.n_kv_heads;
        cv.T_per_seq = T;
        cv.pos0 = 0;
        cv.causal = c.causal;
        cv.cos_t = m->enc_cos;
        cv.sin_t = m->enc_sin;
        layer_tc(m, l, n, cv, s);
    }
    float* h = hidden ? hidden : m->hbuf;
    launch_rmsnorm_f32(m->x, m->final_norm, (float)c.rms_eps, n, c.hidden, h, s);
    if (out) {
        if (c.n_labels > 0) {
            launch_cls_head(h, n, c.hidden, m->cls_w, m->cls_b, c.n_labels, out, s);
        } else {
            // tied vocabulary head at every position: the final states in bf16
            // (the embedding's type) times the embedding rows, one GEMM
            launch_rmsnorm_bf16(m->x, m->final_norm, (float)c.rms_eps, n, c.hidden, m->hb, s);
            GemmEpilogue e{};
            e.mode = EPI_STORE;
            e.out_f32 = out;
            e.ldo = c.vocab;
            launch_gemm(m->p_head, n, e, m->status, s);
        }
    }
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_rope_store(const float* x, int32_t n_tok, int32_t n_heads,
                                         int32_t head_dim, const float* cos_t, const float* sin_t,
                                         uint16_t* out, ember_stream_t stream) {
    if (!x || !cos_t || !sin_t || !out) return fail(EMBER_ERR_INVALID_ARG, "NULL pointer");
    if (n_tok <= 0 || n_heads <= 0 || head_dim <= 0 || head_dim % 2)
        return fail(EMBER_ERR_INVALID_ARG, "bad sizes");
    launch_rope_store(x, n_tok, n_heads, head_dim, cos_t, sin_t, out, (cudaStream_t)stream);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_gemm_bf16(const uint16_t* A, const uint16_t* Bm, float* Dm, int32_t M,
                                        int32_t N, int32_t K, ember_stream_t stream) {
    if (!A || !Bm || !Dm) return fail(EMBER_ERR_INVALID_ARG, "NULL pointer");
    if (M <= 0 || N <= 0 || K <= 0 || K % 8 || N % 4)
        return fail(EMBER_ERR_INVALID_ARG, "M, N, K must be > 0, K %% 8 == 0, N %% 4 == 0");
    GemmPlan p;
    if (!make_gemm_plan(p, A, M, K, Bm, N, K, K, false))
        return fail(EMBER_ERR_INVALID_ARG, "TMA tensor map rejected (alignment?)");
    alignas(64) unsigned char omap[128];
    if (!make_out_map(omap, Dm, M, N, N, false))
        return fail(EMBER_ERR_INVALID_ARG, "TMA tensor map rejected for D (alignment?)");
    GemmEpilogue e{};
    e.mode = EPI_STORE;
    e.out_f32 = Dm;
    e.ldo = N;
    e.out_map = omap;   // copied into the launch's parameters
    launch_gemm(p, M, e, nullptr, (cudaStream_t)stream);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_gemv_bf16(const uint16_t* W, int32_t N, int32_t K, const float* x,
                                        int32_t nb, float* y, ember_stream_t stream) {
    if (!W || !x || !y) return fail(EMBER_ERR_INVALID_ARG, "NULL pointer");
    if (N <= 0 || K <= 0 || K % 8 || K > 16384 || nb <= 0 || nb > GEMV_MAX_BATCH)
        return fail(EMBER_ERR_INVALID_ARG, "N, K > 0, K %% 8 == 0, K <= 16384, 1 <= nb <= 8");
    if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(x)) & 15)
        return fail(EMBER_ERR_INVALID_ARG, "W and x must be 16-byte aligned");
    int dev = 0, sms = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    GemvArgs g{};
    g.W = W;
    g.N = N;
    g.K = K;
    g.x = x;
    g.ldx = K;
    g.out = y;
    g.ldo = N;
    g.nb = nb;
    g.mode = EPI_STORE;
    launch_gemv(g, (cudaStream_t)stream, sms);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_q8_0_quantize(const uint16_t* w, int64_t n, int8_t* q, uint16_t* d,
                                           ember_stream_t stream) {
    if (!w || !q || !d) return fail(EMBER_ERR_INVALID_ARG, "NULL pointer");
    if (n <= 0 || n % 32) return fail(EMBER_ERR_INVALID_ARG, "n must be a positive multiple of 32");
    launch_q8_0_quantize(w, n, q, d, nullptr, 0, (cudaStream_t)stream);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_gemv_q8_0(const int8_t* q, const uint16_t* d, int32_t N, int32_t K,
                                        const float* x, int32_t nb, float* y, ember_stream_t stream) {
    if (!q || !d || !x || !y) return fail(EMBER_ERR_INVALID_ARG, "NULL pointer");
    if (N <= 0 || K <= 0 || K % 32 || K > 16384 || nb <= 0 || nb > GEMV_MAX_BATCH)
        return fail(EMBER_ERR_INVALID_ARG, "N, K > 0, K %% 32 == 0, K <= 16384, 1 <= nb <= 8");
    if ((reinterpret_cast<uintptr_t>(q) & 7) | (reinterpret_cast<uintptr_t>(d) & 1) |
        (reinterpret_cast<uintptr_t>(x) & 15))
        return fail(EMBER_ERR_INVALID_ARG, "q must be 8-byte, d 2-byte and x 16-byte aligned");
    int dev = 0, sms = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    GemvArgs g{};
    g.Wq = q;
    g.Wd = d;
    g.N = N;
    g.K = K;
    g.x = x;
    g.ldx = K;
    g.out = y;
    g.ldo = N;
    g.nb = nb;
    g.mode = EPI_STORE;
    launch_gemv(g, (cudaStream_t)stream, sms);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" ember_status ember_sample(const float* logits, int32_t B, int32_t V, int32_t ldl,
                                     float temperature, int32_t top_k, float top_p, const float* r,
                                     int32_t* out, ember_stream_t stream) {
    if (!logits || !out || (temperature > 0.f && !r))
        return fail(EMBER_ERR_INVALID_ARG, "NULL logits, out, or draws (r is needed when temperature > 0)");
    if (B <= 0 || V <= 0 || ldl < V) return fail(EMBER_ERR_INVALID_ARG, "bad sizes (B, V > 0, ldl >= V)");
    if (top_k < 0) return fail(EMBER_ERR_INVALID_ARG, "top_k < 0");
    if (top_p != top_p || temperature != temperature) return fail(EMBER_ERR_INVALID_ARG, "NaN temperature or top_p");
    SampleArgs a{};
    a.logits = logits;
    a.B = B;
    a.V = V;
    a.ldl = ldl;
    a.t = temperature;
    a.k = top_k;
    a.p = top_p;
    a.r = r;
    a.out = out;
    const cudaError_t e = launch_sample(a, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(EMBER_ERR_CUDA, "sampler launch failed: %s", cudaGetErrorString(e));
    return EMBER_OK;
}

extern "C" ember_status ember_test_bounded_wait(ember_model* m, int32_t which, int64_t budget_cycles,
                                                ember_stream_t stream) {
    if (!m) return fail(EMBER_ERR_INVALID_ARG, "NULL model");
    if (which != 0 && which != 1) return fail(EMBER_ERR_INVALID_ARG, "which must be 0 or 1");
    if (budget_cycles < 0 || budget_cycles > 200000000ll)
        return fail(EMBER_ERR_INVALID_ARG, "budget must be in [0, 2e8] cycles");
    launch_wait_probe(which, budget_cycles, m->status, (cudaStream_t)stream);
    CK(cudaGetLastError());
    return EMBER_OK;
}

extern "C" uint64_t ember_kernel_launches(void) { return (uint64_t)launches_so_far(); }

// ====================================== greedy LM head without allocation ==
// ember_gemv_argmax_noalloc: the split GEMV with its argmax epilogue, for a
// caller that may not allocate device memory (its whole budget is already
// handed out, e.g. to a KV pool, or it cannot afford the device-wide stall a
// cudaMalloc / cudaFree can cause on its latency path).  The per-row argmax
// keys live in a fixed file-scope device array instead of a caller buffer.

namespace {

// One u64 key per input row: (order-preserving logit bits << 32 | ~index).
// The GEMV CTAs atomicMax into it, so it must hold zero when a call starts;
// the set-up zeroes it once and every call's finishing kernel zeroes it again
// after reading it.  64 bytes per device.
static __device__ __align__(256) unsigned long long g_noalloc_keys[EMBER_NOALLOC_MAX_ROWS];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
unsigned long long* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};
int g_noalloc_sms[NOALLOC_MAX_DEVICES] = {};

// keys -> int32 argmax, then clear the keys for the next call
__global__ void k_noalloc_finish(unsigned long long* keys, int nb, int32_t* argmax) {
    pdl_wait();
    const int b = threadIdx.x;
    if (b < nb) {
        argmax[b] = argmax_key_index(keys[b]);
        keys[b] = 0ull;
    }
}

// First call on a device (that device current): resolve the scratch address
// and clear it, ordered on the caller's stream.  Returns nullptr on failure.
unsigned long long* noalloc_scratch(int dev, cudaStream_t s, int* sms, ember_status* st) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev]) {
        *sms = g_noalloc_sms[dev];
        return g_noalloc_ptr[dev];
    }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_keys);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&g_noalloc_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(g_noalloc_keys), s);
    if (e != cudaSuccess) {
        *st = fail(EMBER_ERR_CUDA, "no-alloc set-up on device %d failed: %s", dev,
                   cudaGetErrorString(e));
        return nullptr;
    }
    g_noalloc_ptr[dev] = static_cast<unsigned long long*>(p);
    *sms = g_noalloc_sms[dev];
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" ember_status ember_gemv_argmax_noalloc(const uint16_t* W, int32_t N, int32_t K,
                                                  const float* x, int32_t nb, float* y,
                                                  int32_t* argmax, ember_stream_t stream) {
    if (!W || !x || !argmax) return fail(EMBER_ERR_INVALID_ARG, "NULL pointer");
    if (nb > EMBER_NOALLOC_MAX_ROWS)
        return fail(EMBER_ERR_CAPACITY,
                    "nb = %d rows exceeds the fixed scratch of EMBER_NOALLOC_MAX_ROWS = %d rows",
                    nb, EMBER_NOALLOC_MAX_ROWS);
    if (N <= 0 || K <= 0 || K % 8 || K > 16384 || nb <= 0)
        return fail(EMBER_ERR_INVALID_ARG, "N, K > 0, K %% 8 == 0, K <= 16384, nb >= 1");
    if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(x)) & 15)
        return fail(EMBER_ERR_INVALID_ARG, "W and x must be 16-byte aligned");
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES)
        return fail(EMBER_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, NOALLOC_MAX_DEVICES);
    const cudaStream_t s = (cudaStream_t)stream;
    int sms = 0;
    ember_status st = EMBER_OK;
    unsigned long long* keys = noalloc_scratch(dev, s, &sms, &st);
    if (!keys) return st;

    GemvArgs g{};
    g.W = W;
    g.N = N;
    g.K = K;
    g.x = x;
    g.ldx = K;
    g.out = y;   // logits too, when the caller wants them
    g.ldo = N;
    g.nb = nb;
    g.mode = EPI_ARGMAX;
    g.keys = keys;
    // Only the two launches' own return codes are checked: an error the caller
    // left pending on this thread is not this call's failure.  Once the GEMV
    // may be queued, any failure leaves keys that nothing clears, so the next
    // call redoes the set-up (which clears them on its stream).
    cudaError_t e = launch_gemv(g, s, sms);
    if (e == cudaSuccess) e = launch_k(k_noalloc_finish, dim3(1), dim3(32), 0, s, keys, (int)nb, argmax);
    if (e != cudaSuccess) {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        g_noalloc_ptr[dev] = nullptr;
        return fail(EMBER_ERR_CUDA, "no-alloc LM head launch failed: %s", cudaGetErrorString(e));
    }
    return EMBER_OK;
}
