// Host runtime behind the C ABI of include/qwdecode.h: configuration checks,
// weight upload and repacking, workspaces, the paged KV pool, and the launch
// sequences of prefill, decode and sampling.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <vector>

#include "qw_common.cuh"
#include "qw_fused.h"
#include "qw_internal.h"

using namespace qw;
namespace qw {
unsigned long long launches_so_far();
}

namespace {
thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}
}  // namespace

namespace qw {
int report_error(int code, const char* msg) { return fail(code, msg); }
}  // namespace qw

#define QW_CUDA(call)                                                                              \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess) return fail(QW_ECUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
    } while (0)
#define QW_TRY(call, what)                                  \
    do {                                                    \
        int rc_ = (call);                                   \
        if (rc_ != QW_OK) return fail(rc_, what);           \
    } while (0)

struct LayerW {
    uint16_t *wqkv, *wo, *wgu, *wd;  // [qkv_dim][D], [D][Hq*d], [2I][D] (gate, up rows interleaved), [D][I]
    float *in_norm, *post_norm, *q_norm, *k_norm;
    CUtensorMap tm_qkv, tm_o, tm_gu, tm_d;
    CUtensorMap tm_o256, tm_d256;   // o_proj / down_proj with 256-row boxes (large-M products)
    CUtensorMap tm_qkv128, tm_gu128;  // q|k|v and gate/up with 128-row boxes (CTA-pair halves)
    CUtensorMap tm_qkv32, tm_gu64, tm_o32, tm_d32;  // narrow boxes for decode batches
};

// Per-kernel-class device time (qw_debug_profile): CUDA events recorded on the launching
// stream around each launch of a class while enabled.
struct Profiler {
    bool on = false;
    std::vector<cudaEvent_t> ev;       // pairs (start, end); reused across enables
    std::vector<int> cls;              // class of pair i
    size_t used = 0;                   // pairs recorded since the last enable
};

struct qw_ctx {
    qw_config cfg;
    int dev = 0, n_sm = 0;
    int qkv_dim = 0, attn_dim = 0;
    uint8_t* wbuf = nullptr;
    uint8_t* qbuf = nullptr;   // weight_bits 8: int8 codes and per-output-channel scales
    uint16_t* E = nullptr;
    float* final_norm = nullptr;
    float* inv_freq = nullptr;
    std::vector<LayerW> L;
    CUtensorMap tm_E;
    // workspaces
    uint8_t* wsbuf = nullptr;
    float *x = nullptr, *qkv = nullptr, *q = nullptr, *logits = nullptr, *part = nullptr, *hidden = nullptr;
    uint16_t *h = nullptr, *attn = nullptr, *act = nullptr, *q_bf16 = nullptr;
    float2* rope_tab = nullptr;   // [rows][64] RoPE (cos, sin) of the current prefill
    float2* tile_part = nullptr;  // [max_batch][n_part] per-256-column (max, argmax) of the context's logits
    int n_part = 0;
    int part_rows = 0;            // rows of the context's logits that tile_part describes (0: none)
    int* gen_pos = nullptr;       // [GEN_CHUNK] positions of a qw_generate chunk
    int *tok_seq = nullptr, *iota = nullptr, *rows_last = nullptr, *err = nullptr;
    int4* tiles = nullptr;
    int max_rows = 0, max_splits = 128, max_tiles = 0;
    int last_rows = 0, logits_rows = 0;
    int decode_path = 0;
    int prefill_attn = 0;   // 0: tcgen05 kernel, 1: mma.sync kernel
    FusedDecode* fused = nullptr;
    bool last_fused = false;   // the last decode step ran the fused kernel (its argmax is valid)
    Profiler prof;
};

// Records the start of a launch of class `cls` on construction and its end on destruction
// (nothing unless profiling is on).
struct ProfScope {
    qw_ctx* c;
    int idx = -1;
    cudaStream_t st;
    ProfScope(qw_ctx* ctx, int cls, cudaStream_t s) : c(ctx), st(s) {
        Profiler& p = c->prof;
        if (!p.on) return;
        if (p.used * 2 + 2 > p.ev.size()) {
            cudaEvent_t a, b;
            if (cudaEventCreate(&a) != cudaSuccess) return;
            if (cudaEventCreate(&b) != cudaSuccess) {
                cudaEventDestroy(a);
                return;
            }
            p.ev.push_back(a);
            p.ev.push_back(b);
            p.cls.push_back(cls);
        }
        idx = (int)p.used++;
        p.cls[idx] = cls;
        cudaEventRecord(p.ev[2 * idx], st);
    }
    ~ProfScope() {
        if (idx >= 0) cudaEventRecord(c->prof.ev[2 * idx + 1], st);
    }
};
#define QW_PROF(cls) ProfScope prof_scope_(ctx, cls, st)

struct qw_kv {
    qw_ctx* ctx;
    uint16_t* base;
    int32_t n_pages;
    int64_t page_elems;   // elements per page (2 * n_kv * 16 * 128)
    int64_t layer_elems;  // elements per layer (n_pages * page_elems)
};

extern "C" {

void qw_config_default(qw_config* c) {
    if (!c) return;
    c->n_layers = 28;
    c->hidden = 1024;
    c->n_heads = 16;
    c->n_kv_heads = 8;
    c->head_dim = QW_HEAD_DIM;
    c->intermediate = 3072;
    c->vocab = 151936;
    c->max_batch = 64;
    c->max_tokens = 16384;
    c->debug_hidden = 0;
    c->rms_eps = 1e-6f;
    c->rope_theta = 1e6;
    c->weight_bits = 16;
}

const char* qw_last_error_message(void) { return g_last_error.c_str(); }

static int validate_config(const qw_config* c) {
    if (c->n_layers < 1 || c->n_layers > 256) return fail(QW_EINVAL, "n_layers must be in [1, 256]");
    if (c->hidden < 256 || c->hidden % 256 || c->hidden > 4096)
        return fail(QW_EINVAL, "hidden must be a multiple of 256 in [256, 4096]");
    if (c->head_dim != QW_HEAD_DIM) return fail(QW_EINVAL, "head_dim must be 128");
    if (!group_size_ok(c->n_heads, c->n_kv_heads))
        return fail(QW_EINVAL, "n_heads must be n_kv_heads times 1, 2, 4, 8 or 16 (query heads per KV head)");
    if ((c->n_heads * c->head_dim) % 256) return fail(QW_EINVAL, "n_heads * head_dim must be a multiple of 256");
    if (c->intermediate < 128 || c->intermediate % 128) return fail(QW_EINVAL, "intermediate must be a multiple of 128");
    if (c->vocab < 32 || c->vocab % 32) return fail(QW_EINVAL, "vocab must be a positive multiple of 32");
    if (c->max_batch < 1 || c->max_batch > 256) return fail(QW_EINVAL, "max_batch must be in [1, 256]");
    if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) return fail(QW_EINVAL, "max_tokens must be in [1, 2^20]");
    if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.0)) return fail(QW_EINVAL, "rms_eps > 0 and rope_theta > 1 required");
    if (c->weight_bits != 16 && c->weight_bits != 8) return fail(QW_EINVAL, "weight_bits must be 16 or 8");
    return QW_OK;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int upload_norm(float* dst, const uint16_t* src, int n, int on_device) {
    if (on_device) {
        QW_TRY(launch_bf16_to_f32(src, dst, n, 0), "bf16_to_f32 launch");
        return QW_OK;
    }
    std::vector<float> tmp(n);
    for (int i = 0; i < n; ++i) {
        uint32_t b = (uint32_t)src[i] << 16;
        memcpy(&tmp[i], &b, 4);
    }
    QW_CUDA(cudaMemcpy(dst, tmp.data(), n * sizeof(float), cudaMemcpyHostToDevice));
    return QW_OK;
}

static void free_ctx(qw_ctx* c) {
    if (!c) return;
    for (cudaEvent_t e : c->prof.ev) cudaEventDestroy(e);
    if (c->fused) fused_destroy(c->fused);
    if (c->wbuf) cudaFree(c->wbuf);
    if (c->qbuf) cudaFree(c->qbuf);
    if (c->wsbuf) cudaFree(c->wsbuf);
    delete c;
}

int qw_init(const qw_config* cfg, const qw_weights* w, qw_ctx** out) {
    if (!cfg || !w || !out) return fail(QW_EINVAL, "null argument");
    *out = nullptr;
    int rc = validate_config(cfg);
    if (rc) return rc;
    const qw_config& c = *cfg;
    if (!w->embed_tokens || !w->norm || !w->input_layernorm || !w->q_proj || !w->k_proj || !w->v_proj ||
        !w->q_norm || !w->k_norm || !w->o_proj || !w->post_attention_layernorm || !w->gate_proj || !w->up_proj ||
        !w->down_proj)
        return fail(QW_EINVAL, "null weight pointer");
    for (int l = 0; l < c.n_layers; ++l)
        if (!w->input_layernorm[l] || !w->q_proj[l] || !w->k_proj[l] || !w->v_proj[l] || !w->q_norm[l] ||
            !w->k_norm[l] || !w->o_proj[l] || !w->post_attention_layernorm[l] || !w->gate_proj[l] ||
            !w->up_proj[l] || !w->down_proj[l])
            return fail(QW_EINVAL, "null per-layer weight pointer");

    qw_ctx* ctx = new qw_ctx();
    ctx->cfg = c;
    cudaGetDevice(&ctx->dev);
    cudaDeviceGetAttribute(&ctx->n_sm, cudaDevAttrMultiProcessorCount, ctx->dev);
    const int D = c.hidden, Hq = c.n_heads, Hkv = c.n_kv_heads, d = c.head_dim, I = c.intermediate, V = c.vocab;
    ctx->qkv_dim = (Hq + 2 * Hkv) * d;
    ctx->attn_dim = Hq * d;

    // ---- weights: one allocation, 1 KiB-aligned pieces
    const size_t A = 1024;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, A);
        return o;
    };
    const size_t oE = take((size_t)V * D * 2);
    const size_t oFinal = take((size_t)D * 4);
    const size_t oFreq = take(64 * 4);
    struct Offs { size_t qkv, o, gu, dn, inn, post, qn, kn; };
    std::vector<Offs> lo(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        lo[l].qkv = take((size_t)ctx->qkv_dim * D * 2);
        lo[l].o = take((size_t)D * ctx->attn_dim * 2);
        lo[l].gu = take((size_t)2 * I * D * 2);
        lo[l].dn = take((size_t)D * I * 2);
        lo[l].inn = take((size_t)D * 4);
        lo[l].post = take((size_t)D * 4);
        lo[l].qn = take((size_t)d * 4);
        lo[l].kn = take((size_t)d * 4);
    }
    if (cudaMalloc(&ctx->wbuf, off) != cudaSuccess) {
        free_ctx(ctx);
        return fail(QW_ENOMEM, "weight allocation failed");
    }
    const cudaMemcpyKind kind = w->on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    uint8_t* B = ctx->wbuf;
    ctx->E = (uint16_t*)(B + oE);
    ctx->final_norm = (float*)(B + oFinal);
    ctx->inv_freq = (float*)(B + oFreq);
#define QW_INIT_CUDA(call)                                                                          \
    do {                                                                                            \
        cudaError_t e_ = (call);                                                                    \
        if (e_ != cudaSuccess) {                                                                    \
            free_ctx(ctx);                                                                          \
            return fail(QW_ECUDA, std::string(#call) + ": " + cudaGetErrorString(e_));              \
        }                                                                                           \
    } while (0)
    QW_INIT_CUDA(cudaMemcpy(ctx->E, w->embed_tokens, (size_t)V * D * 2, kind));
    if ((rc = upload_norm(ctx->final_norm, w->norm, D, w->on_device))) {
        free_ctx(ctx);
        return rc;
    }
    {
        // RoPE inverse frequencies (Step 4): float32(theta^(-i/half)), evaluated in double
        float f[64];
        for (int i = 0; i < d / 2; ++i) f[i] = (float)(1.0 / pow(c.rope_theta, (double)i / (double)(d / 2)));
        QW_INIT_CUDA(cudaMemcpy(ctx->inv_freq, f, sizeof(float) * (d / 2), cudaMemcpyHostToDevice));
    }
    ctx->L.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        LayerW& Lw = ctx->L[l];
        Lw.wqkv = (uint16_t*)(B + lo[l].qkv);
        Lw.wo = (uint16_t*)(B + lo[l].o);
        Lw.wgu = (uint16_t*)(B + lo[l].gu);
        Lw.wd = (uint16_t*)(B + lo[l].dn);
        Lw.in_norm = (float*)(B + lo[l].inn);
        Lw.post_norm = (float*)(B + lo[l].post);
        Lw.q_norm = (float*)(B + lo[l].qn);
        Lw.k_norm = (float*)(B + lo[l].kn);
        const size_t rowb = (size_t)D * 2;
        QW_INIT_CUDA(cudaMemcpy(Lw.wqkv, w->q_proj[l], (size_t)Hq * d * rowb, kind));
        QW_INIT_CUDA(cudaMemcpy(Lw.wqkv + (size_t)Hq * d * D, w->k_proj[l], (size_t)Hkv * d * rowb, kind));
        QW_INIT_CUDA(cudaMemcpy(Lw.wqkv + (size_t)(Hq + Hkv) * d * D, w->v_proj[l], (size_t)Hkv * d * rowb, kind));
        QW_INIT_CUDA(cudaMemcpy(Lw.wo, w->o_proj[l], (size_t)D * ctx->attn_dim * 2, kind));
        // gate row j -> packed row 2j, up row j -> packed row 2j+1
        QW_INIT_CUDA(cudaMemcpy2D(Lw.wgu, 2 * rowb, w->gate_proj[l], rowb, rowb, I, kind));
        QW_INIT_CUDA(cudaMemcpy2D(Lw.wgu + D, 2 * rowb, w->up_proj[l], rowb, rowb, I, kind));
        QW_INIT_CUDA(cudaMemcpy(Lw.wd, w->down_proj[l], (size_t)D * I * 2, kind));
        if ((rc = upload_norm(Lw.in_norm, w->input_layernorm[l], D, w->on_device)) ||
            (rc = upload_norm(Lw.post_norm, w->post_attention_layernorm[l], D, w->on_device)) ||
            (rc = upload_norm(Lw.q_norm, w->q_norm[l], d, w->on_device)) ||
            (rc = upload_norm(Lw.k_norm, w->k_norm[l], d, w->on_device))) {
            free_ctx(ctx);
            return rc;
        }
        if (make_tmap_bf16(&Lw.tm_qkv, Lw.wqkv, D, ctx->qkv_dim, rowb, 64, 256) ||
            make_tmap_bf16(&Lw.tm_o, Lw.wo, ctx->attn_dim, D, (size_t)ctx->attn_dim * 2, 64, 128) ||
            make_tmap_bf16(&Lw.tm_gu, Lw.wgu, D, 2 * I, rowb, 64, 256) ||
            make_tmap_bf16(&Lw.tm_d, Lw.wd, I, D, (size_t)I * 2, 64, 128) ||
            make_tmap_bf16(&Lw.tm_o256, Lw.wo, ctx->attn_dim, D, (size_t)ctx->attn_dim * 2, 64, 256) ||
            make_tmap_bf16(&Lw.tm_d256, Lw.wd, I, D, (size_t)I * 2, 64, 256) ||
            make_tmap_bf16(&Lw.tm_qkv128, Lw.wqkv, D, ctx->qkv_dim, rowb, 64, 128) ||
            make_tmap_bf16(&Lw.tm_gu128, Lw.wgu, D, 2 * I, rowb, 64, 128) ||
            make_tmap_bf16(&Lw.tm_qkv32, Lw.wqkv, D, ctx->qkv_dim, rowb, 64, 32) ||
            make_tmap_bf16(&Lw.tm_gu64, Lw.wgu, D, 2 * I, rowb, 64, 64) ||
            make_tmap_bf16(&Lw.tm_o32, Lw.wo, ctx->attn_dim, D, (size_t)ctx->attn_dim * 2, 64, 32) ||
            make_tmap_bf16(&Lw.tm_d32, Lw.wd, I, D, (size_t)I * 2, 64, 32)) {
            free_ctx(ctx);
            return fail(QW_ECUDA, "cuTensorMapEncodeTiled failed for a weight");
        }
    }
    if (make_tmap_bf16(&ctx->tm_E, ctx->E, D, V, (size_t)D * 2, 64, 256)) {
        free_ctx(ctx);
        return fail(QW_ECUDA, "cuTensorMapEncodeTiled failed for the embedding");
    }

    // ---- weight-only int8: codes and scales per output channel; the bf16 matrices become the
    // dequantised weights, so every path (prefill, decode batches, the fused batch-1 kernel that
    // streams the codes) computes with the same model
    FusedWeights fw;
    if (c.weight_bits == 8) {
        size_t qoff = 0;
        auto qtake = [&](size_t bytes) {
            size_t o = qoff;
            qoff = align_up(qoff + bytes, A);
            return o;
        };
        struct QOffs { size_t qkv, o, gu, dn, sqkv, so, sgu, sd; };
        const size_t oEq = qtake((size_t)V * D), osE = qtake((size_t)V * 4);
        std::vector<QOffs> qo(c.n_layers);
        for (int l = 0; l < c.n_layers; ++l) {
            qo[l].qkv = qtake((size_t)ctx->qkv_dim * D);
            qo[l].o = qtake((size_t)D * ctx->attn_dim);
            qo[l].gu = qtake((size_t)2 * I * D);
            qo[l].dn = qtake((size_t)D * I);
            qo[l].sqkv = qtake((size_t)ctx->qkv_dim * 4);
            qo[l].so = qtake((size_t)D * 4);
            qo[l].sgu = qtake((size_t)2 * I * 4);
            qo[l].sd = qtake((size_t)D * 4);
        }
        if (cudaMalloc(&ctx->qbuf, qoff) != cudaSuccess) {
            free_ctx(ctx);
            return fail(QW_ENOMEM, "int8 weight allocation failed");
        }
        uint8_t* Q = ctx->qbuf;
        auto quant = [&](uint16_t* Wm, int rows, int cols, size_t oq, size_t os) {
            return launch_quantize_rows(Wm, rows, cols, cols, (int8_t*)(Q + oq), (float*)(Q + os), 0);
        };
        int qrc = quant(ctx->E, V, D, oEq, osE);
        fw.q8 = true;
        fw.Eq = (const int8_t*)(Q + oEq);
        fw.sE = (const float*)(Q + osE);
        for (int l = 0; l < c.n_layers && qrc == QW_OK; ++l) {
            LayerW& Lw = ctx->L[l];
            if ((qrc = quant(Lw.wqkv, ctx->qkv_dim, D, qo[l].qkv, qo[l].sqkv)) ||
                (qrc = quant(Lw.wo, D, ctx->attn_dim, qo[l].o, qo[l].so)) ||
                (qrc = quant(Lw.wgu, 2 * I, D, qo[l].gu, qo[l].sgu)) || (qrc = quant(Lw.wd, D, I, qo[l].dn, qo[l].sd)))
                break;
            fw.wqkv_q.push_back((const int8_t*)(Q + qo[l].qkv));
            fw.wo_q.push_back((const int8_t*)(Q + qo[l].o));
            fw.wgu_q.push_back((const int8_t*)(Q + qo[l].gu));
            fw.wd_q.push_back((const int8_t*)(Q + qo[l].dn));
            fw.s_qkv.push_back((const float*)(Q + qo[l].sqkv));
            fw.s_o.push_back((const float*)(Q + qo[l].so));
            fw.s_gu.push_back((const float*)(Q + qo[l].sgu));
            fw.s_d.push_back((const float*)(Q + qo[l].sd));
        }
        if (qrc != QW_OK) {
            free_ctx(ctx);
            return fail(qrc, "weight quantisation launch failed");
        }
    }

    // ---- workspaces
    const int T = std::max(c.max_tokens, c.max_batch);
    ctx->max_rows = T;
    const int TA = std::max(T, split_rows(SPLIT_MAX_M));   // rows of the bf16 activation buffers
    ctx->max_tiles = c.max_tokens / 64 + c.max_tokens + 1;
    off = 0;
    const size_t ox = take((size_t)T * D * 4);
    const size_t oqkv = take((size_t)T * ctx->qkv_dim * 4);
    const size_t oq = take((size_t)T * ctx->attn_dim * 4);
    const size_t oqb = take((size_t)T * ctx->attn_dim * 2);
    const size_t orope = take((size_t)T * 64 * 8);
    const size_t ogen = take((size_t)GEN_CHUNK * 4);
    const size_t ologits = take((size_t)c.max_batch * V * 4);
    ctx->n_part = (V + 255) / 256;
    const size_t otpart = take((size_t)c.max_batch * ctx->n_part * 8);
    const size_t opart = take((size_t)c.max_batch * Hq * ctx->max_splits * (d + 2) * 4);
    const size_t oh = take((size_t)TA * D * 2);
    const size_t oattn = take((size_t)TA * ctx->attn_dim * 2);
    const size_t oact = take((size_t)TA * I * 2);
    const size_t otok = take((size_t)T * 4);
    const size_t oiota = take((size_t)c.max_batch * 4);
    const size_t orows = take((size_t)T * 4);
    const size_t oerr = take(64);
    const size_t otiles = take((size_t)ctx->max_tiles * 16);
    const size_t ohid = c.debug_hidden ? take((size_t)c.n_layers * T * D * 4) : 0;
    if (cudaMalloc(&ctx->wsbuf, off) != cudaSuccess) {
        free_ctx(ctx);
        return fail(QW_ENOMEM, "workspace allocation failed");
    }
    uint8_t* W = ctx->wsbuf;
    ctx->x = (float*)(W + ox);
    ctx->qkv = (float*)(W + oqkv);
    ctx->q = (float*)(W + oq);
    ctx->q_bf16 = (uint16_t*)(W + oqb);
    ctx->rope_tab = (float2*)(W + orope);
    ctx->gen_pos = (int*)(W + ogen);
    ctx->logits = (float*)(W + ologits);
    ctx->tile_part = (float2*)(W + otpart);
    ctx->part = (float*)(W + opart);
    ctx->h = (uint16_t*)(W + oh);
    ctx->attn = (uint16_t*)(W + oattn);
    ctx->act = (uint16_t*)(W + oact);
    ctx->tok_seq = (int*)(W + otok);
    ctx->iota = (int*)(W + oiota);
    ctx->rows_last = (int*)(W + orows);
    ctx->err = (int*)(W + oerr);
    ctx->tiles = (int4*)(W + otiles);
    ctx->hidden = c.debug_hidden ? (float*)(W + ohid) : nullptr;
    {
        std::vector<int> iota(c.max_batch);
        for (int i = 0; i < c.max_batch; ++i) iota[i] = i;
        QW_INIT_CUDA(cudaMemcpy(ctx->iota, iota.data(), iota.size() * 4, cudaMemcpyHostToDevice));
        QW_INIT_CUDA(cudaMemset(ctx->err, 0, 64));
    }
    {
        fw.E = ctx->E;
        fw.final_norm = ctx->final_norm;
        fw.inv_freq = ctx->inv_freq;
        for (int l = 0; l < c.n_layers; ++l) {
            const LayerW& Lw = ctx->L[l];
            fw.wqkv.push_back(Lw.wqkv);
            fw.wo.push_back(Lw.wo);
            fw.wgu.push_back(Lw.wgu);
            fw.wd.push_back(Lw.wd);
            fw.in_norm.push_back(Lw.in_norm);
            fw.post_norm.push_back(Lw.post_norm);
            fw.q_norm.push_back(Lw.q_norm);
            fw.k_norm.push_back(Lw.k_norm);
        }
        ctx->fused = fused_create(fw, c.n_layers, V, c.rms_eps, D, Hq, Hkv, I);
        cudaGetLastError();  // a shape the fused kernel does not take is not an error
    }
    QW_INIT_CUDA(cudaDeviceSynchronize());
#undef QW_INIT_CUDA
    *out = ctx;
    return QW_OK;
}

int qw_destroy(qw_ctx* ctx) {
    if (!ctx) return fail(QW_EINVAL, "null context");
    cudaDeviceSynchronize();
    free_ctx(ctx);
    return QW_OK;
}

int qw_kv_create(qw_ctx* ctx, int32_t n_pages, qw_kv** out) {
    if (!ctx || !out || n_pages < 1) return fail(QW_EINVAL, "qw_kv_create: bad argument");
    *out = nullptr;
    const int64_t page_elems = (int64_t)2 * ctx->cfg.n_kv_heads * QW_PAGE_SIZE * QW_HEAD_DIM;
    const size_t bytes = (size_t)ctx->cfg.n_layers * n_pages * page_elems * 2;
    size_t free_b = 0, total_b = 0;
    QW_CUDA(cudaMemGetInfo(&free_b, &total_b));
    if (bytes + ((size_t)256 << 20) > free_b) return fail(QW_EKVFULL, "KV pool larger than free device memory");
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return fail(QW_ENOMEM, "KV pool allocation failed");
    // zeroed once: slots never written hold finite values, so masked keys contribute exactly 0
    if (cudaMemset(p, 0, bytes) != cudaSuccess) {
        cudaFree(p);
        return fail(QW_ECUDA, "KV pool clear failed");
    }
    qw_kv* kv = new qw_kv{ctx, (uint16_t*)p, n_pages, page_elems, (int64_t)n_pages * page_elems};
    *out = kv;
    return QW_OK;
}

int qw_kv_destroy(qw_kv* kv) {
    if (!kv) return fail(QW_EINVAL, "null kv");
    cudaDeviceSynchronize();
    cudaFree(kv->base);
    delete kv;
    return QW_OK;
}

int qw_kv_layout(const qw_kv* kv, void** base, int64_t* layer_stride, int64_t* page_stride, int32_t* n_pages) {
    if (!kv) return fail(QW_EINVAL, "null kv");
    if (base) *base = kv->base;
    if (layer_stride) *layer_stride = kv->layer_elems * 2;
    if (page_stride) *page_stride = kv->page_elems * 2;
    if (n_pages) *n_pages = kv->n_pages;
    return QW_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- the layer stack
// mode 0: prefill attention over `tiles`; mode 1: split-KV decode attention.
static int run_layers(qw_ctx* ctx, int n, const int* ids, const int* positions, const int* tok_seq, qw_kv* kv,
                      const int* bt, int bt_stride, int mode, int n_tiles, cudaStream_t st) {
    const qw_config& c = ctx->cfg;
    const int D = c.hidden, Hq = c.n_heads, Hkv = c.n_kv_heads, I = c.intermediate;
    const int split = n <= SPLIT_MAX_M;   // small-M projections take hi/lo activation pairs
    { QW_PROF(QW_PROF_OTHER); QW_TRY(launch_embed(ids, n, ctx->E, c.vocab, D, ctx->x, ctx->err, st), "embed launch"); }
    const bool fused_qkv = mode == 0 && ctx->prefill_attn == 0 && !split;  // q|k|v GEMM epilogue does Steps 4-5
    if (fused_qkv) { QW_PROF(QW_PROF_OTHER); QW_TRY(launch_rope_table(positions, n, ctx->inv_freq, ctx->rope_tab, st), "rope table launch"); }
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerW& Lw = ctx->L[l];
        KvView kvv{kv->base + (int64_t)l * kv->layer_elems, kv->page_elems, kv->n_pages, bt, bt_stride};
        { QW_PROF(QW_PROF_OTHER); QW_TRY(launch_rmsnorm_bf16(ctx->x, nullptr, n, D, Lw.in_norm, c.rms_eps, ctx->h, split, st),
               "rmsnorm launch"); }
        const bool tc_attn = mode == 0 && ctx->prefill_attn == 0;
        GemmEpilogue e{ctx->qkv, nullptr, ctx->qkv_dim, ctx->err, split};
        if (fused_qkv) {
            // prefill: QK-Norm, RoPE, bf16 q and the cache write happen in the GEMM epilogue
            e.rope = QkvRope{positions, tok_seq, kvv, Lw.q_norm, Lw.k_norm, ctx->rope_tab, c.rms_eps, ctx->q_bf16,
                             Hq, Hkv};
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->h, D, Lw.tm_qkv, 256, n, ctx->qkv_dim, D, EPI_QKV_ROPE, e, st, &Lw.tm_qkv128),
                   "qkv gemm"); }
        } else {
            // small M: 128-wide tiles (32 CTAs stream the weight for a 4096-wide q|k|v), measured
            // faster than split-K with atomic accumulation into a zeroed target
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->h, D, split ? Lw.tm_qkv32 : Lw.tm_qkv, split ? 32 : 256, n, ctx->qkv_dim, D,
                             EPI_STORE_F32, e, st),
                   "qkv gemm"); }
            { QW_PROF(QW_PROF_OTHER); QW_TRY(launch_qkv_post(ctx->qkv, n, positions, tok_seq, Hq, Hkv, Lw.q_norm, Lw.k_norm, ctx->inv_freq,
                                   c.rms_eps, tc_attn ? nullptr : ctx->q, tc_attn ? ctx->q_bf16 : nullptr, kvv,
                                   ctx->err, st),
                   "qk-norm/rope/kv-write launch"); }
        }
        if (tc_attn)
            { QW_PROF(QW_PROF_ATTN); QW_TRY(launch_attn_prefill_tc(ctx->q_bf16, n, positions, ctx->tiles, n_tiles, Hq, Hkv, kvv, ctx->attn,
                                          split, ctx->err, st),
                   "prefill attention launch"); }
        else if (mode == 0)
            { QW_PROF(QW_PROF_ATTN); QW_TRY(launch_attn_prefill(ctx->q, positions, ctx->tiles, n_tiles, Hq, Hkv, kvv, ctx->attn, split,
                                       ctx->err, st),
                   "prefill attention launch"); }
        else
            { QW_PROF(QW_PROF_ATTN); QW_TRY(launch_attn_decode(ctx->q, positions, n, Hq, Hkv, kvv, ctx->part, ctx->max_splits, ctx->attn,
                                      split, ctx->err, ctx->n_sm, st),
                   "decode attention launch"); }
        e = GemmEpilogue{ctx->x, nullptr, D, ctx->err, split};
        // N = hidden is narrow: 128-wide tiles give split-K decode batches more units,
        // 256-wide tiles halve the activation re-reads of a prefill
        if (split)
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->attn, ctx->attn_dim, Lw.tm_o32, 32, n, D, ctx->attn_dim, EPI_ADD_ATOMIC, e, st),
                   "o_proj gemm"); }
        else
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->attn, ctx->attn_dim, Lw.tm_o256, 256, n, D, ctx->attn_dim, EPI_RESID_ADD, e, st,
                             &Lw.tm_o),
                   "o_proj gemm"); }
        { QW_PROF(QW_PROF_OTHER); QW_TRY(launch_rmsnorm_bf16(ctx->x, nullptr, n, D, Lw.post_norm, c.rms_eps, ctx->h, split, st),
               "rmsnorm launch"); }
        if (split) {
            // small M: 128-wide tiles with the SwiGLU epilogue writing the hi/lo activation pairs
            e = GemmEpilogue{nullptr, ctx->act, I, ctx->err, split};
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->h, D, Lw.tm_gu64, 64, n, 2 * I, D, EPI_SWIGLU, e, st), "gate/up gemm"); }
        } else {
            e = GemmEpilogue{nullptr, ctx->act, I, ctx->err, split};
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->h, D, Lw.tm_gu, 256, n, 2 * I, D, EPI_SWIGLU, e, st, &Lw.tm_gu128), "gate/up gemm"); }
        }
        e = GemmEpilogue{ctx->x, nullptr, D, ctx->err, split};
        if (split)
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->act, I, Lw.tm_d32, 32, n, D, I, EPI_ADD_ATOMIC, e, st), "down gemm"); }
        else
            { QW_PROF(QW_PROF_GEMM); QW_TRY(gemm_bf16(ctx->act, I, Lw.tm_d256, 256, n, D, I, EPI_RESID_ADD, e, st, &Lw.tm_d), "down gemm"); }
        if (ctx->hidden)
            QW_CUDA(cudaMemcpyAsync(ctx->hidden + (size_t)l * ctx->max_rows * D, ctx->x, (size_t)n * D * 4,
                                    cudaMemcpyDeviceToDevice, st));
    }
    return QW_OK;
}

// final RMSNorm of the selected rows and the tied LM head (Step 8)
static int lm_head(qw_ctx* ctx, const int* rows, int n, float* out, cudaStream_t st) {
    const qw_config& c = ctx->cfg;
    const int split = n <= SPLIT_MAX_M;
    { QW_PROF(QW_PROF_LMHEAD); QW_TRY(launch_rmsnorm_bf16(ctx->x, rows, n, c.hidden, ctx->final_norm, c.rms_eps, ctx->h, split, st), "final norm"); }
    GemmEpilogue e{out, nullptr, c.vocab, ctx->err, split};
    if (out == ctx->logits && n <= c.max_batch) {   // the sampler's argmax and max start from these
        e.tile_max = ctx->tile_part;
        e.tile_ld = ctx->n_part;
    }
    { QW_PROF(QW_PROF_LMHEAD); QW_TRY(gemm_bf16(ctx->h, c.hidden, ctx->tm_E, 256, n, c.vocab, c.hidden, EPI_STORE_F32, e, st), "lm head gemm"); }
    ctx->part_rows = e.tile_max ? n : 0;
    return QW_OK;
}

extern "C" {

int qw_prefill(qw_ctx* ctx, const int32_t* ids, const int32_t* positions, const int32_t* cu, int32_t n_seqs,
               qw_kv* kv, const int32_t* bt, int32_t bt_stride, float* last_logits, void* stream) {
    if (!ctx || !ids || !positions || !cu || !kv || !bt) return fail(QW_EINVAL, "qw_prefill: null argument");
    if (kv->ctx != ctx) return fail(QW_EINVAL, "qw_prefill: kv pool belongs to another context");
    if (n_seqs < 1 || bt_stride < 1) return fail(QW_EINVAL, "qw_prefill: n_seqs and bt_stride must be >= 1");
    if (cu[0] != 0) return fail(QW_EINVAL, "qw_prefill: cu_seqlens[0] must be 0");
    for (int s = 0; s < n_seqs; ++s)
        if (cu[s + 1] <= cu[s]) return fail(QW_EINVAL, "qw_prefill: every sequence needs at least one token");
    const int n = cu[n_seqs];
    if (n > ctx->cfg.max_tokens) return fail(QW_EINVAL, "qw_prefill: more tokens than max_tokens");
    if (!last_logits && n_seqs > ctx->cfg.max_batch)
        return fail(QW_EINVAL, "qw_prefill: more than max_batch sequences need a caller logits buffer");
    cudaStream_t st = (cudaStream_t)stream;
    std::vector<int> tok_seq(n), last(n_seqs);
    std::vector<int4> tiles;
    // query tiles: 128 / G positions (G query heads per KV head fill the 128 MMA rows of the
    // tcgen05 kernel); the mma.sync comparison kernel takes 64 positions of two heads
    const int tile = ctx->prefill_attn == 0 ? 128 / (ctx->cfg.n_heads / ctx->cfg.n_kv_heads) : 64;
    for (int s = 0; s < n_seqs; ++s) {
        const int len = cu[s + 1] - cu[s];
        for (int t = cu[s]; t < cu[s + 1]; ++t) tok_seq[t] = s;
        last[s] = cu[s + 1] - 1;
        for (int q0 = 0; q0 < len; q0 += tile) tiles.push_back(make_int4(s, cu[s] + q0, std::min(tile, len - q0), q0));
    }
    // longest causal rows first, so the heaviest tiles start in the first wave
    std::stable_sort(tiles.begin(), tiles.end(), [](const int4& a, const int4& b) { return a.w > b.w; });
    if ((int)tiles.size() > ctx->max_tiles) return fail(QW_EINVAL, "qw_prefill: too many query tiles");
    QW_CUDA(cudaMemcpyAsync(ctx->tok_seq, tok_seq.data(), n * 4, cudaMemcpyHostToDevice, st));
    QW_CUDA(cudaMemcpyAsync(ctx->rows_last, last.data(), n_seqs * 4, cudaMemcpyHostToDevice, st));
    QW_CUDA(cudaMemcpyAsync(ctx->tiles, tiles.data(), tiles.size() * 16, cudaMemcpyHostToDevice, st));
    int rc = run_layers(ctx, n, ids, positions, ctx->tok_seq, kv, bt, bt_stride, 0, (int)tiles.size(), st);
    if (rc) return rc;
    ctx->last_rows = n;
    ctx->last_fused = false;
    float* out = last_logits ? last_logits : ctx->logits;
    if ((rc = lm_head(ctx, ctx->rows_last, n_seqs, out, st))) return rc;
    ctx->logits_rows = last_logits ? 0 : n_seqs;
    return QW_OK;
}

int qw_decode_step(qw_ctx* ctx, const int32_t* tokens, const int32_t* positions, int32_t batch, qw_kv* kv,
                   const int32_t* bt, int32_t bt_stride, float* logits, void* stream) {
    if (!ctx || !tokens || !positions || !kv || !bt) return fail(QW_EINVAL, "qw_decode_step: null argument");
    if (kv->ctx != ctx) return fail(QW_EINVAL, "qw_decode_step: kv pool belongs to another context");
    if (batch < 1 || batch > ctx->cfg.max_batch) return fail(QW_EINVAL, "qw_decode_step: batch out of [1, max_batch]");
    if (bt_stride < 1) return fail(QW_EINVAL, "qw_decode_step: bt_stride must be >= 1");
    cudaStream_t st = (cudaStream_t)stream;
    float* out = logits ? logits : ctx->logits;
    // automatic choice: the fused kernel for batch 1, unless per-layer residuals are kept for checking
    const bool fused = fused_supported(ctx->fused, batch, bt_stride) &&
                       (ctx->decode_path == 2 || (ctx->decode_path == 0 && !ctx->hidden));
    if (ctx->decode_path == 2 && !fused)
        return fail(QW_EINVAL, "qw_decode_step: the fused path takes batch 1 and block tables of at most 4088 pages");
    int rc;
    ctx->last_fused = fused;
    if (fused) {
        QW_PROF(QW_PROF_FUSED);
        ctx->part_rows = 0;
        rc = fused_decode(ctx->fused, tokens, positions, batch, kv->base, kv->layer_elems, kv->page_elems,
                          kv->n_pages, bt, bt_stride, out, ctx->err, st);
        if (rc) return fail(rc, "fused decode launch failed");
        ctx->last_rows = batch;
    } else {
        if ((rc = run_layers(ctx, batch, tokens, positions, ctx->iota, kv, bt, bt_stride, 1, 0, st))) return rc;
        ctx->last_rows = batch;
        if ((rc = lm_head(ctx, nullptr, batch, out, st))) return rc;
    }
    ctx->logits_rows = logits ? 0 : batch;
    return QW_OK;
}

int qw_sample(qw_ctx* ctx, const float* logits, int32_t batch, const qw_sample_params* params, uint64_t rng_counter,
              int32_t* out_ids, void* stream) {
    if (!ctx || !params || !out_ids) return fail(QW_EINVAL, "qw_sample: null argument");
    if (batch < 1 || batch > ctx->cfg.max_batch) return fail(QW_EINVAL, "qw_sample: batch out of [1, max_batch]");
    if (!logits) {
        if (ctx->logits_rows < batch) return fail(QW_EINVAL, "qw_sample: the context holds fewer logits rows than batch");
        logits = ctx->logits;
    }
    const bool own = logits == ctx->logits;   // the context's logits of the last call
    const int* hint = (own && ctx->last_fused && batch == 1) ? fused_argmax(ctx->fused) : nullptr;
    const float2* part = (own && ctx->part_rows >= batch) ? ctx->tile_part : nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    QW_PROF(QW_PROF_SAMPLE);
    QW_TRY(launch_sample(logits, batch, ctx->cfg.vocab, params, rng_counter, out_ids, part, ctx->n_part, hint,
                         ctx->err, (cudaStream_t)stream),
           "sample launch");
    return QW_OK;
}

int qw_generate(qw_ctx* ctx, qw_kv* kv, const int32_t* bt, int32_t bt_stride, const int32_t* first_token,
                int32_t start_pos, int32_t n_steps, const qw_sample_params* params, uint64_t rng_counter,
                int32_t* out_ids, void* stream) {
    if (!ctx || !kv || !bt || !first_token || !params || !out_ids) return fail(QW_EINVAL, "qw_generate: null argument");
    if (n_steps < 1 || start_pos < 0 || bt_stride < 1 ||
        (int64_t)start_pos + n_steps > (int64_t)bt_stride * QW_PAGE_SIZE)
        return fail(QW_EINVAL, "qw_generate: n_steps < 1, start_pos < 0 or positions beyond the block table");
    cudaStream_t st = (cudaStream_t)stream;
    for (int32_t i = 0; i < n_steps; ++i) {
        if (i % GEN_CHUNK == 0)  // positions of the next chunk (stream-ordered after the previous steps)
            QW_TRY(launch_positions(ctx->gen_pos, start_pos + i, std::min<int32_t>(GEN_CHUNK, n_steps - i), st),
                   "positions launch");
        const int32_t* tok = i == 0 ? first_token : out_ids + i - 1;
        int rc = qw_decode_step(ctx, tok, ctx->gen_pos + i % GEN_CHUNK, 1, kv, bt, bt_stride, nullptr, stream);
        if (rc) return rc;
        rc = qw_sample(ctx, nullptr, 1, params, rng_counter + (uint64_t)i, out_ids + i, stream);
        if (rc) return rc;
    }
    return QW_OK;
}

int qw_attn_decode(qw_ctx* ctx, const float* q, const int32_t* positions, int32_t batch, qw_kv* kv, int32_t layer,
                   const int32_t* bt, int32_t bt_stride, uint16_t* out, void* stream) {
    if (!ctx || !q || !positions || !kv || !bt || !out) return fail(QW_EINVAL, "qw_attn_decode: null argument");
    if (kv->ctx != ctx) return fail(QW_EINVAL, "qw_attn_decode: kv pool belongs to another context");
    if (batch < 1 || batch > ctx->cfg.max_batch || layer < 0 || layer >= ctx->cfg.n_layers || bt_stride < 1)
        return fail(QW_EINVAL, "qw_attn_decode: batch, layer or bt_stride out of range");
    KvView kvv{kv->base + (int64_t)layer * kv->layer_elems, kv->page_elems, kv->n_pages, bt, bt_stride};
    QW_TRY(launch_attn_decode(q, positions, batch, ctx->cfg.n_heads, ctx->cfg.n_kv_heads, kvv, ctx->part,
                              ctx->max_splits, out, 0, ctx->err, ctx->n_sm, (cudaStream_t)stream),
           "decode attention launch");
    return QW_OK;
}

int qw_check(qw_ctx* ctx, void* stream) {
    if (!ctx) return fail(QW_EINVAL, "null context");
    QW_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    int h = 0;
    QW_CUDA(cudaMemcpy(&h, ctx->err, 4, cudaMemcpyDeviceToHost));
    if (h) {
        QW_CUDA(cudaMemset(ctx->err, 0, 4));
        if (ctx->fused) {
            fused_reset(ctx->fused, (cudaStream_t)stream);
            QW_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
        }
        return fail(h, h == QW_ERANGE ? "device: token id, position or page id out of range"
                       : h == QW_ETIMEOUT ? "device: a bounded wait timed out"
                                          : "device: invalid sampling parameters or too many tied logits");
    }
    return QW_OK;
}

int qw_debug_hidden(qw_ctx* ctx, int32_t layer, float* out, int32_t n_rows, void* stream) {
    if (!ctx || !out) return fail(QW_EINVAL, "null argument");
    if (!ctx->hidden) return fail(QW_EINVAL, "context was created without debug_hidden");
    if (layer < 0 || layer >= ctx->cfg.n_layers) return fail(QW_EINVAL, "layer out of range");
    if (n_rows < 1 || n_rows > ctx->last_rows) return fail(QW_EINVAL, "n_rows exceeds the rows of the last call");
    if (ctx->last_fused) return fail(QW_EINVAL, "the fused decode path keeps no per-layer residuals");
    QW_CUDA(cudaMemcpyAsync(out, ctx->hidden + (size_t)layer * ctx->max_rows * ctx->cfg.hidden,
                            (size_t)n_rows * ctx->cfg.hidden * 4, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    return QW_OK;
}

int qw_debug_gemm(const uint16_t* A, const uint16_t* B, void* C, int32_t M, int32_t N, int32_t K, int32_t epi,
                  int32_t bn, int32_t split, void* stream) {
    if (!A || !B || !C || M < 1 || N < 32 || K < 64 || K % 64 || N % 32 || epi < 0 || epi > 3 ||
        (bn != 128 && bn != 256 && !(split == 1 && (bn == 32 || bn == 64))))
        return fail(QW_EINVAL, "qw_debug_gemm: bad argument");
    if (split < 0 || split > 2) return fail(QW_EINVAL, "qw_debug_gemm: bad split");
    CUtensorMap tb, tb_half;
    QW_TRY(make_tmap_bf16(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64, (uint32_t)bn), "tensor map for B");
    QW_TRY(make_tmap_bf16(&tb_half, B, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64, 128), "tensor map for B");
    GemmEpilogue e{epi == 2 ? nullptr : (float*)C, epi == 2 ? (uint16_t*)C : nullptr, epi == 2 ? N / 2 : N, nullptr,
                   split == 1 ? 1 : 0};
    QW_TRY(gemm_bf16(A, K, tb, bn, M, N, K, epi, e, (cudaStream_t)stream, split == 2 ? &tb_half : nullptr),
           "gemm launch");
    return QW_OK;
}

int qw_debug_trace(qw_ctx* ctx, int32_t enable, uint64_t* host_out, int64_t n, int64_t* n_needed) {
    if (!ctx) return fail(QW_EINVAL, "null context");
    if (!ctx->fused) return fail(QW_EINVAL, "no fused decode kernel in this context");
    QW_TRY(fused_trace(ctx->fused, enable, host_out, n, n_needed), "trace copy failed");
    return QW_OK;
}

int qw_debug_profile(qw_ctx* ctx, int32_t enable, double* ms_out, int64_t* count_out) {
    if (!ctx) return fail(QW_EINVAL, "null context");
    Profiler& p = ctx->prof;
    if (ms_out || count_out) {
        QW_CUDA(cudaDeviceSynchronize());
        for (int k = 0; k < QW_PROF_CLASSES; ++k) {
            if (ms_out) ms_out[k] = 0.0;
            if (count_out) count_out[k] = 0;
        }
        for (size_t i = 0; i < p.used; ++i) {
            float ms = 0.f;
            QW_CUDA(cudaEventElapsedTime(&ms, p.ev[2 * i], p.ev[2 * i + 1]));
            if (ms_out) ms_out[p.cls[i]] += ms;
            if (count_out) count_out[p.cls[i]] += 1;
        }
    }
    if (enable) p.used = 0;
    p.on = enable != 0;
    return QW_OK;
}

int qw_debug_inject_timeout(qw_ctx* ctx) {
    if (!ctx) return fail(QW_EINVAL, "null context");
    if (!ctx->fused) return fail(QW_EINVAL, "no fused decode kernel in this context");
    return fused_inject_timeout(ctx->fused);
}

int qw_set_prefill_attention(qw_ctx* ctx, int32_t variant) {
    if (!ctx || variant < 0 || variant > 1) return fail(QW_EINVAL, "qw_set_prefill_attention: bad argument");
    ctx->prefill_attn = variant;
    return QW_OK;
}

uint64_t qw_kernel_launches(void) { return (uint64_t)launches_so_far(); }

int qw_set_decode_path(qw_ctx* ctx, int32_t path) {
    if (!ctx || path < 0 || path > 2) return fail(QW_EINVAL, "qw_set_decode_path: bad argument");
    if (path == 2 && !ctx->fused) return fail(QW_EINVAL, "the fused decode path is not available for this configuration");
    ctx->decode_path = path;
    return QW_OK;
}

}  // extern "C"
