/*
 * Plain single-precision CPU oracle of the Qwen3-0.6B decoder forward pass, KV cache,
 * sampler and generation loop.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU baseline
 * call it; the product path never does.  It shares no code with the CUDA library.
 *
 * Source: "Inside an LLM: Pure Python Inference for Qwen3-0.6B on MLX" (English page),
 * Steps 2-9; each function names the step it restates.  The article's script is not
 * reproduced: this is the definition written out with plain loops.
 *
 * Precision: every stored value is a float (activations, cache, logits); bf16 weights are
 * widened exactly on use; every dot product, norm sum and softmax sum accumulates in
 * double and is rounded to float once.  RoPE keeps the article's float32 inverse
 * frequencies and angles: inv_freq_i = float(theta^(-i/half)) evaluated in double,
 * angle = float(float(pos) * inv_freq_i); cos and sin are taken in double of that angle.
 *
 * Readings of points the article leaves open (the same as the numpy oracle's):
 *   - forward(ids, cache, pos) is never shown: embedding (Step 2) -> blocks (Step 7) ->
 *     final RMSNorm and tied LM head (Step 8).
 *   - the causal mask (Step 5) is "key at position j visible to a query at position p iff
 *     j <= p"; masked keys are skipped.
 *   - sample() (Step 8): top-k caps the top-p cutoff; ties in the sort go to the lower id;
 *     the categorical draw is inverse CDF on the kept, renormalised list.
 *   - the draw u of a row comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) with
 *     key = 64-bit seed and counter = (rng_counter, 0, 0): u = (word0 >> 8) * 2^-24.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define QWO_MAX_HEAD_DIM 512

typedef struct qwo_model {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab;
    float eps;
    double theta;
    const uint16_t* embed;        /* [vocab][hidden]; also the tied LM head */
    const uint16_t* final_norm;   /* [hidden] */
    /* per layer: arrays of n_layers pointers, checkpoint layout [out][in] */
    const uint16_t* const* in_norm;
    const uint16_t* const* wq;
    const uint16_t* const* wk;
    const uint16_t* const* wv;
    const uint16_t* const* q_norm;
    const uint16_t* const* k_norm;
    const uint16_t* const* wo;
    const uint16_t* const* post_norm;
    const uint16_t* const* wg;
    const uint16_t* const* wu;
    const uint16_t* const* wd;
} qwo_model;

/* Cache of one sequence (Step 5, "The KV cache"): post-RoPE keys and values of every layer.
 * k, v: float [n_layers][n_kv_heads][cap][head_dim]; pos: int [cap] position of entry i;
 * len: entries filled.  Allocated by the caller. */
typedef struct qwo_cache {
    int32_t cap, len;
    float* k;
    float* v;
    int32_t* pos;
} qwo_cache;

static float bf(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Step 3: y = x / sqrt(mean(x^2) + eps) * w over n entries. */
void qwo_rms_norm(const float* x, const uint16_t* w, int n, float eps, float* y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
    const double s = 1.0 / sqrt(ss / n + (double)eps);
    for (int i = 0; i < n; ++i) y[i] = (float)((double)x[i] * s * (double)bf(w[i]));
}

/* y[t][r] = sum_c W[r][c] x[t][c] for T rows x[T][cols] and a bf16 matrix W [rows][cols]. */
static void mat_mul(const uint16_t* W, const float* x, int T, int rows, int cols, float* y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t* wr = W + (size_t)r * cols;
        for (int t = 0; t < T; ++t) {
            const float* xt = x + (size_t)t * cols;
            double acc = 0.0;
            for (int c = 0; c < cols; ++c) acc += (double)bf(wr[c]) * (double)xt[c];
            y[(size_t)t * rows + r] = (float)acc;
        }
    }
}

/* Step 4: half-split rotation of one head vector x[d] at position pos. */
void qwo_rope(float* x, int d, int32_t pos, double theta) {
    const int half = d / 2;
    for (int i = 0; i < half; ++i) {
        const float inv = (float)(1.0 / pow(theta, (double)i / (double)half));
        const float ang = (float)pos * inv;   /* float32 product, rounded once */
        const double c = cos((double)ang), s = sin((double)ang);
        const double a = x[i], b = x[i + half];
        x[i] = (float)(a * c - b * s);
        x[i + half] = (float)(a * s + b * c);
    }
}

/* Step 6: SiLU(g) = g * sigmoid(g). */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Step 5 core for one query head: softmax(q . K^T / sqrt(d)) V over the cached entries whose
 * position is <= qpos.  k, v: [cap][d] of the head's KV head. */
static void attend(const float* q, const float* k, const float* v, const int32_t* pos, int len, int d, int32_t qpos,
                   double* scores, float* out) {
    const double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int j = 0; j < len; ++j) {
        if (pos[j] > qpos) {
            scores[j] = -INFINITY;
            continue;
        }
        double s = 0.0;
        const float* kj = k + (size_t)j * d;
        for (int e = 0; e < d; ++e) s += (double)q[e] * (double)kj[e];
        scores[j] = s * scale;
        if (scores[j] > mx) mx = scores[j];
    }
    double z = 0.0;
    for (int j = 0; j < len; ++j) {
        scores[j] = pos[j] > qpos ? 0.0 : exp(scores[j] - mx);
        z += scores[j];
    }
    double acc[QWO_MAX_HEAD_DIM];
    for (int e = 0; e < d; ++e) acc[e] = 0.0;
    for (int j = 0; j < len; ++j) {   /* o = sum_j p_j v_j, one value row at a time */
        if (scores[j] == 0.0) continue;
        const float* vj = v + (size_t)j * d;
        for (int e = 0; e < d; ++e) acc[e] += scores[j] * (double)vj[e];
    }
    for (int e = 0; e < d; ++e) out[e] = (float)(acc[e] / z);
}

/* Step 5: attention of one layer for T new tokens h[T][hidden] at positions pos[T]; appends
 * their keys and values to the cache at entries c->len .. c->len + T - 1 and returns
 * out[T][hidden] = o_proj(concat of heads).  The caller advances c->len after all layers. */
static int attention(const qwo_model* m, int l, const float* h, const int32_t* pos, int T, qwo_cache* c,
                     float* out) {
    const int D = m->hidden, Hq = m->n_heads, Hkv = m->n_kv_heads, d = m->head_dim;
    const int group = Hq / Hkv;
    if (c->len + T > c->cap) return -1;
    float* q = malloc(sizeof(float) * (size_t)T * Hq * d);
    float* kk = malloc(sizeof(float) * (size_t)T * Hkv * d);
    float* vv = malloc(sizeof(float) * (size_t)T * Hkv * d);
    float* o = malloc(sizeof(float) * (size_t)T * Hq * d);
    if (!q || !kk || !vv || !o) {
        free(q), free(kk), free(vv), free(o);
        return -2;
    }
    float* Kl = c->k + (size_t)l * Hkv * c->cap * d;
    float* Vl = c->v + (size_t)l * Hkv * c->cap * d;
    mat_mul(m->wq[l], h, T, Hq * d, D, q);
    mat_mul(m->wk[l], h, T, Hkv * d, D, kk);
    mat_mul(m->wv[l], h, T, Hkv * d, D, vv);
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < Hq; ++j) {   /* QK-Norm over each head, then RoPE */
            float* qj = q + ((size_t)t * Hq + j) * d;
            qwo_rms_norm(qj, m->q_norm[l], d, m->eps, qj);
            qwo_rope(qj, d, pos[t], m->theta);
        }
        for (int g = 0; g < Hkv; ++g) {
            float* kg = kk + ((size_t)t * Hkv + g) * d;
            qwo_rms_norm(kg, m->k_norm[l], d, m->eps, kg);
            qwo_rope(kg, d, pos[t], m->theta);
            memcpy(Kl + ((size_t)g * c->cap + c->len + t) * d, kg, sizeof(float) * d);
            memcpy(Vl + ((size_t)g * c->cap + c->len + t) * d, vv + ((size_t)t * Hkv + g) * d, sizeof(float) * d);
        }
        c->pos[c->len + t] = pos[t];
    }
    const int len = c->len + T;
    int fail = 0;
#pragma omp parallel
    {
        double* scores = malloc(sizeof(double) * (size_t)len);
        if (!scores) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for collapse(2) schedule(dynamic)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < Hq; ++j) {   /* query head j reads KV head j / group (Step 5, GQA) */
                if (!scores) continue;
                const int g = j / group;
                attend(q + ((size_t)t * Hq + j) * d, Kl + (size_t)g * c->cap * d, Vl + (size_t)g * c->cap * d,
                       c->pos, len, d, pos[t], scores, o + ((size_t)t * Hq + j) * d);
            }
        free(scores);
    }
    if (!fail) mat_mul(m->wo[l], o, T, D, Hq * d, out);
    free(q), free(kk), free(vv), free(o);
    return fail ? -2 : 0;
}

/* Step 6: out = (silu(h Wg^T) * h Wu^T) Wd^T for T rows h[T][hidden]. */
static int ffn(const qwo_model* m, int l, const float* h, int T, float* out) {
    const int D = m->hidden, I = m->intermediate;
    float* g = malloc(sizeof(float) * (size_t)T * I);
    float* u = malloc(sizeof(float) * (size_t)T * I);
    if (!g || !u) {
        free(g), free(u);
        return -2;
    }
    mat_mul(m->wg[l], h, T, I, D, g);
    mat_mul(m->wu[l], h, T, I, D, u);
    for (size_t i = 0; i < (size_t)T * I; ++i) g[i] = (float)(silu((double)g[i]) * (double)u[i]);
    mat_mul(m->wd[l], g, T, D, I, out);
    free(g), free(u);
    return 0;
}

/* Steps 2, 7 and 8: logits of one sequence's T tokens (ids at positions pos) given its cache.
 *   logits   float [T][vocab], or [1][vocab] with last_only (nullable: no LM head)
 *   hiddens  nullable float [n_layers][T][hidden]: the residual stream after each block
 * Returns 0, -1 if the cache has no room, -2 if memory ran out, -3 for a bad token id, -4 for a
 * head_dim above QWO_MAX_HEAD_DIM. */
int qwo_forward(const qwo_model* m, const int32_t* ids, const int32_t* pos, int T, qwo_cache* c, int last_only,
                float* logits, float* hiddens) {
    const int D = m->hidden;
    if (m->head_dim > QWO_MAX_HEAD_DIM) return -4;
    for (int t = 0; t < T; ++t)
        if (ids[t] < 0 || ids[t] >= m->vocab) return -3;
    float* x = malloc(sizeof(float) * (size_t)T * D);
    float* h = malloc(sizeof(float) * (size_t)T * D);
    float* a = malloc(sizeof(float) * (size_t)T * D);
    if (!x || !h || !a) {
        free(x), free(h), free(a);
        return -2;
    }
    for (int t = 0; t < T; ++t)   /* Step 2: embedding rows */
        for (int i = 0; i < D; ++i) x[(size_t)t * D + i] = bf(m->embed[(size_t)ids[t] * D + i]);
    int rc = 0;
    for (int l = 0; l < m->n_layers && !rc; ++l) {   /* Step 7: pre-norm block with residuals */
        for (int t = 0; t < T; ++t) qwo_rms_norm(x + (size_t)t * D, m->in_norm[l], D, m->eps, h + (size_t)t * D);
        rc = attention(m, l, h, pos, T, c, a);
        if (rc) break;
        for (size_t i = 0; i < (size_t)T * D; ++i) x[i] += a[i];
        for (int t = 0; t < T; ++t) qwo_rms_norm(x + (size_t)t * D, m->post_norm[l], D, m->eps, h + (size_t)t * D);
        rc = ffn(m, l, h, T, a);
        if (rc) break;
        for (size_t i = 0; i < (size_t)T * D; ++i) x[i] += a[i];
        if (hiddens) memcpy(hiddens + (size_t)l * T * D, x, sizeof(float) * (size_t)T * D);
    }
    if (!rc) {
        c->len += T;
        if (logits) {   /* Step 8: final norm and the LM head tied to the embedding */
            const int t0 = last_only ? T - 1 : 0;
            for (int t = t0; t < T; ++t) {
                qwo_rms_norm(x + (size_t)t * D, m->final_norm, D, m->eps, h);
                mat_mul(m->embed, h, 1, m->vocab, D, logits + (size_t)(t - t0) * m->vocab);
            }
        }
    }
    free(x), free(h), free(a);
    return rc;
}

/* ---------------------------------------------------------------- Step 8: sampling */
typedef struct qwo_sample_info {
    int32_t id;
    int32_t cutoff;             /* kept entries (0 for greedy) */
    double cum_at_cutoff;       /* cumulative probability of the kept list */
    double cum_before_cutoff;   /* ... without its last entry */
    double draw_gap;            /* distance of u to the nearest cumulative kept boundary */
} qwo_sample_info;

static const float* g_sort_p;   /* qsort has no context argument: probabilities of the current row */
static int by_prob_then_id(const void* a, const void* b) {
    const int i = *(const int*)a, j = *(const int*)b;
    if (g_sort_p[i] != g_sort_p[j]) return g_sort_p[i] > g_sort_p[j] ? -1 : 1;
    return i < j ? -1 : (i > j);
}

/* sample() of Step 8 with a top-k cap (top_k <= 0: none) and the uniform draw u in [0, 1).
 * Greedy (lowest id on ties) when temperature == 0.  Otherwise p = softmax(logits / T) over
 * the whole vocabulary, sorted descending (ties: lower id first), cutoff =
 * #(cumsum < top_p) + 1 capped at top_k, the kept probabilities renormalised, and the first
 * kept j whose cumulative kept mass exceeds u is returned.  Not thread-safe. */
int qwo_sample(const float* logits, int V, float temperature, int top_k, float top_p, double u,
               qwo_sample_info* info) {
    qwo_sample_info tmp;
    if (!info) info = &tmp;
    memset(info, 0, sizeof(*info));
    int best = 0;
    for (int i = 1; i < V; ++i)
        if (logits[i] > logits[best]) best = i;
    if (temperature == 0.f) {
        info->id = best;
        return best;
    }
    float* p = malloc(sizeof(float) * V);
    int* order = malloc(sizeof(int) * V);
    if (!p || !order) {
        free(p), free(order);
        return -2;
    }
    const double mx = (double)logits[best] / temperature;
    double z = 0.0;
    for (int i = 0; i < V; ++i) z += exp((double)logits[i] / temperature - mx);
    for (int i = 0; i < V; ++i) {
        p[i] = (float)(exp((double)logits[i] / temperature - mx) / z);
        order[i] = i;
    }
    g_sort_p = p;
    qsort(order, V, sizeof(int), by_prob_then_id);
    int cutoff = 0;
    double cum = 0.0, prev = 0.0;
    for (int i = 0; i < V; ++i) {   /* #(cumsum < top_p) + 1 */
        prev = cum;
        cum += p[order[i]];
        ++cutoff;
        if (!(cum < (double)top_p)) break;
    }
    if (top_k > 0 && cutoff > top_k) cutoff = top_k;
    cum = prev = 0.0;
    for (int i = 0; i < cutoff; ++i) {
        prev = cum;
        cum += p[order[i]];
    }
    info->cutoff = cutoff;
    info->cum_at_cutoff = cum;
    info->cum_before_cutoff = prev;
    /* first kept j with cumulative kept mass > u (the last one when rounding leaves it below u) */
    double ck = 0.0, gap = INFINITY;
    int j = -1;
    for (int i = 0; i < cutoff; ++i) {
        ck += p[order[i]] / cum;
        if (fabs(ck - u) < gap) gap = fabs(ck - u);
        if (j < 0 && ck > u) j = i;
    }
    if (j < 0) j = cutoff - 1;
    info->draw_gap = gap;
    info->id = order[j];
    free(p), free(order);
    return info->id;
}

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11): ten rounds on a 4-word counter with a 2-word key bumped by the Weyl constants. */
void qwo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c0 = n0;
        c1 = (uint32_t)p1;
        c2 = n2;
        c3 = (uint32_t)p0;
    }
    out[0] = c0, out[1] = c1, out[2] = c2, out[3] = c3;
}

/* The draw of one row at one step: key = seed, counter = (rng_counter, 0, 0). */
double qwo_sampling_uniform(uint64_t seed, uint64_t rng_counter) {
    const uint32_t ctr[4] = {(uint32_t)rng_counter, (uint32_t)(rng_counter >> 32), 0, 0};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    qwo_philox4x32_10(ctr, key, r);
    return (double)(r[0] >> 8) * (1.0 / 16777216.0);
}

/* Step 9: prefill the prompt at positions 0 .. T-1, sample, then decode each chosen token at
 * the next position, n_steps ids in all (no EOS).  Step i draws with rng_counter = i.
 *   cache   empty, cap >= T + n_steps - 1
 *   out_ids int [n_steps]; rows nullable float [n_steps][vocab]: the logits of each step */
int qwo_generate(const qwo_model* m, const int32_t* prompt, int T, int n_steps, float temperature, int top_k,
                 float top_p, uint64_t seed, qwo_cache* c, int32_t* out_ids, float* rows) {
    float* logits = malloc(sizeof(float) * m->vocab);
    int32_t* pos = malloc(sizeof(int32_t) * (T > 1 ? T : 1));
    if (!logits || !pos) {
        free(logits), free(pos);
        return -2;
    }
    for (int t = 0; t < T; ++t) pos[t] = t;
    int rc = qwo_forward(m, prompt, pos, T, c, 1, logits, NULL);
    for (int i = 0; i < n_steps && !rc; ++i) {
        if (i > 0) {
            const int32_t p = T + i - 1;
            rc = qwo_forward(m, &out_ids[i - 1], &p, 1, c, 1, logits, NULL);
            if (rc) break;
        }
        if (rows) memcpy(rows + (size_t)i * m->vocab, logits, sizeof(float) * m->vocab);
        const int id = qwo_sample(logits, m->vocab, temperature, top_k, top_p, qwo_sampling_uniform(seed, i), NULL);
        if (id < 0) rc = id;
        out_ids[i] = id;
    }
    free(logits), free(pos);
    return rc;
}

/* Threads the parallel loops use (OpenMP), for reporting. */
int qwo_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
