// Fused persistent decode for one sequence (batch 1): one cooperative launch per
// step runs the article's whole forward pass (Steps 2-8) for the new token.
//
// Every CTA (one per SM) owns fixed slices of every weight matrix.  Warp 0 streams
// those slices -- q|k|v rows, the transposed o_proj rows, gate/up row pairs, the
// transposed down_proj rows of all layers, then the tied LM-head rows -- through a
// shared-memory ring with cp.async.bulk, in the order the consumers use them and
// independent of any data dependency, so HBM keeps streaming while the consumers
// wait.  Warps 1..8 consume the ring:
//
//   P1  x -> RMSNorm -> q|k|v rows (dot products)          -> raw q|k|v in global
//   P2  attention split (KV head g, part s of the cache)   -> partial (m, l, o)
//   P3  merge the splits of the CTA's attention dims, o_proj as a sum of scaled rows
//       of Wo^T (one row per attention dim)                -> atomic adds into oacc
//   P4  x + oacc -> RMSNorm -> gate/up pairs -> SwiGLU -> down_proj as scaled rows of
//       Wd^T                                                -> atomic adds into dacc
//   LM  x + oacc + dacc -> final RMSNorm -> LM-head rows -> logits, argmax
//
// Phases meet through monotonically increasing counters in global memory (one
// launch adds a known amount, so the targets are epoch * amount); every wait is
// bounded by %globaltimer and ends in QW_ETIMEOUT instead of a hang.  The residual
// stream stays in fp32: R (materialised once per layer), oacc and dacc are
// double-buffered by layer parity and zeroed by their owner CTA once no reader can
// be left.
#include <cooperative_groups.h>

#include <vector>

#include "qw_common.cuh"
#include "qw_fused.h"
#include "qw_internal.h"

namespace qw {
namespace fused {

constexpr int D = 1024, HQ = 16, HKV = 8, HD = 128, INTER = 3072, QKVR = 4096, AD = 2048;
constexpr int NS = 6;                 // ring stages
constexpr int STAGE = 32768;          // bytes per stage
constexpr int ROW_B = D * 2;          // every streamed row is 1024 bf16
constexpr int ROWS_PER_STAGE = STAGE / ROW_B;   // 16
constexpr int PAGE_B = QW_PAGE_SIZE * HD * 2;   // K (or V) of one head in one page: 4 KB
constexpr int PAGES_PER_STAGE = STAGE / (2 * PAGE_B);  // 4
constexpr int NCW = 8;                // consumer warps
constexpr int THREADS = 32 * (NCW + 1);
constexpr int CNT_STRIDE = 32;        // counters 128 bytes apart
constexpr int PART = HD + 2;
constexpr int MAX_ROWS = 64;          // per-phase result slots (q|k|v rows per CTA <= 4096/G + 1)
constexpr int MAX_LAYERS = 64;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int TRACE_SLOTS = QW_TRACE_SLOTS;
constexpr int NSH = 8;   // accumulator shards: CTA c adds into shard c % NSH (fewer adds per address)

struct LayerPtrs {
    const uint16_t *wqkv, *woT, *wgu, *wdT;
    const float *in_norm, *post_norm, *q_norm, *k_norm;
};

struct Params {
    const LayerPtrs* layers;
    int n_layers;
    const uint16_t* E;
    const float* final_norm;
    const float* inv_freq;
    int V;
    float eps;
    const int* tokens;
    const int* positions;
    const int* bt;
    int bt_stride;
    uint16_t* kv;
    int64_t layer_elems, page_elems;
    int n_pages;
    float* logits;
    float* R;      // [2][D]
    float* oacc;   // [2][NSH][D]
    float* dacc;   // [2][NSH][D]
    float* qkv;    // [QKVR]
    float* part;   // [HQ][nsa][PART]
    float* lm_part;  // [G][2]
    int* argmax;     // [1]
    unsigned* sync;  // counters
    int* err;
    int nsa;         // attention splits per KV head
    unsigned long long* trace;  // nullable: [G][n_layers + 1][TRACE_SLOTS] %globaltimer stamps
};

// counter slots
QW_DEV unsigned* c_epoch(const Params& p) { return p.sync; }
QW_DEV unsigned* c_qkvh(const Params& p, int l, int g) { return p.sync + CNT_STRIDE * (1 + l * 18 + g); }
QW_DEV unsigned* c_split(const Params& p, int l, int g) { return p.sync + CNT_STRIDE * (1 + l * 18 + 8 + g); }
QW_DEV unsigned* c_o(const Params& p, int l) { return p.sync + CNT_STRIDE * (1 + l * 18 + 16); }
QW_DEV unsigned* c_x(const Params& p, int l) { return p.sync + CNT_STRIDE * (1 + l * 18 + 17); }
QW_DEV unsigned* c_lm(const Params& p) { return p.sync + CNT_STRIDE * (1 + p.n_layers * 18); }

QW_DEV unsigned ld_acquire(const unsigned* ptr) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}
QW_DEV uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
QW_DEV void bar_consumers() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// Phase-boundary timestamp (tracing builds of a step only).
QW_DEV void stamp(const Params& p, int l, int k) {
    if (p.trace) p.trace[((size_t)blockIdx.x * (p.n_layers + 1) + l) * TRACE_SLOTS + k] = gtimer();
}

struct Smem {
    uint64_t full[NS], empty[NS];
    int spg[NS][PAGES_PER_STAGE];  // page ids of a KV stage (-1: none or out of range)
    volatile int abort_flag;
    int pad;
    alignas(16) float h[D];  // normalised activation of the current phase (read as float4)
    float res[MAX_ROWS];   // dot products of the current phase
    float coef[MAX_ROWS];  // scale of each row in the scaled-row phases
    float wsum[NCW];
    // rotated queries, pre-scaled to log2 units: dim 8 u + 4 h + e of head hh at q[hh][h][u][e], so
    // that the float4 reads of 8 different chunks u hit 8 different bank groups
    alignas(16) float q[2][2][HD / 8][4];
    alignas(16) uint16_t kn_b[HD];   // the new key and value as bf16 (as the cache holds them)
    alignas(16) uint16_t vn_b[HD];
    alignas(16) float pp[2][2][64];  // attention: exp2(s - m_w) per key slot (two stage buffers)
    float am[2][NCW][2], al[2][NCW][2];  // per-warp max and sum of those (two stage buffers)
    alignas(16) float ao[PAGES_PER_STAGE][2][HD];  // per-page partial outputs
    float alq[PAGES_PER_STAGE][2];
    float lm_val[NCW];
    int lm_idx[NCW];
    int last_cta;
};
constexpr int SMEM_BYTES = NS * STAGE + 1024 + (int)sizeof(Smem);

// Bounded wait for a global counter (one thread); false on timeout or abort.
QW_DEV bool wait_count(const unsigned* ptr, unsigned target, Smem& sm, int* err) {
    if ((int)(ld_acquire(ptr) - target) >= 0) return true;
    const uint64_t t0 = gtimer();
    for (unsigned i = 0;; ++i) {
        if ((int)(ld_acquire(ptr) - target) >= 0) return true;
        if ((i & 63) == 63) {
            if (sm.abort_flag) return false;
            if (gtimer() - t0 > WAIT_NS) {
                set_error(err, QW_ETIMEOUT);
                sm.abort_flag = 1;
                return false;
            }
        }
    }
}

// Publish: called by one thread after a barrier of every thread whose writes it
// publishes; the release orders those writes (through the barrier) before the add.
QW_DEV void signal_add(unsigned* ptr, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

QW_DEV void unpack8(uint4 w, float (&f)[8]) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

// Row slices: CTA c of G owns [n*c/G, n*(c+1)/G).
QW_DEV int slice_lo(int n, int c, int G) { return (int)((long)n * c / G); }

struct Work {
    int q0, q1;    // q|k|v rows
    int j0, j1;    // attention dims (rows of Wo^T)
    int p0, p1;    // gate/up pairs (rows of Wd^T)
    int v0, v1;    // LM-head rows
    int d0, d1;    // residual rows owned (materialise R, zero the accumulators)
    int g, s;      // attention item (g < 0: none)
    int pg_lo, pg_hi;  // pages of the attention item
    bool has_new;      // the item holds the new token's page
};

QW_DEV Work make_work(const Params& p, int c, int G, int pos, bool bad_pos) {
    Work w;
    w.q0 = slice_lo(QKVR, c, G);
    w.q1 = slice_lo(QKVR, c + 1, G);
    w.j0 = slice_lo(AD, c, G);
    w.j1 = slice_lo(AD, c + 1, G);
    w.p0 = slice_lo(INTER, c, G);
    w.p1 = slice_lo(INTER, c + 1, G);
    w.v0 = slice_lo(p.V, c, G);
    w.v1 = slice_lo(p.V, c + 1, G);
    w.d0 = 4 * slice_lo(D / 4, c, G);      // owned residual entries, in float4 groups
    w.d1 = 4 * slice_lo(D / 4, c + 1, G);
    w.g = -1;
    w.s = 0;
    w.pg_lo = w.pg_hi = 0;
    w.has_new = false;
    if (c < HKV * p.nsa) {
        if (bad_pos) pos = 0;
        w.g = c / p.nsa;
        w.s = c % p.nsa;
        const int np = pos / QW_PAGE_SIZE + 1;  // pages holding positions 0..pos
        w.pg_lo = (int)((long)np * w.s / p.nsa);
        w.pg_hi = (int)((long)np * (w.s + 1) / p.nsa);
        w.has_new = (pos / QW_PAGE_SIZE) >= w.pg_lo && (pos / QW_PAGE_SIZE) < w.pg_hi;
    }
    return w;
}

// ---------------------------------------------------------------- producer
struct Producer {
    uint8_t* ring;
    Smem* sm;
    int* err;
    unsigned it = 0;
    bool stop = false;

    QW_DEV bool acquire(int& s) {
        s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        for (uint32_t i = 0; i < QW_SPIN_LIMIT; ++i) {
            if (mbar_try_wait(&sm->empty[s], ph ^ 1)) return true;
            if ((i & 63) == 63 && sm->abort_flag) return false;
            if (i > 64) __nanosleep(64);
        }
        set_error(err, QW_ETIMEOUT);
        sm->abort_flag = 1;
        return false;
    }
    QW_DEV void rows(const uint16_t* base, int nrows) {
        for (int r0 = 0; r0 < nrows && !stop; r0 += ROWS_PER_STAGE) {
            const int n = min(ROWS_PER_STAGE, nrows - r0);
            int s;
            if (!acquire(s)) {
                stop = true;
                return;
            }
            mbar_arrive_expect_tx(&sm->full[s], n * ROW_B);
            bulk_load(ring + s * STAGE, base + (size_t)r0 * D, n * ROW_B, &sm->full[s]);
            ++it;
        }
    }
    // K and V of KV head g for pages [lo, hi) of one sequence: page i of a stage holds K at
    // i * 8 KB and V at i * 8 KB + 4 KB.
    QW_DEV void pages(const uint16_t* kv_layer, int64_t page_elems, int n_pages, const int* bt, int g, int lo,
                      int hi) {
        for (int p0 = lo; p0 < hi && !stop; p0 += PAGES_PER_STAGE) {
            const int n = min(PAGES_PER_STAGE, hi - p0);
            int s;
            if (!acquire(s)) {
                stop = true;
                return;
            }
            int pgs[PAGES_PER_STAGE];
            int valid = 0;
            for (int i = 0; i < PAGES_PER_STAGE; ++i) pgs[i] = i < n ? __ldg(bt + p0 + i) : -1;  // loads in flight together
            for (int i = 0; i < PAGES_PER_STAGE; ++i) {
                if (pgs[i] < 0 || pgs[i] >= n_pages) pgs[i] = -1;
                valid += pgs[i] >= 0;
                sm->spg[s][i] = pgs[i];  // published to the consumers by the arrive below
            }
            mbar_arrive_expect_tx(&sm->full[s], valid * 2 * PAGE_B);
            for (int i = 0; i < n; ++i) {
                const int pg = pgs[i];
                if (pg < 0) continue;
                const uint16_t* kp = kv_layer + (int64_t)pg * page_elems + (int64_t)g * QW_PAGE_SIZE * HD;
                bulk_load(ring + s * STAGE + i * 2 * PAGE_B, kp, PAGE_B, &sm->full[s]);
                bulk_load(ring + s * STAGE + i * 2 * PAGE_B + PAGE_B, kp + (int64_t)HKV * QW_PAGE_SIZE * HD, PAGE_B,
                          &sm->full[s]);
            }
            ++it;
        }
    }
    // Before the CTA exits: every copy issued must have landed.
    QW_DEV void drain() {
        const unsigned first = it > (unsigned)NS ? it - NS : 0;
        for (unsigned i = first; i < it; ++i) mbar_wait(&sm->full[i % NS], (i / NS) & 1, err);
    }
};

// ---------------------------------------------------------------- consumer helpers
struct Consumer {
    uint8_t* ring;
    Smem* sm;
    int* err;
    int cw, lane;   // consumer warp 0..7, lane
    unsigned it = 0;

    QW_DEV const uint8_t* stage_wait(bool& ok) {
        const int s = it % NS;
        ok = ok && !sm->abort_flag && mbar_wait(&sm->full[s], (it / NS) & 1, err);
        if (!ok) sm->abort_flag = 1;
        return ring + s * STAGE;
    }
    QW_DEV int slot() const { return it % NS; }
    QW_DEV void stage_release() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[it % NS]);
        ++it;
    }
    // Dot products of `nrows` streamed rows with sm->h; results to sm->res[0..nrows).
    QW_DEV bool dot_rows(int nrows, bool ok, const Params* tp = nullptr, int tl = 0, int tslot = 0) {
        float hreg[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 a = *(const float4*)&sm->h[8 * lane + 256 * i];
            const float4 b = *(const float4*)&sm->h[8 * lane + 256 * i + 4];
            hreg[i][0] = a.x; hreg[i][1] = a.y; hreg[i][2] = a.z; hreg[i][3] = a.w;
            hreg[i][4] = b.x; hreg[i][5] = b.y; hreg[i][6] = b.z; hreg[i][7] = b.w;
        }
        for (int r0 = 0; r0 < nrows; r0 += ROWS_PER_STAGE) {
            const int n = min(ROWS_PER_STAGE, nrows - r0);
            const uint8_t* st = stage_wait(ok);
            if (tp && r0 == 0 && cw == 0 && lane == 0) stamp(*tp, tl, tslot);
            if (ok) {
                // rows cw and cw + 8 together: two independent chains per row, loads issued first
                for (int r = cw; r < n; r += 2 * NCW) {
                    const bool two = r + NCW < n;
                    const uint4* ra = (const uint4*)(st + r * ROW_B);
                    const uint4* rb = (const uint4*)(st + (two ? r + NCW : r) * ROW_B);
                    uint4 wa[4], wb[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        wa[i] = ra[lane + 32 * i];
                        wb[i] = rb[lane + 32 * i];
                    }
                    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float fa[8], fb[8];
                        unpack8(wa[i], fa);
                        unpack8(wb[i], fb);
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            a0 = fmaf(hreg[i][e], fa[e], a0);
                            a1 = fmaf(hreg[i][e + 1], fa[e + 1], a1);
                            b0 = fmaf(hreg[i][e], fb[e], b0);
                            b1 = fmaf(hreg[i][e + 1], fb[e + 1], b1);
                        }
                    }
                    float a = a0 + a1, b = b0 + b1;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        a += __shfl_xor_sync(0xffffffffu, a, o);
                        b += __shfl_xor_sync(0xffffffffu, b, o);
                    }
                    if (lane == 0) {
                        sm->res[r0 + r] = a;
                        if (two) sm->res[r0 + r + NCW] = b;
                    }
                }
            }
            stage_release();
        }
        return ok;
    }
    // acc (columns 128 cw + 4 lane .. +3) += sum over streamed rows r of sm->coef[r] * row_r.
    // Each warp covers its own 128 output columns of every row, so no cross-warp sum is needed.
    QW_DEV bool scaled_rows(int nrows, float (&acc)[4], bool ok) {
        for (int r0 = 0; r0 < nrows; r0 += ROWS_PER_STAGE) {
            const int n = min(ROWS_PER_STAGE, nrows - r0);
            const uint8_t* st = stage_wait(ok);
            if (ok) {
                const uint8_t* col = st + (128 * cw + 4 * lane) * 2;
#pragma unroll 4
                for (int r = 0; r < n; ++r) {
                    const uint2 wv = *(const uint2*)(col + r * ROW_B);
                    const float a = sm->coef[r0 + r];
                    acc[0] = fmaf(a, bf16_lo(wv.x), acc[0]);
                    acc[1] = fmaf(a, bf16_hi(wv.x), acc[1]);
                    acc[2] = fmaf(a, bf16_lo(wv.y), acc[2]);
                    acc[3] = fmaf(a, bf16_hi(wv.y), acc[3]);
                }
            }
            stage_release();
        }
        return ok;
    }
};

// Sum over the NSH shards of a [NSH][D] accumulator at entries k0 .. k0+3 (loads in flight together).
QW_DEV float4 sum_shards(const float* base, int k0) {
    float4 v[NSH];
#pragma unroll
    for (int s = 0; s < NSH; ++s) v[s] = __ldcg((const float4*)(base + s * D + k0));
    float4 t = v[0];
#pragma unroll
    for (int s = 1; s < NSH; ++s) {
        t.x += v[s].x;
        t.y += v[s].y;
        t.z += v[s].z;
        t.w += v[s].w;
    }
    return t;
}

// Add this lane's 4 output columns into global dst (one 16-byte atomic).
QW_DEV void add_columns(const float (&acc)[4], float* dst, int cw, int lane) {
    atomicAdd((float4*)(dst + 128 * cw + 4 * lane), make_float4(acc[0], acc[1], acc[2], acc[3]));
}

// x (4 entries per consumer thread) -> sm.h = x / rms(x) * w.  Consumer barriers inside.
QW_DEV void norm_into_h(Smem& sm, const float (&x)[4], int k0, const float* w, float eps, int tid) {
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    ss = warp_sum(ss);
    if ((tid & 31) == 0) sm.wsum[tid >> 5] = ss;
    bar_consumers();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NCW; ++i) tot += sm.wsum[i];
    const float s = 1.0f / sqrtf(tot / (float)D + eps);
#pragma unroll
    for (int e = 0; e < 4; ++e) sm.h[k0 + e] = x[e] * s * w[k0 + e];
    bar_consumers();
}

__global__ void __launch_bounds__(THREADS, 1) fused_decode_kernel(Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Smem& sm = *(Smem*)(ring + NS * STAGE);
    const int G = gridDim.x, c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], NCW);
        }
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int pos = p.positions[0];
    const int tok = p.tokens[0];
    const unsigned epoch = ld_acquire(c_epoch(p)) + 1;  // this launch's targets are epoch * amount
    const bool bad_pos = pos < 0 || pos >= p.bt_stride * QW_PAGE_SIZE;
    const Work w = make_work(p, c, G, pos, bad_pos);
    if (bad_pos && c == 0 && threadIdx.x == 0) set_error(p.err, QW_ERANGE);

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            Producer pr{ring, &sm, p.err};
            for (int l = 0; l < p.n_layers && !pr.stop; ++l) {
                const LayerPtrs& L = p.layers[l];
                pr.rows(L.wqkv + (size_t)w.q0 * D, w.q1 - w.q0);
                if (w.g >= 0 && !bad_pos)
                    pr.pages(p.kv + (int64_t)l * p.layer_elems, p.page_elems, p.n_pages, p.bt, w.g, w.pg_lo,
                             w.pg_hi);
                pr.rows(L.woT + (size_t)w.j0 * D, w.j1 - w.j0);
                pr.rows(L.wgu + (size_t)2 * w.p0 * D, 2 * (w.p1 - w.p0));
                pr.rows(L.wdT + (size_t)w.p0 * D, w.p1 - w.p0);
                stamp(p, l, 9);
            }
            pr.rows(p.E + (size_t)w.v0 * D, w.v1 - w.v0);
            pr.drain();
        }
        return;
    }

    // ------------------------------------------------ consumers (warps 1..8)
    const int tid = threadIdx.x - 32;  // 0..255
    const int cw = tid >> 5;
    Consumer cs{ring, &sm, p.err, cw, lane};
    bool ok = !bad_pos;
    const int k0 = 4 * tid;  // this thread's 4 residual entries in the norm phases
    const bool own = k0 >= w.d0 && k0 < w.d1;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
    __shared__ bool s_ok;

    for (int l = 0; l < p.n_layers; ++l) {
        const LayerPtrs& L = p.layers[l];
        const int pb = l & 1, qb = pb ^ 1;
        // ---------------- P1: x -> norm -> q|k|v rows
        if (tid == 0) {
            stamp(p, l, 0);
            s_ok = ok && (l == 0 || wait_count(c_x(p, l - 1), epoch * G, sm, p.err));
            stamp(p, l, 1);
        }
        bar_consumers();
        ok = s_ok;
        float x[4];
        if (l == 0) {
            const uint2 e = (tok >= 0 && tok < p.V) ? *(const uint2*)(p.E + (size_t)tok * D + k0) : make_uint2(0, 0);
            x[0] = bf16_lo(e.x); x[1] = bf16_hi(e.x); x[2] = bf16_lo(e.y); x[3] = bf16_hi(e.y);
            if (c == 0 && tid == 0 && !(tok >= 0 && tok < p.V)) set_error(p.err, QW_ERANGE);
        } else {
            const float4 r = __ldcg((const float4*)(p.R + qb * D + k0));
            const float4 o = sum_shards(p.oacc + qb * NSH * D, k0);
            const float4 d = sum_shards(p.dacc + qb * NSH * D, k0);
            x[0] = r.x + o.x + d.x; x[1] = r.y + o.y + d.y; x[2] = r.z + o.z + d.z; x[3] = r.w + o.w + d.w;
        }
        if (own) *(float4*)(p.R + pb * D + k0) = make_float4(x[0], x[1], x[2], x[3]);
        norm_into_h(sm, x, k0, L.in_norm, p.eps, tid);
        if (tid == 0) stamp(p, l, 10);
        ok = cs.dot_rows(w.q1 - w.q0, ok, &p, l, 16);
        if (tid == 0) stamp(p, l, 11);
        bar_consumers();
        for (int r = tid; r < w.q1 - w.q0; r += 256) p.qkv[w.q0 + r] = sm.res[r];
        bar_consumers();
        if (tid == 0) {
            // rows of KV-head group g: q rows [256g, 256g+256), k rows 2048 + [128g, ..), v rows 3072 + [128g, ..)
            for (int g = 0; g < HKV; ++g) {
                int n = 0;
                const int ranges[3][2] = {{256 * g, 256 * g + 256}, {2048 + 128 * g, 2048 + 128 * g + 128},
                                          {3072 + 128 * g, 3072 + 128 * g + 128}};
                for (int t = 0; t < 3; ++t) n += max(0, min(w.q1, ranges[t][1]) - max(w.q0, ranges[t][0]));
                if (n) signal_add(c_qkvh(p, l, g), (unsigned)n);
            }
            stamp(p, l, 2);
        }
        // ---------------- P2: attention split
        if (w.g >= 0) {
            const int g = w.g;
            if (tid == 0) {
                s_ok = ok && wait_count(c_qkvh(p, l, g), epoch * 512, sm, p.err);
                stamp(p, l, 3);
            }
            bar_consumers();
            ok = s_ok;
            if (cw < 4 && ok) {
                // warp 0,1: q heads 2g, 2g+1; warp 2: k head g; warp 3: v head g
                const int off = cw < 2 ? (2 * g + cw) * HD : (cw == 2 ? 2048 + g * HD : 3072 + g * HD);
                float y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = __ldcg(p.qkv + off + lane + 32 * i);
                if (cw < 3) {
                    const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
                    const float sc = 1.0f / sqrtf(ss / (float)HD + p.eps);
                    const float* nw = cw < 2 ? L.q_norm : L.k_norm;
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[i] = y[i] * sc * nw[lane + 32 * i];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float ang = __fmul_rn((float)pos, p.inv_freq[lane + 32 * j]);
                        float sn, cs_;
                        sincosf(ang, &sn, &cs_);
                        const float a = y[j], b = y[j + 2];
                        y[j] = a * cs_ - b * sn;
                        y[j + 2] = a * sn + b * cs_;
                    }
                }
                if (cw >= 2) {
                    // the new K and V enter the cache as bf16; attention uses those values
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[i] = __uint_as_float((uint32_t)f2bf(y[i]) << 16);
                    if (w.has_new) {
                        const int pg = p.bt[pos / QW_PAGE_SIZE];
                        if (pg >= 0 && pg < p.n_pages) {
                            uint16_t* dst = p.kv + (int64_t)l * p.layer_elems + (int64_t)pg * p.page_elems +
                                            ((int64_t)((cw - 2) * HKV + g) * QW_PAGE_SIZE + pos % QW_PAGE_SIZE) * HD;
#pragma unroll
                            for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = f2bf(y[i]);
                        } else if (lane == 0) {
                            set_error(p.err, QW_ERANGE);
                        }
                    }
                }
                if (cw < 2) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int dd = lane + 32 * i;
                        sm.q[cw][(dd >> 2) & 1][dd >> 3][dd & 3] = y[i] * scale_log2;
                    }
                } else {
                    uint16_t* db = cw == 2 ? sm.kn_b : sm.vn_b;
#pragma unroll
                    for (int i = 0; i < 4; ++i) db[lane + 32 * i] = f2bf(y[i]);
                }
            }
            bar_consumers();
            if (tid == 0) stamp(p, l, 18);
            // Each stage holds up to 4 pages (64 key slots).  Scores: warp cw takes slots
            // 8 cw .. 8 cw + 7, one per 4-lane group (kg = lane >> 2); lane dq = lane & 3 of a group
            // takes the 16-byte chunks u = 4 c' + dq, c' = c ^ (kg & 1), of the key row (the xor
            // puts the 8 lanes of each shared-memory phase on 8 different bank groups), and publishes exp2(s - m_w) with its warp max m_w and sum
            // l_w.  P.V: thread (page pi = tid >> 6, dim pair dp = tid & 63) sums the 16 slots of
            // page pi for both query heads under one running max M shared by all threads, so
            // the four page partials add up without rescaling at the end.
            const int kg = lane >> 2, dq = lane & 3;
            const int vpi = tid >> 6, dp = tid & 63;
            float Mr[2] = {-INFINITY, -INFINITY}, lq[2] = {0.f, 0.f}, oq[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            int buf = 0;
            for (int pg0 = w.pg_lo; pg0 < w.pg_hi; pg0 += PAGES_PER_STAGE, buf ^= 1) {
                const int n = min(PAGES_PER_STAGE, w.pg_hi - pg0);
                const uint8_t* st = cs.stage_wait(ok);
                if (tid == 0 && pg0 == w.pg_lo) {
                    stamp(p, l, 20);
                    if (p.trace) p.trace[((size_t)blockIdx.x * (p.n_layers + 1) + l) * TRACE_SLOTS + 22] = clock64();
                }
                {
                    const int pi = cw >> 1, slot = 8 * (cw & 1) + kg;
                    const int kpos = (pg0 + pi) * QW_PAGE_SIZE + slot;
                    const bool vis = ok && pi < n && kpos <= pos && sm.spg[cs.slot()][pi] >= 0;
                    // the new token's key comes from the bf16 copy made above, not the (older) stage
                    const uint8_t* krow = kpos == pos ? (const uint8_t*)sm.kn_b
                                                      : st + (pi < n ? pi : 0) * 2 * PAGE_B + slot * HD * 2;
                    float sc[2] = {0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int u = 4 * (c ^ (kg & 1)) + dq;
                        float kf[8];
                        unpack8(((const uint4*)krow)[u], kf);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const float4 qa = *(const float4*)sm.q[hh][0][u];
                            const float4 qb = *(const float4*)sm.q[hh][1][u];
                            sc[hh] += qa.x * kf[0] + qa.y * kf[1] + qa.z * kf[2] + qa.w * kf[3] + qb.x * kf[4] +
                                      qb.y * kf[5] + qb.z * kf[6] + qb.w * kf[7];
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 1);
                        sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 2);
                        float mw = vis ? sc[hh] : -INFINITY;
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
                        const float pe = vis ? exp2f(sc[hh] - mw) : 0.f;
                        float lw = pe;
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
                        if (dq == 0) sm.pp[buf][hh][8 * cw + kg] = pe;
                        if (lane == 0) {
                            sm.am[buf][cw][hh] = mw;
                            sm.al[buf][cw][hh] = lw;
                        }
                    }
                }
                bar_consumers();
                if (tid == 0 && pg0 == w.pg_lo) {
                    if (p.trace) p.trace[((size_t)blockIdx.x * (p.n_layers + 1) + l) * TRACE_SLOTS + 23] = clock64();
                    stamp(p, l, 21);
                }
                // P.V over page vpi; the buffers of this stage are not rewritten before the
                // barrier of the next stage, which every thread reaches only after this part.
                float Ms[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    Ms[hh] = Mr[hh];
#pragma unroll
                    for (int i = 0; i < NCW; ++i) Ms[hh] = fmaxf(Ms[hh], sm.am[buf][i][hh]);
                }
                float fa[2], fb[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (Ms[hh] == -INFINITY) {  // nothing visible yet for this head
                        fa[hh] = fb[hh] = 0.f;
                        continue;
                    }
                    const float ma = sm.am[buf][2 * vpi][hh], mb = sm.am[buf][2 * vpi + 1][hh];
                    const float alpha = Mr[hh] == -INFINITY ? 0.f : exp2f(Mr[hh] - Ms[hh]);
                    fa[hh] = ma == -INFINITY ? 0.f : exp2f(ma - Ms[hh]);
                    fb[hh] = mb == -INFINITY ? 0.f : exp2f(mb - Ms[hh]);
                    lq[hh] = lq[hh] * alpha + fa[hh] * sm.al[buf][2 * vpi][hh] + fb[hh] * sm.al[buf][2 * vpi + 1][hh];
                    oq[hh][0] *= alpha;
                    oq[hh][1] *= alpha;
                    Mr[hh] = Ms[hh];
                }
                if (fa[0] + fb[0] + fa[1] + fb[1] > 0.f) {  // page vpi has a visible key
                    const uint8_t* vpage = st + vpi * 2 * PAGE_B + PAGE_B + 4 * dp;
                    const int knew = pos - (pg0 + vpi) * QW_PAGE_SIZE;  // slot of the new token, if here
                    float s0[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, s1[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const float4* pa = (const float4*)&sm.pp[buf][0][16 * vpi + 8 * half];
                        const float4* pb = (const float4*)&sm.pp[buf][1][16 * vpi + 8 * half];
                        const float4 pa0 = pa[0], pa1 = pa[1], pb0 = pb[0], pb1 = pb[1];
                        const float p0[8] = {pa0.x, pa0.y, pa0.z, pa0.w, pa1.x, pa1.y, pa1.z, pa1.w};
                        const float p1[8] = {pb0.x, pb0.y, pb0.z, pb0.w, pb1.x, pb1.y, pb1.z, pb1.w};
                        float (&acc)[2][2] = half ? s1 : s0;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int slot = 8 * half + k;
                            const uint32_t v = slot == knew ? *(const uint32_t*)((const uint8_t*)sm.vn_b + 4 * dp)
                                                            : *(const uint32_t*)(vpage + slot * HD * 2);
                            const float v0 = bf16_lo(v), v1 = bf16_hi(v);
                            acc[0][0] = fmaf(p0[k], v0, acc[0][0]);
                            acc[0][1] = fmaf(p0[k], v1, acc[0][1]);
                            acc[1][0] = fmaf(p1[k], v0, acc[1][0]);
                            acc[1][1] = fmaf(p1[k], v1, acc[1][1]);
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int e = 0; e < 2; ++e) oq[hh][e] += fa[hh] * s0[hh][e] + fb[hh] * s1[hh][e];
                }
                cs.stage_release();
            }
            if (tid == 0) stamp(p, l, 19);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                *(float2*)&sm.ao[vpi][hh][2 * dp] = make_float2(oq[hh][0], oq[hh][1]);
                if (dp == 0) sm.alq[vpi][hh] = lq[hh];
            }
            bar_consumers();
            {
                const int hh = tid >> 7, d = tid & 127;
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int i = 0; i < PAGES_PER_STAGE; ++i) {
                    Ls += sm.alq[i][hh];
                    O += sm.ao[i][hh][d];
                }
                float* dst = p.part + ((size_t)(2 * g + hh) * p.nsa + w.s) * PART;
                dst[d] = O;
                if (d == 0) {
                    dst[HD] = Mr[hh];
                    dst[HD + 1] = Ls;
                }
            }
            bar_consumers();
            if (tid == 0) {
                signal_add(c_split(p, l, g), 1u);
                stamp(p, l, 4);
            }
        }
        // ---------------- P3: merge splits of this CTA's attention dims, o_proj rows of Wo^T
        {
            const int nj = w.j1 - w.j0;
            if (tid == 0) {
                bool good = ok;
                const int g_lo = w.j0 / (2 * HD), g_hi = (w.j1 - 1) / (2 * HD);
                for (int g = g_lo; g <= g_hi && good; ++g) good = wait_count(c_split(p, l, g), epoch * p.nsa, sm, p.err);
                s_ok = good;
                stamp(p, l, 5);
            }
            bar_consumers();
            ok = s_ok;
            if (ok) {
                // at most two dims per warp: issue all loads before the reductions
                float ms[2], ls[2], os[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int jj = cw + NCW * k;
                    ms[k] = -INFINITY;
                    ls[k] = os[k] = 0.f;
                    if (jj < nj && lane < p.nsa) {
                        const int j = w.j0 + jj;
                        const float* base = p.part + ((size_t)(j / HD) * p.nsa + lane) * PART;
                        ms[k] = __ldcg(base + HD);
                        ls[k] = __ldcg(base + HD + 1);
                        os[k] = __ldcg(base + j % HD);
                    }
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int jj = cw + NCW * k;
                    const float M = warp_max(ls[k] > 0.f ? ms[k] : -INFINITY);
                    const float f = ls[k] > 0.f ? exp2f(ms[k] - M) : 0.f;
                    const float Lt = warp_sum(ls[k] * f), Ot = warp_sum(os[k] * f);
                    if (lane == 0 && jj < nj) sm.coef[jj] = Lt > 0.f ? Ot / Lt : 0.f;
                }
            }
            bar_consumers();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (tid == 0) stamp(p, l, 15);
            ok = cs.scaled_rows(nj, acc, ok);
            add_columns(acc, p.oacc + (pb * NSH + c % NSH) * D, cw, lane);
            bar_consumers();
            if (tid == 0) {
                signal_add(c_o(p, l), 1u);
                stamp(p, l, 6);
            }
        }
        // ---------------- P4: norm -> gate/up -> SwiGLU -> down_proj rows of Wd^T
        {
            if (tid == 0) {
                s_ok = ok && wait_count(c_o(p, l), epoch * G, sm, p.err);
                stamp(p, l, 7);
            }
            bar_consumers();
            ok = s_ok;
            const float4 r = __ldcg((const float4*)(p.R + pb * D + k0));
            const float4 oa = sum_shards(p.oacc + pb * NSH * D, k0);
            float xm[4] = {r.x + oa.x, r.y + oa.y, r.z + oa.z, r.w + oa.w};
            if (own && l > 0) {  // every reader of the previous layer's accumulators is done
#pragma unroll
                for (int sh = 0; sh < NSH; ++sh) {
                    *(float4*)(p.oacc + (qb * NSH + sh) * D + k0) = make_float4(0.f, 0.f, 0.f, 0.f);
                    *(float4*)(p.dacc + (qb * NSH + sh) * D + k0) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            norm_into_h(sm, xm, k0, L.post_norm, p.eps, tid);
            if (tid == 0) stamp(p, l, 12);
            const int np2 = w.p1 - w.p0;
            ok = cs.dot_rows(2 * np2, ok, &p, l, 17);
            if (tid == 0) stamp(p, l, 13);
            bar_consumers();
            for (int j = tid; j < np2; j += 256) {
                const float gt = sm.res[2 * j], up = sm.res[2 * j + 1];
                sm.coef[j] = gt / (1.0f + expf(-gt)) * up;
            }
            bar_consumers();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            ok = cs.scaled_rows(np2, acc, ok);
            if (tid == 0) stamp(p, l, 14);
            add_columns(acc, p.dacc + (pb * NSH + c % NSH) * D, cw, lane);
            bar_consumers();
            if (tid == 0) {
                signal_add(c_x(p, l), 1u);
                stamp(p, l, 8);
            }
        }
    }
    // ---------------- LM head: final norm, tied embedding rows, argmax
    {
        const int pl = (p.n_layers - 1) & 1;
        if (tid == 0) {
            stamp(p, p.n_layers, 0);
            s_ok = ok && wait_count(c_x(p, p.n_layers - 1), epoch * G, sm, p.err);
            stamp(p, p.n_layers, 1);
        }
        bar_consumers();
        ok = s_ok;
        const float4 r = __ldcg((const float4*)(p.R + pl * D + k0));
        const float4 oa = sum_shards(p.oacc + pl * NSH * D, k0);
        const float4 da = sum_shards(p.dacc + pl * NSH * D, k0);
        float xf[4] = {r.x + oa.x + da.x, r.y + oa.y + da.y, r.z + oa.z + da.z, r.w + oa.w + da.w};
        norm_into_h(sm, xf, k0, p.final_norm, p.eps, tid);
        float hreg[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) hreg[i][e] = sm.h[8 * lane + 256 * i + e];
        float best = -INFINITY;
        int bidx = 0x7FFFFFFF;
        const int nv = w.v1 - w.v0;
        for (int r0 = 0; r0 < nv; r0 += ROWS_PER_STAGE) {
            const int n = min(ROWS_PER_STAGE, nv - r0);
            const uint8_t* st = cs.stage_wait(ok);
            if (ok) {
                for (int rr = cw; rr < n; rr += NCW) {
                    const uint4* row = (const uint4*)(st + rr * ROW_B);
                    float a = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float f[8];
                        unpack8(row[lane + 32 * i], f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) a = fmaf(hreg[i][e], f[e], a);
                    }
                    a = warp_sum(a);
                    const int v = w.v0 + r0 + rr;
                    if (lane == 0) p.logits[v] = a;
                    if (a > best || (a == best && v < bidx)) {
                        best = a;
                        bidx = v;
                    }
                }
            }
            cs.stage_release();
        }
        if (lane == 0) {
            sm.lm_val[cw] = best;
            sm.lm_idx[cw] = bidx;
        }
        bar_consumers();
        if (tid == 0) {
            for (int i = 1; i < NCW; ++i)
                if (sm.lm_val[i] > best || (sm.lm_val[i] == best && sm.lm_idx[i] < bidx)) {
                    best = sm.lm_val[i];
                    bidx = sm.lm_idx[i];
                }
            stamp(p, p.n_layers, 2);
            p.lm_part[2 * c] = best;
            p.lm_part[2 * c + 1] = __int_as_float(bidx);
            unsigned prev;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(c_lm(p)) : "memory");
            sm.last_cta = prev == epoch * G - 1;
            if (sm.last_cta) {
                // last CTA: global argmax (lowest id on ties); below, reset the accumulators, next epoch
                __threadfence();
                float bv = -INFINITY;
                int bi = 0x7FFFFFFF;
                for (int i = 0; i < G; ++i) {
                    const float v = __ldcg(p.lm_part + 2 * i);
                    const int ix = __float_as_int(__ldcg(p.lm_part + 2 * i + 1));
                    if (v > bv || (v == bv && ix < bi)) {
                        bv = v;
                        bi = ix;
                    }
                }
                *p.argmax = bi;
            }
        }
        bar_consumers();
        if (sm.last_cta) {  // every CTA has read the last layer's accumulators
            for (int k = tid; k < NSH * D; k += 256) {
                p.oacc[pl * NSH * D + k] = 0.f;
                p.dacc[pl * NSH * D + k] = 0.f;
            }
            bar_consumers();
            if (tid == 0) signal_add(c_epoch(p), 1u);
        }
    }
}

// Wt[j][i] = W[i][j] for a [rows][cols] bf16 matrix.
__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ W, uint16_t* __restrict__ Wt, int rows, int cols) {
    __shared__ uint16_t tile[32][33];
    const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
    for (int y = threadIdx.y; y < 32; y += 8) {
        const int r = by + y, cc = bx + threadIdx.x;
        if (r < rows && cc < cols) tile[y][threadIdx.x] = W[(size_t)r * cols + cc];
    }
    __syncthreads();
    for (int y = threadIdx.y; y < 32; y += 8) {
        const int cc = bx + y, r = by + threadIdx.x;
        if (r < rows && cc < cols) Wt[(size_t)cc * rows + r] = tile[threadIdx.x][y];
    }
}

}  // namespace fused

// ---------------------------------------------------------------- host side
struct FusedDecode {
    int G = 0, nsa = 0, n_layers = 0, V = 0;
    float eps = 0.f;
    uint8_t* buf = nullptr;
    fused::LayerPtrs* d_layers = nullptr;
    const uint16_t* E = nullptr;
    const float* final_norm = nullptr;
    const float* inv_freq = nullptr;
    float *R = nullptr, *oacc = nullptr, *dacc = nullptr, *qkv = nullptr, *part = nullptr, *lm_part = nullptr;
    int* argmax = nullptr;
    unsigned* sync = nullptr;
    unsigned long long* trace = nullptr;
    bool trace_on = false;
};

FusedDecode* fused_create(const FusedWeights& fw, int n_layers, int V, float eps, int hidden, int n_heads,
                          int n_kv_heads, int intermediate) {
    using namespace fused;
    if (hidden != D || n_heads != HQ || n_kv_heads != HKV || intermediate != INTER || n_layers > MAX_LAYERS) return nullptr;
    int dev = 0, n_sm = 0, coop = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (!coop || n_sm < HKV) return nullptr;
    if (cudaFuncSetAttribute(fused_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
        return nullptr;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_decode_kernel, THREADS, SMEM_BYTES) !=
            cudaSuccess ||
        per_sm < 1)
        return nullptr;
    FusedDecode* f = new FusedDecode();
    f->G = n_sm;
    f->nsa = n_sm / HKV;
    if (f->nsa > 32) f->nsa = 32;   // the split merge reads one split per lane
    if ((QKVR + f->G - 1) / f->G > MAX_ROWS || (2 * (INTER + f->G - 1) / f->G) > MAX_ROWS ||
        (AD + f->G - 1) / f->G > 2 * NCW) {  // the split merge takes at most two dims per warp
        delete f;
        return nullptr;
    }
    f->n_layers = n_layers;
    f->V = V;
    f->eps = eps;
    f->E = fw.E;
    f->final_norm = fw.final_norm;
    f->inv_freq = fw.inv_freq;
    const size_t woT = (size_t)AD * D, wdT = (size_t)INTER * D;
    size_t off = 0;
    auto take = [&](size_t b) {
        size_t o = off;
        off = (off + b + 1023) / 1024 * 1024;
        return o;
    };
    const size_t o_w = take((woT + wdT) * 2 * n_layers);
    const size_t o_layers = take(sizeof(LayerPtrs) * n_layers);
    const size_t o_state = take(sizeof(float) * (2 * D + 4 * NSH * D + QKVR));
    const size_t o_part = take(sizeof(float) * HQ * f->nsa * PART);
    const size_t o_lm = take(sizeof(float) * 2 * f->G + 64);
    const size_t o_sync = take(sizeof(unsigned) * CNT_STRIDE * (2 + n_layers * 18));
    const size_t o_trace = take(sizeof(unsigned long long) * f->G * (n_layers + 1) * TRACE_SLOTS);
    if (cudaMalloc(&f->buf, off) != cudaSuccess) {
        delete f;
        return nullptr;
    }
    uint16_t* wt = (uint16_t*)(f->buf + o_w);
    std::vector<LayerPtrs> lp(n_layers);
    for (int l = 0; l < n_layers; ++l) {
        uint16_t* woT_l = wt + (size_t)l * (woT + wdT);
        uint16_t* wdT_l = woT_l + woT;
        transpose_bf16_kernel<<<dim3(AD / 32, D / 32), dim3(32, 8)>>>(fw.wo[l], woT_l, D, AD);
        transpose_bf16_kernel<<<dim3(INTER / 32, D / 32), dim3(32, 8)>>>(fw.wd[l], wdT_l, D, INTER);
        lp[l] = LayerPtrs{fw.wqkv[l], woT_l, fw.wgu[l], wdT_l, fw.in_norm[l], fw.post_norm[l], fw.q_norm[l],
                          fw.k_norm[l]};
    }
    f->d_layers = (LayerPtrs*)(f->buf + o_layers);
    float* st = (float*)(f->buf + o_state);
    f->R = st;
    f->oacc = st + 2 * D;
    f->dacc = st + 2 * D + 2 * NSH * D;
    f->qkv = st + 2 * D + 4 * NSH * D;
    f->part = (float*)(f->buf + o_part);
    f->lm_part = (float*)(f->buf + o_lm);
    f->argmax = (int*)(f->lm_part + 2 * f->G);
    f->sync = (unsigned*)(f->buf + o_sync);
    f->trace = (unsigned long long*)(f->buf + o_trace);
    if (cudaMemcpy(f->d_layers, lp.data(), sizeof(LayerPtrs) * n_layers, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(f->buf + o_state, 0, off - o_state) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(f->buf);
        delete f;
        return nullptr;
    }
    return f;
}

bool fused_supported(const FusedDecode* f, int batch) { return f != nullptr && batch == 1; }

int fused_reset(FusedDecode* f, cudaStream_t st) {
    // after a timeout the counters and accumulators are in an unknown state
    const size_t bytes = (size_t)((uint8_t*)f->sync - (uint8_t*)f->R) +
                         sizeof(unsigned) * fused::CNT_STRIDE * (2 + f->n_layers * 18);
    return cudaMemsetAsync(f->R, 0, bytes, st) == cudaSuccess ? QW_OK : QW_ECUDA;
}

int fused_decode(FusedDecode* f, const int* tokens, const int* positions, int batch, uint16_t* kv_base,
                 int64_t layer_elems, int64_t page_elems, int n_pages, const int* block_tables, int bt_stride,
                 float* logits, int* err, cudaStream_t st) {
    using namespace fused;
    if (!f || batch != 1) return QW_EINVAL;
    Params p;
    p.layers = f->d_layers;
    p.n_layers = f->n_layers;
    p.E = f->E;
    p.final_norm = f->final_norm;
    p.inv_freq = f->inv_freq;
    p.V = f->V;
    p.eps = f->eps;
    p.tokens = tokens;
    p.positions = positions;
    p.bt = block_tables;
    p.bt_stride = bt_stride;
    p.kv = kv_base;
    p.layer_elems = layer_elems;
    p.page_elems = page_elems;
    p.n_pages = n_pages;
    p.logits = logits;
    p.R = f->R;
    p.oacc = f->oacc;
    p.dacc = f->dacc;
    p.qkv = f->qkv;
    p.part = f->part;
    p.lm_part = f->lm_part;
    p.argmax = f->argmax;
    p.sync = f->sync;
    p.err = err;
    p.nsa = f->nsa;
    p.trace = f->trace_on ? f->trace : nullptr;
    void* args[] = {&p};
    cudaError_t e = cudaLaunchCooperativeKernel((const void*)fused_decode_kernel, dim3(f->G), dim3(THREADS), args,
                                                SMEM_BYTES, st);
    count_launches(1);
    return e == cudaSuccess ? QW_OK : QW_ECUDA;
}

const int* fused_argmax(const FusedDecode* f) { return f ? f->argmax : nullptr; }

int fused_trace(FusedDecode* f, int enable, uint64_t* host_out, int64_t n, int64_t* n_needed) {
    if (!f) return QW_EINVAL;
    const int64_t total = (int64_t)f->G * (f->n_layers + 1) * fused::TRACE_SLOTS;
    if (n_needed) *n_needed = total;
    if (host_out) {
        if (cudaDeviceSynchronize() != cudaSuccess) return QW_ECUDA;
        if (cudaMemcpy(host_out, f->trace, sizeof(uint64_t) * (n < total ? n : total), cudaMemcpyDeviceToHost) !=
            cudaSuccess)
            return QW_ECUDA;
    }
    if (enable && !f->trace_on && cudaMemset(f->trace, 0, sizeof(uint64_t) * total) != cudaSuccess) return QW_ECUDA;
    f->trace_on = enable != 0;
    return QW_OK;
}

void fused_destroy(FusedDecode* f) {
    if (!f) return;
    cudaFree(f->buf);
    delete f;
}

}  // namespace qw
