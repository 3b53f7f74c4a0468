// Fused persistent decode for one sequence (batch 1): one cooperative launch per
// step runs the article's whole forward pass (Steps 2-8) for the new token.
//
// The grid is made of clusters of 8 CTAs (one CTA per SM).  Clusters 0..7 each own
// one KV head group g (two query heads sharing KV head g, Step 5) and do the whole
// attention sublayer of that group without leaving the cluster:
//
//   A1  x -> RMSNorm -> this CTA's 64 of the group's 512 q|k|v rows; the values are
//       pushed into every cluster peer's shared memory (st.async, counted by an mbarrier)
//   A2  QK-Norm, RoPE, the new K/V into the cache; attention over this CTA's eighth of
//       the cached pages -> partial (max, sum, weighted values), pushed to the peers
//       that own each output dimension
//   A3  merge of the 8 partials for this CTA's 32 attention dims, o_proj as the sum of
//       32 scaled rows of Wo^T, a reduction of the 8 CTAs' partial outputs through
//       shared memory, and one store of this CTA's 128 outputs into the group's slot
//
// Then every cluster runs the feed-forward sublayer (Step 6), each CTA owning a slice
// of the SwiGLU units:
//
//   M1  x + sum of the 8 group slots -> RMSNorm -> gate/up row pairs -> SwiGLU ->
//       down_proj as scaled rows of Wd^T -> reduction inside the cluster -> one slot
//       per cluster
//   LM  x + sum of the cluster slots -> final RMSNorm -> tied LM-head rows, argmax
//
// So a layer crosses the GPU twice (group slots -> feed-forward, cluster slots -> next
// layer), each time through per-cluster counters (release add / acquire poll, bounded
// by %globaltimer); everything else moves between the 8 SMs of a cluster.  Every CTA
// keeps its own copy of the fp32 residual stream and adds the slots in a fixed order,
// so the step is deterministic.  Warp 0 of each CTA streams the CTA's weight rows and
// KV pages of every layer, then the LM-head rows, through a shared-memory ring with
// cp.async.bulk in consumption order, independent of the data, so HBM keeps streaming
// while the consumers wait.
#include <vector>

#include "qw_common.cuh"
#include "qw_fused.h"
#include "qw_internal.h"

namespace qw {
namespace fused {

constexpr int D = 1024, HQ = 16, HKV = 8, HD = 128, INTER = 3072, AD = 2048;
constexpr int CL = 8;                 // CTAs per cluster
constexpr int MAX_CLUSTERS = 16;
constexpr int NS = 6;                 // ring stages
constexpr int STAGE = 32768;          // bytes per stage
// Streamed weight rows are 1024 wide: bf16 (2 KB, 16 per stage) or, with weight-only int8
// (Q8), int8 codes (1 KB, 32 per stage) with one fp32 scale per output channel.
template <bool Q8> constexpr int row_bytes() { return Q8 ? D : 2 * D; }
template <bool Q8> constexpr int rows_per_stage() { return STAGE / row_bytes<Q8>(); }
constexpr int PAGE_B = QW_PAGE_SIZE * HD * 2;   // K (or V) of one head in one page: 4 KB
constexpr int PAGES_PER_STAGE = STAGE / (2 * PAGE_B);  // 4
constexpr int NCW = 8;                // consumer warps
constexpr int THREADS = 32 * (NCW + 1);
constexpr int CNT_STRIDE = 32;        // counters 128 bytes apart
constexpr int QROWS = 512 / CL;       // q|k|v rows per attention CTA: 64
constexpr int ODIMS = 2 * HD / CL;    // attention dims per attention CTA: 32
constexpr int OWN = D / CL;           // outputs each CTA reduces for its cluster: 128
constexpr int MAX_ROWS = 128;         // per-phase result slots
constexpr int MAX_LAYERS = 64;
constexpr int PF = 8;                 // L2 prefetch distance beyond the ring, in stages
constexpr int MAX_PAGES = 512;        // pages per attention CTA: caches up to 8 * 512 * 16 = 65536 positions
constexpr int CNT_PER_LAYER = HKV + MAX_CLUSTERS;
constexpr uint64_t WAIT_NS = 2000000000ull;        // 2 s: far beyond any legitimate wait
constexpr uint64_t FAULT_WAIT_NS = 2000000ull;     // 2 ms: the injected timeout of the test hook
constexpr int TRACE_SLOTS = QW_TRACE_SLOTS;
constexpr uint32_t QKV_BYTES = 512 * 4;                 // per layer into each attention CTA
constexpr uint32_t PART_BYTES = CL * ODIMS * 4 + CL * 16;  // O of my dims + (M, L) of both heads, 8 sources
constexpr uint32_t RED_BYTES = CL * OWN * 4;            // 8 partial vectors of my 128 outputs

struct LayerPtrs {
    const uint8_t *wqkv, *woT, *wgu, *wdT;        // rows of bf16 or of int8 codes
    const float *in_norm, *post_norm, *q_norm, *k_norm;
    const float *s_qkv, *s_o, *s_gu, *s_d;        // int8: scale of each output channel (else null)
};

struct Params {
    const LayerPtrs* layers;
    int n_layers;
    const uint8_t* E;        // embedding / tied LM head rows (bf16 or int8 codes)
    const float* s_E;        // int8: scale of each vocabulary row
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
    float* oslot;    // [2][HKV][D]  o_proj outputs of each KV group (layer parity)
    float* dslot;    // [2][MAX_CLUSTERS][D]  down_proj outputs of each cluster
    float* lm_part;  // [G][2]
    int* argmax;     // [1]
    unsigned* sync;  // counters
    int* err;
    int n_clusters;
    unsigned long long* trace;  // nullable: [G][n_layers + 1][TRACE_SLOTS] %globaltimer stamps
    uint64_t wait_ns;           // limit of every bounded wait
    unsigned fault_extra;       // test hook: layer 0's feed-forward waits for this many arrivals more than come
};

// counter slots
QW_DEV unsigned* c_epoch(const Params& p) { return p.sync; }
QW_DEV unsigned* c_abort(const Params& p) { return p.sync + CNT_STRIDE; }
QW_DEV unsigned* c_o(const Params& p, int l, int g) { return p.sync + CNT_STRIDE * (2 + l * CNT_PER_LAYER + g); }
QW_DEV unsigned* c_x(const Params& p, int l, int c) {
    return p.sync + CNT_STRIDE * (2 + l * CNT_PER_LAYER + HKV + c);
}
QW_DEV unsigned* c_lm(const Params& p) { return p.sync + CNT_STRIDE * (2 + p.n_layers * CNT_PER_LAYER); }


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
QW_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
QW_DEV uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
QW_DEV void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of this CTA's shared variable `local` in the shared memory of cluster peer `rank`.
QW_DEV uint32_t peer_addr(const void* local, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}
// 16 (8) bytes into a peer's shared memory; the peer's mbarrier counts them on arrival.
QW_DEV void push4(uint32_t raddr, float4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     raddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
                 : "memory");
}
QW_DEV void push2(uint32_t raddr, float a, float b, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
                 "f"(a), "f"(b), "r"(rbar)
                 : "memory");
}
QW_DEV bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
QW_DEV bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

struct Smem {
    uint64_t full[NS], empty[NS];
    uint64_t bar_qkv, bar_part, bar_redo, bar_redd;  // cluster exchanges (one phase per layer)
    int spg[NS][PAGES_PER_STAGE];  // page ids of a KV stage (-1: none or out of range)
    int pages[MAX_PAGES];          // page ids of this CTA's share of the cache (-1: out of range)
    volatile int abort_flag;
    int s_ok_x, s_ok_o;              // results of the two global waits of a layer (one slot each)
    alignas(16) float h[D];          // normalised activation of the current phase (read as float4)
    alignas(16) float res[MAX_ROWS]; // dot products of the current phase
    float coef[MAX_ROWS];            // scale of each row in the scaled-row phases
    float wsum[NCW];
    float wmax[NCW];
    alignas(16) float qkv_s[512];         // the group's q head 2g | q head 2g+1 | k | v, pushed by the peers
    alignas(16) float part_o[CL][ODIMS];  // attention outputs of my 32 dims from each peer (unnormalised)
    alignas(16) float part_ml[CL][4];     // (max, sum) of both heads from each peer
    alignas(16) float red_o[CL][OWN];     // o_proj partials of my 128 outputs from each peer
    alignas(16) float red_d[CL][OWN];     // down_proj partials of my 128 outputs from each peer
    // rotated queries, pre-scaled to log2 units: dim 8 u + 4 h + e of head hh at q[hh][h][u][e], so
    // that the float4 reads of 8 different chunks u hit 8 different bank groups
    alignas(16) float q[2][2][HD / 8][4];
    alignas(16) uint16_t kn_b[HD];   // the new key and value as bf16 (as the cache holds them)
    alignas(16) uint16_t vn_b[HD];
    alignas(16) float wo[NCW][2][HD];  // attention: each warp's weighted values of both heads
    float wml[NCW][4];                 // each warp's (max, sum) of both heads
    float lm_val[NCW];
    int lm_idx[NCW];
    int last_cta;
};
constexpr int SMEM_BYTES = NS * STAGE + 1024 + (int)sizeof(Smem);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// Phase-boundary timestamp (tracing builds of a step only).
QW_DEV void stamp(const Params& p, int l, int k) {
    if (p.trace) p.trace[((size_t)blockIdx.x * (p.n_layers + 1) + l) * TRACE_SLOTS + k] = gtimer();
}

QW_DEV void give_up(const Params& p, Smem& sm) {
    set_error(p.err, QW_ETIMEOUT);
    sm.abort_flag = 1;
    atomicExch(c_abort(p), 1u);
}

// Bounded wait of one warp for `n` counters (lane i polls first + i * CNT_STRIDE) to reach
// `target`; warp-uniform result, false on timeout or abort.
__device__ __noinline__ bool wait_counters(const Params& p, const unsigned* first, int n, unsigned target, Smem& sm) {
    const int lane = threadIdx.x & 31;
    const unsigned* ptr = first + (lane < n ? lane : 0) * CNT_STRIDE;
    auto done = [&]() { return __all_sync(0xffffffffu, lane >= n || (int)(ld_acquire(ptr) - target) >= 0); };
    if (done()) return true;
    const uint64_t t0 = gtimer();
    for (unsigned i = 0;; ++i) {
        if (done()) return true;
        if ((i & 63) == 63) {
            int bad = 0;
            if (lane == 0) bad = sm.abort_flag || ld_acquire(c_abort(p)) != 0 || gtimer() - t0 > p.wait_ns;
            if (__shfl_sync(0xffffffffu, bad, 0)) {
                if (lane == 0 && !sm.abort_flag) give_up(p, sm);
                return false;
            }
        }
    }
}

// Bounded wait for phase `parity` of a cluster-exchange mbarrier: lane 0 of each calling warp
// polls (one poller per warp, not 32), __syncwarp orders the other lanes after its acquire.
__device__ __noinline__ bool wait_cluster(const Params& p, uint64_t* bar, uint32_t parity, Smem& sm) {
    int good = 1;
    if ((threadIdx.x & 31) == 0 && !mbar_test_wait_cluster(bar, parity)) {
        const uint64_t t0 = gtimer();
        for (unsigned i = 0;; ++i) {
            if (mbar_test_wait_cluster(bar, parity) || mbar_try_wait_cluster(bar, parity)) break;
            if ((i & 63) == 63) {
                if (sm.abort_flag || ld_acquire(c_abort(p)) != 0) {
                    good = 0;
                    break;
                }
                if (gtimer() - t0 > p.wait_ns) {
                    give_up(p, sm);
                    good = 0;
                    break;
                }
            }
        }
    }
    good = __shfl_sync(0xffffffffu, good, 0);
    __syncwarp();
    return good != 0;
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
    int cid, rank;     // cluster and rank in it
    bool attn;         // the cluster owns KV group g = cid
    int qrow0;         // first of this CTA's 64 q|k|v rows
    int j0;            // first of this CTA's 32 attention dims (rows of Wo^T)
    int pg_lo, pg_hi;  // pages of this CTA's share of the cache
    bool has_new;      // that share holds the new token's page
    int p0, p1;        // SwiGLU units (gate/up row pairs, rows of Wd^T)
    int v0, v1;        // LM-head rows
};

QW_DEV Work make_work(const Params& p, int pos, bool bad_pos) {
    Work w;
    const int G = gridDim.x, c = blockIdx.x;
    w.cid = (int)cluster_id();
    w.rank = (int)cluster_rank();
    w.attn = w.cid < HKV;
    const int g = w.cid, r = w.rank;
    // q head 2g: ranks 0,1; q head 2g+1: ranks 2,3; k head g: ranks 4,5; v head g: ranks 6,7
    w.qrow0 = r < 4 ? 256 * g + 64 * r : (r < 6 ? 2048 + 128 * g + 64 * (r - 4) : 3072 + 128 * g + 64 * (r - 6));
    w.j0 = 256 * g + ODIMS * r;
    if (bad_pos) pos = 0;
    const int np = pos / QW_PAGE_SIZE + 1;  // pages holding positions 0..pos
    w.pg_lo = (int)((long)np * r / CL);
    w.pg_hi = (int)((long)np * (r + 1) / CL);
    w.has_new = (pos / QW_PAGE_SIZE) >= w.pg_lo && (pos / QW_PAGE_SIZE) < w.pg_hi;
    w.p0 = slice_lo(INTER, c, G);
    w.p1 = slice_lo(INTER, c + 1, G);
    w.v0 = slice_lo(p.V, c, G);
    w.v1 = slice_lo(p.V, c + 1, G);
    return w;
}

// ---------------------------------------------------------------- producer
// The stages a CTA streams, in consumption order.  Layer l (attention CTAs): part 0 its q|k|v
// rows, part 1 its KV pages, part 2 its Wo^T rows; every CTA: part 3 its gate/up row pairs,
// part 4 its Wd^T rows.  After the last layer, part 5: its LM-head rows.
struct Seq {
    int l = 0, part = 0, i = 0;   // layer, part, stage within the part
};
struct StageDesc {
    const uint8_t* rows;    // row stages: first row
    int n;                  // rows, or pages
    int pg0;                // page stages: index of the first page in this CTA's page list
    int l;                  // page stages: layer
    bool pages;
};

template <bool Q8>
struct Producer {
    static constexpr int RB = row_bytes<Q8>(), RPS = rows_per_stage<Q8>();
    uint8_t* ring;
    Smem* sm;
    const Params* p;
    const Work* w;
    bool bad_pos;
    unsigned it = 0;
    bool stop = false;
    Seq ld, pf;               // next stage to load into the ring / to prefetch into L2
    unsigned pf_count = NS;   // index of the stage pf points at (the first NS stages load directly)

    // The stage at q (advancing q); false past the end.
    QW_DEV bool next(Seq& q, StageDesc& d) const {
        for (;;) {
            if (q.l > p->n_layers) return false;
            const int part = q.l == p->n_layers ? 5 : q.part;
            const uint8_t* base = nullptr;
            int total = 0;
            bool pages = false;
            if (part == 5) {
                base = p->E + (size_t)w->v0 * RB;
                total = w->v1 - w->v0;
            } else if (part <= 2 && !w->attn) {
                total = 0;
            } else {
                const LayerPtrs& L = p->layers[q.l];
                if (part == 0) base = L.wqkv + (size_t)w->qrow0 * RB, total = QROWS;
                else if (part == 1) pages = true, total = bad_pos ? 0 : w->pg_hi - w->pg_lo;
                else if (part == 2) base = L.woT + (size_t)w->j0 * RB, total = ODIMS;
                else if (part == 3) base = L.wgu + (size_t)2 * w->p0 * RB, total = 2 * (w->p1 - w->p0);
                else base = L.wdT + (size_t)w->p0 * RB, total = w->p1 - w->p0;
            }
            const int per = pages ? PAGES_PER_STAGE : RPS;
            if (q.i * per < total) {
                d.pages = pages;
                d.l = q.l;
                d.n = min(per, total - q.i * per);
                d.pg0 = q.i * per;
                d.rows = pages ? nullptr : base + (size_t)q.i * per * RB;
                ++q.i;
                return true;
            }
            q.i = 0;
            if (part == 5 || ++q.part == 5) {
                q.part = 0;
                ++q.l;
            }
        }
    }
    QW_DEV const uint16_t* page_ptr(int l, int idx, int which) const {
        const int pg = sm->pages[idx];
        return p->kv + (int64_t)l * p->layer_elems + (int64_t)pg * p->page_elems +
               ((int64_t)which * HKV + w->cid) * QW_PAGE_SIZE * HD;
    }
    QW_DEV bool acquire(int& s) {
        s = it % NS;
        const uint32_t ph = (it / NS) & 1;
        if (mbar_test_wait(&sm->empty[s], ph ^ 1)) return true;
        for (uint32_t i = 0; i < QW_SPIN_LIMIT; ++i) {
            if (mbar_try_wait(&sm->empty[s], ph ^ 1)) return true;
            if ((i & 63) == 63 && (sm->abort_flag || ld_acquire(c_abort(*p)) != 0)) return false;
            if (i > 64) __nanosleep(64);
        }
        give_up(*p, *sm);
        return false;
    }
    // L2 prefetch of the stages up to index `upto`: HBM streams at the pace of consumption,
    // PF stages ahead of the ring, and the ring loads then hit L2.
    QW_DEV void prefetch_until(unsigned upto) {
        StageDesc d;
        while (pf_count <= upto && next(pf, d)) {
            ++pf_count;
            if (!d.pages) {
                prefetch_l2(d.rows, d.n * RB);
            } else {
                for (int i = 0; i < d.n; ++i) {
                    if (sm->pages[d.pg0 + i] < 0) continue;
                    prefetch_l2(page_ptr(d.l, d.pg0 + i, 0), PAGE_B);
                    prefetch_l2(page_ptr(d.l, d.pg0 + i, 1), PAGE_B);
                }
            }
        }
    }
    // Stream every stage through the ring.
    QW_DEV void run() {
        StageDesc d;
        while (!stop && next(ld, d)) {
            prefetch_until(it + NS + PF - 1);
            int s;
            if (!acquire(s)) {
                stop = true;
                return;
            }
            if (!d.pages) {
                mbar_arrive_expect_tx(&sm->full[s], d.n * RB);
                bulk_load(ring + s * STAGE, d.rows, d.n * RB, &sm->full[s]);
            } else {
                // page i of a stage holds K at i * 8 KB and V at i * 8 KB + 4 KB
                int valid = 0;
                for (int i = 0; i < PAGES_PER_STAGE; ++i) {
                    const int pg = i < d.n ? sm->pages[d.pg0 + i] : -1;
                    valid += pg >= 0;
                    sm->spg[s][i] = pg;  // published to the consumers by the arrive below
                }
                mbar_arrive_expect_tx(&sm->full[s], valid * 2 * PAGE_B);
                for (int i = 0; i < d.n; ++i) {
                    if (sm->pages[d.pg0 + i] < 0) continue;
                    bulk_load(ring + s * STAGE + i * 2 * PAGE_B, page_ptr(d.l, d.pg0 + i, 0), PAGE_B, &sm->full[s]);
                    bulk_load(ring + s * STAGE + i * 2 * PAGE_B + PAGE_B, page_ptr(d.l, d.pg0 + i, 1), PAGE_B,
                              &sm->full[s]);
                }
            }
            ++it;
        }
    }
    // Before the CTA exits: every copy issued must have landed.
    QW_DEV void drain() {
        const unsigned first = it > (unsigned)NS ? it - NS : 0;
        for (unsigned i = first; i < it; ++i) mbar_wait(&sm->full[i % NS], (i / NS) & 1, p->err);
    }
};

// ---------------------------------------------------------------- consumer helpers
QW_DEV uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
QW_DEV void unpack2(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
QW_DEV float hsum2(uint64_t v) {
    float lo, hi;
    unpack2(v, lo, hi);
    return lo + hi;
}
// acc.{lo,hi} += a.{lo,hi} * b.{lo,hi} (packed fp32, the rounding of two fmaf)
QW_DEV void ffma2(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// acc.{lo,hi} += b.{lo,hi}
QW_DEV void add2(uint64_t& acc, uint64_t b) {
    float a0, a1, b0, b1;
    unpack2(acc, a0, a1);
    unpack2(b, b0, b1);
    acc = pack2(a0 + b0, a1 + b1);
}
// a bf16 pair (low element in the low half) as packed fp32
QW_DEV uint64_t bf2_to_f2(uint32_t w) { return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)); }

// int32 d = c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (dp2a.lo) or bytes 2, 3 (dp2a.hi), signed
QW_DEV int dp2a_lo(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
QW_DEV int dp2a_hi(int a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Two values rounded to int16 (round half to even, clamped) packed low, high.
QW_DEV int pack_i16(float a, float b) {
    const int ia = max(-32767, min(32767, __float2int_rn(a)));
    const int ib = max(-32767, min(32767, __float2int_rn(b)));
    return (ia & 0xFFFF) | (ib << 16);
}
// Transposed butterfly over the warp: v[k] (k < n, n a power of two <= 8) of every lane in, on
// return lanes with (lane >> (5 - log2 n)) == k hold the warp sum of value k.
template <int N>
QW_DEV float warp_reduce_n(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16, n = N; n > 1; o >>= 1, n >>= 1) {
        const bool up = lane & o;
#pragma unroll
        for (int k = 0; k < n / 2; ++k) {
            const float send = up ? v[k] : v[k + n / 2];
            v[k] = (up ? v[k + n / 2] : v[k]) + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (int o = 16 / N; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    return v[0];
}

template <bool Q8>
struct Consumer {
    static constexpr int RB = row_bytes<Q8>(), RPS = rows_per_stage<Q8>();
    uint8_t* ring;
    Smem* sm;
    int* err;
    int cw, lane;   // consumer warp 0..7, lane
    unsigned it = 0;

    // One lane of the warp waits for the stage (256 threads polling one mbarrier serialise on
    // it); __syncwarp then orders the other lanes' reads of the stage after that acquire.
    QW_DEV const uint8_t* stage_wait(bool& ok) {
        const int s = it % NS;
        int good = ok;
        if (lane == 0) good = good && !sm->abort_flag && mbar_wait(&sm->full[s], (it / NS) & 1, err);
        ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        __syncwarp();
        if (!ok) sm->abort_flag = 1;
        return ring + s * STAGE;
    }
    QW_DEV int slot() const { return it % NS; }
    // Wait for the next n (<= NS) stages at once: lane k tests stage it + k, so one round of
    // mbarrier tests covers the whole phase; the stages are then read at ring + ((it + k) % NS) *
    // STAGE and handed back one by one.  Returns the first stage.
    QW_DEV const uint8_t* phase_wait(int n, bool& ok) {
        const unsigned k = it + lane;
        bool ready = lane >= n || mbar_test_wait(&sm->full[k % NS], (k / NS) & 1);
        if (!__all_sync(0xffffffffu, ready)) {
            int good = ok;
            if (lane < n) good = good && mbar_wait(&sm->full[k % NS], (k / NS) & 1, err);
            ok = __all_sync(0xffffffffu, good != 0);
        }
        __syncwarp();
        if (!ok || sm->abort_flag) {
            ok = false;
            sm->abort_flag = 1;
        }
        return ring + (it % NS) * STAGE;
    }
    // Done with the current stage: hand its slot back to the producer.
    QW_DEV void stage_release() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[it % NS]);
        ++it;
    }
    // Dot products of `nrows` (at most 64, so at most 4 stages) streamed rows with sm->h.  Warp cw
    // takes rows 2 cw and 2 cw + 1 of every stage; lane l keeps one packed fp32 partial per row over
    // its columns 8 l + 256 i .. + 7 (i < 4) for the whole phase, and the warp reduces its 8 rows
    // once at the end with a transposed butterfly (each exchange halves the values a lane carries:
    // 9 shuffles for 8 rows), so nothing but the stage barrier separates the stages.  On return,
    // lanes 4 k .. 4 k + 3 hold the sum of the warp's row k, which is row 16 (k >> 1) + 2 cw + (k & 1)
    // of the phase (rows past nrows give 0).
    QW_DEV float dot_rows(int nrows, bool& ok) {
        uint64_t h2[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 a = *(const float4*)&sm->h[8 * lane + 256 * i];
            const float4 b = *(const float4*)&sm->h[8 * lane + 256 * i + 4];
            h2[i][0] = pack2(a.x, a.y);
            h2[i][1] = pack2(a.z, a.w);
            h2[i][2] = pack2(b.x, b.y);
            h2[i][3] = pack2(b.z, b.w);
        }
        uint64_t acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0;
        const int nst = (nrows + RPS - 1) / RPS;
        const uint8_t* st0 = phase_wait(nst, ok);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            if (s < nst) {
                const int n = min(RPS, nrows - RPS * s);
                const uint8_t* st = ring + ((it + s) % NS) * STAGE;
                if (ok) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int r = 2 * cw + j;
                        if (r < n) {
                            const uint4* ra = (const uint4*)(st + r * RB);
                            uint4 wa[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) wa[i] = ra[lane + 32 * i];
                            uint64_t a1 = 0;
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                ffma2(acc[2 * s + j], h2[i][0], bf2_to_f2(wa[i].x));
                                ffma2(a1, h2[i][1], bf2_to_f2(wa[i].y));
                                ffma2(acc[2 * s + j], h2[i][2], bf2_to_f2(wa[i].z));
                                ffma2(a1, h2[i][3], bf2_to_f2(wa[i].w));
                            }
                            add2(acc[2 * s + j], a1);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm->empty[(it + s) % NS]);
            }
        }
        (void)st0;
        it += nst;
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = hsum2(acc[k]);
        return warp_reduce_n<8>(v);
    }
    // Phase row of the value dot_rows leaves in this lane (lanes 4 k .. 4 k + 3 hold warp row k):
    // bf16 row 16 (k >> 1) + 2 cw + (k & 1), int8 row 32 (k >> 2) + 4 cw + (k & 3).  Gate and up
    // of a SwiGLU unit (rows 2u, 2u + 1) sit in lanes 4 apart either way.
    QW_DEV int lane_row() const {
        const int k = lane >> 2;
        return Q8 ? 32 * (k >> 2) + 4 * cw + (k & 3) : 16 * (k >> 1) + 2 * cw + (k & 1);
    }
    // int8 rows (32 per stage, at most 2 stages): warp cw takes rows 4 cw .. 4 cw + 3 of every
    // stage; lane l multiplies columns 16 l + 512 i .. + 15 (i < 2) with the activations rounded
    // to int16 (h * hinv) by dp2a, exact in int32 (at most 32 * 127 * 32767 per lane and row).
    // The result is in units of 1 / hinv (times the row's scale, applied by the caller).
    QW_DEV float dot_rows_q8(int nrows, bool& ok, float hinv) {
        int hq[16];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) {
                const float4 a = *(const float4*)&sm->h[16 * lane + 512 * i + 4 * m4];
                hq[8 * i + 2 * m4] = pack_i16(a.x * hinv, a.y * hinv);
                hq[8 * i + 2 * m4 + 1] = pack_i16(a.z * hinv, a.w * hinv);
            }
        int acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0;
        const int nst = (nrows + RPS - 1) / RPS;
        phase_wait(nst, ok);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (s < nst) {
                const int n = min(RPS, nrows - RPS * s);
                const uint8_t* st = ring + ((it + s) % NS) * STAGE;
                if (ok) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = 4 * cw + j;
                        if (r < n) {
                            int a = acc[4 * s + j];
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const uint4 w = *(const uint4*)(st + r * RB + 16 * lane + 512 * i);
                                a = dp2a_lo(hq[8 * i + 0], w.x, a);
                                a = dp2a_hi(hq[8 * i + 1], w.x, a);
                                a = dp2a_lo(hq[8 * i + 2], w.y, a);
                                a = dp2a_hi(hq[8 * i + 3], w.y, a);
                                a = dp2a_lo(hq[8 * i + 4], w.z, a);
                                a = dp2a_hi(hq[8 * i + 5], w.z, a);
                                a = dp2a_lo(hq[8 * i + 6], w.w, a);
                                a = dp2a_hi(hq[8 * i + 7], w.w, a);
                            }
                            acc[4 * s + j] = a;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm->empty[(it + s) % NS]);
            }
        }
        it += nst;
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (float)acc[k];
        return warp_reduce_n<8>(v);
    }
    // acc (columns 128 cw + 4 lane .. + 3) += sum over the int8 rows r (at most 32, one stage)
    // of sm->coef[r] * code[r][col]: the coefficients rounded to int16 on a step of max|coef| /
    // 32767, rows taken in pairs (a byte permute interleaves two rows' codes for dp2a), exact
    // int32 sums scaled back by the step.  The output channel's scale is applied later.
    QW_DEV bool scaled_rows_q8(int nrows, float (&acc)[4], bool ok) {
        float cm = 0.f;
        for (int r = 0; r < nrows; ++r) cm = fmaxf(cm, fabsf(sm->coef[r]));
        const float cinv = cm > 0.f ? 32767.0f / cm : 0.f, cstep = cm / 32767.0f;
        phase_wait(1, ok);
        int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
        const uint8_t* col = ring + (it % NS) * STAGE + 128 * cw + 4 * lane;
        if (ok) {
#pragma unroll
            for (int r = 0; r < RPS; r += 2) {
                if (r < nrows) {
                    const bool two = r + 1 < nrows;
                    const uint32_t A = *(const uint32_t*)(col + r * RB);
                    const uint32_t B = two ? *(const uint32_t*)(col + (r + 1) * RB) : 0u;
                    const int cp = pack_i16(sm->coef[r] * cinv, two ? sm->coef[r + 1] * cinv : 0.f);
                    const uint32_t P0 = __byte_perm(A, B, 0x5140), P1 = __byte_perm(A, B, 0x7362);
                    a0 = dp2a_lo(cp, P0, a0);
                    a1 = dp2a_hi(cp, P0, a1);
                    a2 = dp2a_lo(cp, P1, a2);
                    a3 = dp2a_hi(cp, P1, a3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[it % NS]);
        ++it;
        acc[0] += (float)a0 * cstep;
        acc[1] += (float)a1 * cstep;
        acc[2] += (float)a2 * cstep;
        acc[3] += (float)a3 * cstep;
        return ok;
    }
    // acc (columns 128 cw + 4 lane .. +3) += sum over streamed rows r of sm->coef[r] * row_r.
    // Each warp covers its own 128 output columns of every row, so no cross-warp sum is needed.
    QW_DEV bool scaled_rows(int nrows, float (&acc)[4], bool ok) {
        const int nst = (nrows + RPS - 1) / RPS;   // at most 2 (host-checked)
        phase_wait(nst, ok);
        uint64_t c01 = pack2(acc[0], acc[1]), c23 = pack2(acc[2], acc[3]), d01 = 0, d23 = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (s < nst) {
                const int n = min(RPS, nrows - RPS * s);
                const uint8_t* col = ring + ((it + s) % NS) * STAGE + (128 * cw + 4 * lane) * 2;
                const float* cf = sm->coef + RPS * s;
                if (ok) {
                    // two accumulator pairs (even and odd rows) halve the dependent FMA chain
#pragma unroll
                    for (int r = 0; r < RPS; r += 2) {
                        if (r < n) {
                            const uint2 wv = *(const uint2*)(col + r * RB);
                            const uint64_t aa = pack2(cf[r], cf[r]);
                            ffma2(c01, aa, bf2_to_f2(wv.x));
                            ffma2(c23, aa, bf2_to_f2(wv.y));
                        }
                        if (r + 1 < n) {
                            const uint2 wv = *(const uint2*)(col + (r + 1) * RB);
                            const uint64_t aa = pack2(cf[r + 1], cf[r + 1]);
                            ffma2(d01, aa, bf2_to_f2(wv.x));
                            ffma2(d23, aa, bf2_to_f2(wv.y));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm->empty[(it + s) % NS]);
            }
        }
        it += nst;
        add2(c01, d01);
        add2(c23, d23);
        unpack2(c01, acc[0], acc[1]);
        unpack2(c23, acc[2], acc[3]);
        return ok;
    }
};

// x (4 entries per consumer thread) -> sm.h = x * w, w = this thread's 4 norm weights (loaded
// ahead, so no global load sits on the critical path); returns 1 / rms(x), by which the products
// with sm.h are scaled.  One consumer barrier inside.
QW_DEV float norm_into_h(Smem& sm, const float (&x)[4], int k0, const float4 w, float eps, int tid, float& hmax) {
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    const float4 h = make_float4(x[0] * w.x, x[1] * w.y, x[2] * w.z, x[3] * w.w);
    float hm = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
    ss = warp_sum(ss);
    hm = warp_max(hm);
    if ((tid & 31) == 0) {
        sm.wsum[tid >> 5] = ss;
        sm.wmax[tid >> 5] = hm;
    }
    *(float4*)&sm.h[k0] = h;
    bar_consumers();
    float tot = 0.f;
    hmax = 0.f;
#pragma unroll
    for (int i = 0; i < NCW; ++i) {
        tot += sm.wsum[i];
        hmax = fmaxf(hmax, sm.wmax[i]);
    }
    return 1.0f / sqrtf(tot / (float)D + eps);
}

// Cluster reduction of one 1024-wide partial per CTA: this thread's 4 columns (128 cw + 4 lane)
// go to peer cw, which owns outputs [128 cw, 128 cw + 128).
QW_DEV void push_partial(Smem& sm, float (&red)[CL][OWN], uint64_t* bar, const float (&acc)[4], int cw, int lane,
                         int rank) {
    push4(peer_addr(&red[rank][4 * lane], cw), make_float4(acc[0], acc[1], acc[2], acc[3]), peer_addr(bar, cw));
}

// Sum of the 8 peers' partials of this CTA's outputs (fixed order) into dst[128 rank + ..]:
// threads 0..31 of the consumers, one float4 each.
QW_DEV void store_reduced(const float (&red)[CL][OWN], float* dst, int rank, int tid, float4 oscale) {
    if (tid < OWN / 4) {
        float4 t = *(const float4*)&red[0][4 * tid];
#pragma unroll
        for (int s = 1; s < CL; ++s) {
            const float4 v = *(const float4*)&red[s][4 * tid];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        t.x *= oscale.x;
        t.y *= oscale.y;
        t.z *= oscale.z;
        t.w *= oscale.w;
        *(float4*)(dst + OWN * rank + 4 * tid) = t;
    }
}

// x += sum over n slots of [n][D] at entries k0 .. k0+3 (fixed order; loads in flight together)
QW_DEV void add_slots(float (&x)[4], const float* base, int n, int k0) {
    float4 v[MAX_CLUSTERS];
#pragma unroll
    for (int s = 0; s < MAX_CLUSTERS; ++s)
        if (s < n) v[s] = __ldcg((const float4*)(base + (size_t)s * D + k0));
#pragma unroll
    for (int s = 0; s < MAX_CLUSTERS; ++s)
        if (s < n) {
            x[0] += v[s].x;
            x[1] += v[s].y;
            x[2] += v[s].z;
            x[3] += v[s].w;
        }
}

template <bool Q8>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) fused_decode_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Smem& sm = *(Smem*)(ring + NS * STAGE);
    const int G = gridDim.x, c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = p.positions[0];
    const int tok = p.tokens[0];
    // a position outside the block table, or a share of the cache longer than the page list
    // (the host takes this kernel only for block tables of at most CL * MAX_PAGES pages)
    const bool bad_pos = pos < 0 || pos >= p.bt_stride * QW_PAGE_SIZE || pos / QW_PAGE_SIZE >= CL * MAX_PAGES - CL;
    const Work w = make_work(p, pos, bad_pos);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], NCW);
        }
        mbar_init(&sm.bar_qkv, 1);
        mbar_init(&sm.bar_part, 1);
        mbar_init(&sm.bar_redo, 1);
        mbar_init(&sm.bar_redd, 1);
        // phase 0 of each exchange: the bytes the peers will push in layer 0
        if (w.attn) {
            mbar_arrive_expect_tx(&sm.bar_qkv, QKV_BYTES);
            mbar_arrive_expect_tx(&sm.bar_part, PART_BYTES);
            mbar_arrive_expect_tx(&sm.bar_redo, RED_BYTES);
        }
        mbar_arrive_expect_tx(&sm.bar_redd, RED_BYTES);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    // every peer's barriers exist before anyone pushes into them
    cluster_sync_all();
    const unsigned epoch = ld_acquire(c_epoch(p)) + 1;  // this launch's targets are epoch * amount
    if (bad_pos && c == 0 && threadIdx.x == 0) set_error(p.err, QW_ERANGE);

    if (warp == 0) {
        // ------------------------------------------------ producer
        // this CTA's page ids, read once for every layer (out-of-range ids become -1 and are reported)
        if (w.attn && !bad_pos)
            for (int i = lane; i < w.pg_hi - w.pg_lo; i += 32) {
                int pg = __ldg(p.bt + w.pg_lo + i);
                if (pg < 0 || pg >= p.n_pages) {
                    set_error(p.err, QW_ERANGE);
                    pg = -1;
                }
                sm.pages[i] = pg;
            }
        __syncwarp();
        if (lane == 0) {
            Producer<Q8> pr{ring, &sm, &p, &w, bad_pos};
            pr.run();
            pr.drain();
        }
        __syncwarp();
        cluster_sync_all();   // no peer pushes into this CTA's shared memory after it exits
        return;
    }

    // ------------------------------------------------ consumers (warps 1..8)
    const int tid = threadIdx.x - 32;  // 0..255
    const int cw = tid >> 5;
    Consumer<Q8> cs{ring, &sm, p.err, cw, lane};
    bool ok = !bad_pos;
    const int k0 = 4 * tid;  // this thread's 4 residual entries
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
    const int NC = p.n_clusters;
    const int g = w.cid, r = w.rank;

    // this thread's entries of the residual stream: x before the layer (xa), after attention (xm)
    float xa[4], xm[4];
    {
        const bool tok_ok = tok >= 0 && tok < p.V;
        if constexpr (Q8) {
            const uint32_t e = tok_ok ? *(const uint32_t*)(p.E + (size_t)tok * D + k0) : 0u;
            const float sc = tok_ok ? p.s_E[tok] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) xa[i] = (float)(int8_t)(e >> (8 * i)) * sc;
        } else {
            const uint2 e = tok_ok ? *(const uint2*)(p.E + ((size_t)tok * D + k0) * 2) : make_uint2(0, 0);
            xa[0] = bf16_lo(e.x); xa[1] = bf16_hi(e.x); xa[2] = bf16_lo(e.y); xa[3] = bf16_hi(e.y);
        }
        if (c == 0 && tid == 0 && !(tok >= 0 && tok < p.V)) set_error(p.err, QW_ERANGE);
    }

    // RoPE rotation of this lane's two pairs (dims lane + 32 j and + 64) at this step's
    // position: the same in every layer, so computed once per step
    float rs[2], rc[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) sincosf(__fmul_rn((float)pos, p.inv_freq[lane + 32 * j]), &rs[j], &rc[j]);
    for (int l = 0; l < p.n_layers; ++l) {
        // this layer's small vectors, loaded before the waits so their latency hides behind them
        const LayerPtrs L = p.layers[l];
        const float4 w_in = __ldg((const float4*)(L.in_norm + k0));
        const float4 w_post = __ldg((const float4*)(L.post_norm + k0));
        float w_qk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w_qk[i] = __ldg((cw < 2 ? L.q_norm : L.k_norm) + lane + 32 * i);
        // int8: the scales of this lane's q|k|v and gate/up rows and of the outputs this thread stores
        float s_row_qkv = 1.f, s_row_gu = 1.f;
        float4 s_out_o = make_float4(1.f, 1.f, 1.f, 1.f), s_out_d = s_out_o;
        if constexpr (Q8) {
            const int row = cs.lane_row();
            if (w.attn) s_row_qkv = __ldg(L.s_qkv + w.qrow0 + row);
            if (row < 2 * (w.p1 - w.p0)) s_row_gu = __ldg(L.s_gu + 2 * w.p0 + row);
            if (tid < OWN / 4) {
                if (w.attn) s_out_o = __ldg((const float4*)(L.s_o + OWN * w.rank + 4 * tid));
                s_out_d = __ldg((const float4*)(L.s_d + OWN * w.rank + 4 * tid));
            }
        }
        const int pb = l & 1;
        const uint32_t par = (uint32_t)(l & 1);
        const bool more = l + 1 < p.n_layers;
        // ---------------- layer input: x = x_mid of the previous layer + its cluster slots
        if (tid == 0) stamp(p, l, 0);
        if (l > 0) {
            if (cw == 0) {
                const bool good = ok && wait_counters(p, c_x(p, l - 1, 0), NC, epoch * CL, sm);
                if (lane == 0) sm.s_ok_x = good;
            }
            bar_consumers();
            ok = sm.s_ok_x;
            xa[0] = xm[0]; xa[1] = xm[1]; xa[2] = xm[2]; xa[3] = xm[3];
            add_slots(xa, p.dslot + (size_t)(pb ^ 1) * MAX_CLUSTERS * D, NC, k0);
        }
        if (tid == 0) stamp(p, l, 1);
        if (w.attn) {
            // ---------------- A1: norm -> this CTA's q|k|v rows -> every peer's qkv_s
            float hmax;
            const float s_in = norm_into_h(sm, xa, k0, w_in, p.eps, tid, hmax);
            {
                float v;
                if constexpr (Q8)
                    v = cs.dot_rows_q8(QROWS, ok, hmax > 0.f ? 32767.0f / hmax : 0.f) * (hmax / 32767.0f) * s_row_qkv;
                else
                    v = cs.dot_rows(QROWS, ok);
                if ((lane & 3) == 0) sm.res[cs.lane_row()] = v * s_in;
            }
            if (tid == 0) stamp(p, l, 2);
            bar_consumers();
            if (ok && tid < 16 * CL) {
                const int dst = tid >> 4, q4 = tid & 15;
                push4(peer_addr(&sm.qkv_s[QROWS * r + 4 * q4], dst), *(const float4*)&sm.res[4 * q4],
                      peer_addr(&sm.bar_qkv, dst));
            }
            ok = ok && wait_cluster(p, &sm.bar_qkv, par, sm);
            if (tid == 0) {
                if (ok && more) mbar_arrive_expect_tx(&sm.bar_qkv, QKV_BYTES);   // next layer's phase
                stamp(p, l, 3);
            }
            // ---------------- A2: QK-Norm, RoPE, cache write, attention over this CTA's pages
            if (cw < 4 && ok) {
                // warp 0,1: q heads 2g, 2g+1; warp 2: k head g; warp 3: v head g
                float y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = sm.qkv_s[HD * cw + lane + 32 * i];
                if (cw < 3) {
                    const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
                    const float sc = 1.0f / sqrtf(ss / (float)HD + p.eps);
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[i] = y[i] * sc * w_qk[i];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float sn = rs[j], cs_ = rc[j];
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
            // Each stage holds up to 4 pages (64 key slots); warp cw owns slots 8 cw .. 8 cw + 7 of
            // every stage and keeps its own running max, sum and weighted values per query head
            // (flash-decoding within the warp), so the key loop needs no CTA barrier; the 8 warps
            // merge once after it.  Scores: one key per 4-lane group (kg = lane >> 2); lane
            // dq = lane & 3 takes the 16-byte chunks u = 4 c' + dq, c' = c ^ (kg & 1), of the key
            // row (the xor puts the 8 lanes of each shared-memory phase on 8 different bank
            // groups).  P.V: lane takes dims 4 lane .. 4 lane + 3 of both heads.  The running sum
            // is kept per key group (the rescaling factor is the same in every lane) and summed
            // over the warp once, after the loop.
            const int kg = lane >> 2, dq = lane & 3;
            float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
            float orun[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int pg0 = w.pg_lo; pg0 < w.pg_hi && !bad_pos; pg0 += PAGES_PER_STAGE) {
                const int n = min(PAGES_PER_STAGE, w.pg_hi - pg0);
                const uint8_t* st = cs.stage_wait(ok);
                const int pi = cw >> 1, slot0 = 8 * (cw & 1);
                const bool page_ok = ok && pi < n && sm.spg[cs.slot()][pi] >= 0;
                const int kbase = (pg0 + pi) * QW_PAGE_SIZE + slot0;   // position of the warp's key 0
                const int kpos = kbase + kg;
                const bool vis = page_ok && kpos <= pos;
                const uint8_t* page = st + (pi < n ? pi : 0) * 2 * PAGE_B;
                // the new token's key and value come from the bf16 copies made above, not the stage
                const uint8_t* krow = kpos == pos ? (const uint8_t*)sm.kn_b : page + (slot0 + kg) * HD * 2;
                // this lane's dims of the 8 keys' values, read before the scores need them (rows of
                // invisible keys hold whatever the ring slot held; they are masked below)
                uint2 vv[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    vv[k] = kbase + k == pos ? *(const uint2*)((const uint8_t*)sm.vn_b + 8 * lane)
                                             : *(const uint2*)(page + PAGE_B + (slot0 + k) * HD * 2 + 8 * lane);
                float sc[2] = {0.f, 0.f};
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int u = 4 * (cc ^ (kg & 1)) + dq;
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
                float pe[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 1);
                    sc[hh] += __shfl_xor_sync(0xffffffffu, sc[hh], 2);
                    float mw = vis ? sc[hh] : -INFINITY;
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
                    const float mnew = fmaxf(mrun[hh], mw);
                    const float alpha = mrun[hh] == -INFINITY ? 0.f : exp2f(mrun[hh] - mnew);
                    pe[hh] = vis ? exp2f(sc[hh] - mnew) : 0.f;
                    lrun[hh] = lrun[hh] * alpha + pe[hh];
                    mrun[hh] = mnew;
#pragma unroll
                    for (int e = 0; e < 4; ++e) orun[hh][e] *= alpha;
                }
                // weights of the 8 keys first, then the products without branches: a key whose
                // weights are both 0 (invisible, or not in the stage) contributes a zero value
                float p0[8], p1[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    p0[k] = __shfl_sync(0xffffffffu, pe[0], 4 * k);
                    p1[k] = __shfl_sync(0xffffffffu, pe[1], 4 * k);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const bool used = p0[k] != 0.f || p1[k] != 0.f;
                    const uint2 v = used ? vv[k] : make_uint2(0u, 0u);
                    const float v0 = bf16_lo(v.x), v1 = bf16_hi(v.x), v2 = bf16_lo(v.y), v3 = bf16_hi(v.y);
                    orun[0][0] = fmaf(p0[k], v0, orun[0][0]);
                    orun[0][1] = fmaf(p0[k], v1, orun[0][1]);
                    orun[0][2] = fmaf(p0[k], v2, orun[0][2]);
                    orun[0][3] = fmaf(p0[k], v3, orun[0][3]);
                    orun[1][0] = fmaf(p1[k], v0, orun[1][0]);
                    orun[1][1] = fmaf(p1[k], v1, orun[1][1]);
                    orun[1][2] = fmaf(p1[k], v2, orun[1][2]);
                    orun[1][3] = fmaf(p1[k], v3, orun[1][3]);
                }
                cs.stage_release();
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) lrun[hh] += __shfl_xor_sync(0xffffffffu, lrun[hh], o);
            if (tid == 0) stamp(p, l, 4);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                *(float4*)&sm.wo[cw][hh][4 * lane] = make_float4(orun[hh][0], orun[hh][1], orun[hh][2], orun[hh][3]);
                if (lane == 0) {
                    sm.wml[cw][2 * hh] = mrun[hh];
                    sm.wml[cw][2 * hh + 1] = lrun[hh];
                }
            }
            bar_consumers();
            {
                // thread (head hh, dim d): merge of the 8 warps (their maxima differ), then this CTA's
                // partial; 4 consecutive dims go to their owner peer in one 16-byte push (owner of
                // group dim 128 hh + d is peer (128 hh + d) / 32)
                const int hh = tid >> 7, d = tid & 127;
                float M = -INFINITY;
#pragma unroll
                for (int i = 0; i < NCW; ++i)
                    if (sm.wml[i][2 * hh + 1] > 0.f) M = fmaxf(M, sm.wml[i][2 * hh]);
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int i = 0; i < NCW; ++i) {
                    const float li = sm.wml[i][2 * hh + 1];
                    const float f = li > 0.f ? exp2f(sm.wml[i][2 * hh] - M) : 0.f;
                    Ls += f * li;
                    O += f * sm.wo[i][hh][d];
                }
                const float o1 = __shfl_down_sync(0xffffffffu, O, 1);
                const float o2 = __shfl_down_sync(0xffffffffu, O, 2);
                const float o3 = __shfl_down_sync(0xffffffffu, O, 3);
                if (ok && (d & 3) == 0) {
                    const int dst = (HD * hh + d) / ODIMS;
                    push4(peer_addr(&sm.part_o[r][d % ODIMS], dst), make_float4(O, o1, o2, o3),
                          peer_addr(&sm.bar_part, dst));
                }
                if (ok && d < CL)   // (max, sum) of head hh to peer d
                    push2(peer_addr(&sm.part_ml[r][2 * hh], d), M, Ls, peer_addr(&sm.bar_part, d));
            }
            ok = ok && wait_cluster(p, &sm.bar_part, par, sm);
            if (tid == 0) {
                if (ok && more) mbar_arrive_expect_tx(&sm.bar_part, PART_BYTES);   // next layer's phase
                stamp(p, l, 5);
            }
            // ---------------- A3: merge my 32 dims, o_proj rows of Wo^T, cluster reduction
            if (cw == 0) {
                const int hh = r / 4;   // my dims are 32 (r % 4) .. + 31 of head 2g + hh
                float M = -INFINITY;
#pragma unroll
                for (int s = 0; s < CL; ++s)
                    if (sm.part_ml[s][2 * hh + 1] > 0.f) M = fmaxf(M, sm.part_ml[s][2 * hh]);
                float Lt = 0.f, Ot = 0.f;
#pragma unroll
                for (int s = 0; s < CL; ++s) {
                    const float Ls = sm.part_ml[s][2 * hh + 1];
                    const float f = Ls > 0.f ? exp2f(sm.part_ml[s][2 * hh] - M) : 0.f;
                    Lt += f * Ls;
                    Ot += f * sm.part_o[s][lane];
                }
                sm.coef[lane] = Lt > 0.f ? Ot / Lt : 0.f;
            }
            bar_consumers();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (Q8) ok = cs.scaled_rows_q8(ODIMS, acc, ok);
            else ok = cs.scaled_rows(ODIMS, acc, ok);
            if (tid == 0) stamp(p, l, 6);
            if (ok) push_partial(sm, sm.red_o, &sm.bar_redo, acc, cw, lane, r);
            ok = ok && wait_cluster(p, &sm.bar_redo, par, sm);
            if (tid == 0) {
                if (ok && more) mbar_arrive_expect_tx(&sm.bar_redo, RED_BYTES);   // next layer's phase
                stamp(p, l, 7);
            }
            // warp 0 stores this CTA's 128 outputs and publishes them (the warp barrier orders its
            // lanes' stores before lane 0's release); the other warps go straight on
            if (cw == 0) {
                if (ok) store_reduced(sm.red_o, p.oslot + ((size_t)pb * HKV + g) * D, r, tid, s_out_o);
                __syncwarp();
                if (lane == 0) {
                    signal_add(c_o(p, l, g), 1u);
                    stamp(p, l, 8);
                }
            }
        }
        // ---------------- M1: x + group slots -> norm -> gate/up -> SwiGLU -> down rows -> cluster slot
        if (tid == 0) stamp(p, l, 9);
        if (cw == 0) {
            const bool good = ok && wait_counters(p, c_o(p, l, 0), HKV, epoch * CL + (l == 0 ? p.fault_extra : 0u), sm);
            if (lane == 0) sm.s_ok_o = good;
        }
        bar_consumers();
        ok = sm.s_ok_o;
        xm[0] = xa[0]; xm[1] = xa[1]; xm[2] = xa[2]; xm[3] = xa[3];
        add_slots(xm, p.oslot + (size_t)pb * HKV * D, HKV, k0);
        if (tid == 0) stamp(p, l, 10);
        float hmax2;
        const float s_post = norm_into_h(sm, xm, k0, w_post, p.eps, tid, hmax2);
        if (tid == 0) stamp(p, l, 17);
        const int np2 = w.p1 - w.p0;
        {
            // rows 2 u, 2 u + 1 (gate, up of SwiGLU unit u = 8 (lane >> 3) + cw) sit in lanes 4 apart
            float v;
            if constexpr (Q8)
                v = cs.dot_rows_q8(2 * np2, ok, hmax2 > 0.f ? 32767.0f / hmax2 : 0.f) * (hmax2 / 32767.0f) * s_row_gu *
                    s_post;
            else
                v = cs.dot_rows(2 * np2, ok) * s_post;
            const float up = __shfl_xor_sync(0xffffffffu, v, 4);
            const int u = cs.lane_row() >> 1;
            if ((lane & 7) == 0 && u < np2) sm.coef[u] = v / (1.0f + expf(-v)) * up;
        }
        if (tid == 0) stamp(p, l, 11);
        bar_consumers();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (Q8) ok = cs.scaled_rows_q8(np2, acc, ok);
        else ok = cs.scaled_rows(np2, acc, ok);
        if (tid == 0) stamp(p, l, 12);
        if (ok) push_partial(sm, sm.red_d, &sm.bar_redd, acc, cw, lane, r);
        ok = ok && wait_cluster(p, &sm.bar_redd, par, sm);
        if (tid == 0) {
            if (ok && more) mbar_arrive_expect_tx(&sm.bar_redd, RED_BYTES);   // next layer's phase
            stamp(p, l, 13);
        }
        if (cw == 0) {
            if (ok) store_reduced(sm.red_d, p.dslot + ((size_t)pb * MAX_CLUSTERS + w.cid) * D, r, tid, s_out_d);
            __syncwarp();
            if (lane == 0) {
                signal_add(c_x(p, l, w.cid), 1u);
                stamp(p, l, 14);
            }
        }
    }
    // ---------------- LM head: final norm, tied embedding rows, argmax
    {
        const int pl = (p.n_layers - 1) & 1;
        const float4 w_fin = __ldg((const float4*)(p.final_norm + k0));
        if (tid == 0) stamp(p, p.n_layers, 0);
        if (cw == 0) {
            const bool good = ok && wait_counters(p, c_x(p, p.n_layers - 1, 0), NC, epoch * CL, sm);
            if (lane == 0) sm.s_ok_x = good;
        }
        bar_consumers();
        ok = sm.s_ok_x;
        if (tid == 0) stamp(p, p.n_layers, 1);
        float xf[4] = {xm[0], xm[1], xm[2], xm[3]};
        add_slots(xf, p.dslot + (size_t)pl * MAX_CLUSTERS * D, NC, k0);
        float hmaxf;
        const float s_fin = norm_into_h(sm, xf, k0, w_fin, p.eps, tid, hmaxf);
        float best = -INFINITY;
        int bidx = 0x7FFFFFFF;
        const int nv = w.v1 - w.v0;
        if constexpr (Q8) {
            // int8 rows, 32 per stage: warp cw takes rows 4 cw .. 4 cw + 3; dp2a on the activations
            // rounded to int16, then a transposed butterfly leaves row j in lanes 8 j .. 8 j + 7
            const float hinv = hmaxf > 0.f ? 32767.0f / hmaxf : 0.f, hstep = hmaxf / 32767.0f * s_fin;
            int hq[16];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int m4 = 0; m4 < 4; ++m4) {
                    const float4 a = *(const float4*)&sm.h[16 * lane + 512 * i + 4 * m4];
                    hq[8 * i + 2 * m4] = pack_i16(a.x * hinv, a.y * hinv);
                    hq[8 * i + 2 * m4 + 1] = pack_i16(a.z * hinv, a.w * hinv);
                }
            constexpr int RPS8 = rows_per_stage<true>();
            for (int r0 = 0; r0 < nv; r0 += RPS8) {
                const int n = min(RPS8, nv - r0);
                const int my = 4 * cw + (lane >> 3);   // the row this lane reports after the reduction
                const float sc = my < n ? __ldg(p.s_E + w.v0 + r0 + my) : 0.f;
                const uint8_t* st = cs.stage_wait(ok);
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (ok) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int rr = 4 * cw + j;
                        if (rr < n) {
                            int a = 0;
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const uint4 wv = *(const uint4*)(st + rr * D + 16 * lane + 512 * i);
                                a = dp2a_lo(hq[8 * i + 0], wv.x, a);
                                a = dp2a_hi(hq[8 * i + 1], wv.x, a);
                                a = dp2a_lo(hq[8 * i + 2], wv.y, a);
                                a = dp2a_hi(hq[8 * i + 3], wv.y, a);
                                a = dp2a_lo(hq[8 * i + 4], wv.z, a);
                                a = dp2a_hi(hq[8 * i + 5], wv.z, a);
                                a = dp2a_lo(hq[8 * i + 6], wv.w, a);
                                a = dp2a_hi(hq[8 * i + 7], wv.w, a);
                            }
                            v[j] = (float)a;
                        }
                    }
                }
                cs.stage_release();
                const float a = warp_reduce_n<4>(v) * hstep * sc;
                const int vid = w.v0 + r0 + my;
                if ((lane & 7) == 0 && my < n) {
                    p.logits[vid] = a;
                    if (a > best || (a == best && vid < bidx)) {
                        best = a;
                        bidx = vid;
                    }
                }
            }
            // lanes 0, 8, 16, 24 hold the warp's candidates
#pragma unroll
            for (int o = 8; o < 32; o <<= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
                if (ob > best || (ob == best && oi < bidx)) {
                    best = ob;
                    bidx = oi;
                }
            }
        } else {
            float hreg[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) hreg[i][e] = sm.h[8 * lane + 256 * i + e] * s_fin;
            constexpr int RPS16 = rows_per_stage<false>();
            for (int r0 = 0; r0 < nv; r0 += RPS16) {
                const int n = min(RPS16, nv - r0);
                const uint8_t* st = cs.stage_wait(ok);
                if (ok) {
                    for (int rr = cw; rr < n; rr += NCW) {
                        const uint4* row = (const uint4*)(st + rr * 2 * D);
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
            if (prev == epoch * G - 1) {
                // last CTA: global argmax (lowest id on ties), then the next step's epoch
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
                signal_add(c_epoch(p), 1u);
            }
        }
    }
    cluster_sync_all();   // no peer pushes into this CTA's shared memory after it exits
}

// Wt[j][i] = W[i][j] for a [rows][cols] matrix of bf16 (uint16_t) or int8 codes.
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ W, T* __restrict__ Wt, int rows, int cols) {
    __shared__ T tile[32][33];
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
    int G = 0, n_clusters = 0, n_layers = 0, V = 0;
    float eps = 0.f;
    uint8_t* buf = nullptr;
    fused::LayerPtrs* d_layers = nullptr;
    bool q8 = false;             // weight-only int8 rows (else bf16)
    const uint8_t* E = nullptr;
    const float* sE = nullptr;
    const float* final_norm = nullptr;
    const float* inv_freq = nullptr;
    float *oslot = nullptr, *dslot = nullptr, *lm_part = nullptr;
    int* argmax = nullptr;
    unsigned* sync = nullptr;
    size_t state_bytes = 0;   // bytes from oslot through the counters (cleared by fused_reset)
    unsigned long long* trace = nullptr;
    bool trace_on = false;
    bool fault_armed = false;   // the next launch waits for an arrival that never comes (test hook)
};

FusedDecode* fused_create(const FusedWeights& fw, int n_layers, int V, float eps, int hidden, int n_heads,
                          int n_kv_heads, int intermediate) {
    using namespace fused;
    if (hidden != D || n_heads != HQ || n_kv_heads != HKV || intermediate != INTER || n_layers > MAX_LAYERS) return nullptr;
    int dev = 0, coop = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (!coop) return nullptr;
    const bool q8 = fw.q8;
    auto kern = q8 ? fused_decode_kernel<true> : fused_decode_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
        return nullptr;
    // as many clusters of 8 as can be resident at once (15 on a 152-SM GB300); 8 own the KV groups
    int max_clusters = 0;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess) return nullptr;
    }
    const int nc = max_clusters < MAX_CLUSTERS ? max_clusters : MAX_CLUSTERS;
    if (nc < HKV) return nullptr;
    const int G = CL * nc;
    // a GEMV phase takes at most 64 rows (4 bf16 or 2 int8 stages), a scaled-row phase at most 32
    if (2 * ((INTER + G - 1) / G) > 64 || (INTER + G - 1) / G > 32 || ODIMS > 32) return nullptr;
    FusedDecode* f = new FusedDecode();
    f->G = G;
    f->n_clusters = nc;
    f->n_layers = n_layers;
    f->V = V;
    f->eps = eps;
    f->q8 = q8;
    f->E = q8 ? (const uint8_t*)fw.Eq : (const uint8_t*)fw.E;
    f->sE = q8 ? fw.sE : nullptr;
    f->final_norm = fw.final_norm;
    f->inv_freq = fw.inv_freq;
    const size_t woT = (size_t)AD * D, wdT = (size_t)INTER * D;
    size_t off = 0;
    auto take = [&](size_t b) {
        size_t o = off;
        off = (off + b + 1023) / 1024 * 1024;
        return o;
    };
    const size_t esz = q8 ? 1 : 2;   // bytes per weight element
    const size_t o_w = take((woT + wdT) * esz * n_layers);
    const size_t o_layers = take(sizeof(LayerPtrs) * n_layers);
    const size_t o_state = take(sizeof(float) * 2 * (HKV + MAX_CLUSTERS) * D);
    const size_t o_lm = take(sizeof(float) * 2 * G + 64);
    const size_t o_sync = take(sizeof(unsigned) * CNT_STRIDE * (3 + n_layers * CNT_PER_LAYER));
    const size_t o_trace = take(sizeof(unsigned long long) * G * (n_layers + 1) * TRACE_SLOTS);
    if (cudaMalloc(&f->buf, off) != cudaSuccess) {
        delete f;
        return nullptr;
    }
    std::vector<LayerPtrs> lp(n_layers);
    for (int l = 0; l < n_layers; ++l) {
        uint8_t* woT_l = f->buf + o_w + (size_t)l * (woT + wdT) * esz;
        uint8_t* wdT_l = woT_l + woT * esz;
        LayerPtrs& L = lp[l];
        L.in_norm = fw.in_norm[l];
        L.post_norm = fw.post_norm[l];
        L.q_norm = fw.q_norm[l];
        L.k_norm = fw.k_norm[l];
        L.woT = woT_l;
        L.wdT = wdT_l;
        if (q8) {
            transpose_kernel<int8_t><<<dim3(AD / 32, D / 32), dim3(32, 8)>>>(fw.wo_q[l], (int8_t*)woT_l, D, AD);
            transpose_kernel<int8_t><<<dim3(INTER / 32, D / 32), dim3(32, 8)>>>(fw.wd_q[l], (int8_t*)wdT_l, D, INTER);
            L.wqkv = (const uint8_t*)fw.wqkv_q[l];
            L.wgu = (const uint8_t*)fw.wgu_q[l];
            L.s_qkv = fw.s_qkv[l];
            L.s_o = fw.s_o[l];
            L.s_gu = fw.s_gu[l];
            L.s_d = fw.s_d[l];
        } else {
            transpose_kernel<uint16_t><<<dim3(AD / 32, D / 32), dim3(32, 8)>>>(fw.wo[l], (uint16_t*)woT_l, D, AD);
            transpose_kernel<uint16_t><<<dim3(INTER / 32, D / 32), dim3(32, 8)>>>(fw.wd[l], (uint16_t*)wdT_l, D, INTER);
            L.wqkv = (const uint8_t*)fw.wqkv[l];
            L.wgu = (const uint8_t*)fw.wgu[l];
            L.s_qkv = L.s_o = L.s_gu = L.s_d = nullptr;
        }
    }
    f->d_layers = (LayerPtrs*)(f->buf + o_layers);
    f->oslot = (float*)(f->buf + o_state);
    f->dslot = f->oslot + 2 * HKV * D;
    f->lm_part = (float*)(f->buf + o_lm);
    f->argmax = (int*)(f->lm_part + 2 * G);
    f->sync = (unsigned*)(f->buf + o_sync);
    f->state_bytes = o_trace - o_state;
    f->trace = (unsigned long long*)(f->buf + o_trace);
    if (cudaMemcpy(f->d_layers, lp.data(), sizeof(LayerPtrs) * n_layers, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(f->buf + o_state, 0, off - o_state) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(f->buf);
        delete f;
        return nullptr;
    }
    return f;
}

bool fused_supported(const FusedDecode* f, int batch, int bt_stride) {
    return f != nullptr && batch == 1 && bt_stride <= fused::CL * fused::MAX_PAGES - fused::CL;
}

int fused_reset(FusedDecode* f, cudaStream_t st) {
    // after a timeout the counters and slots are in an unknown state
    return cudaMemsetAsync(f->oslot, 0, f->state_bytes, st) == cudaSuccess ? QW_OK : QW_ECUDA;
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
    p.s_E = f->sE;
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
    p.oslot = f->oslot;
    p.dslot = f->dslot;
    p.lm_part = f->lm_part;
    p.argmax = f->argmax;
    p.sync = f->sync;
    p.err = err;
    p.n_clusters = f->n_clusters;
    p.trace = f->trace_on ? f->trace : nullptr;
    p.wait_ns = f->fault_armed ? FAULT_WAIT_NS : WAIT_NS;
    p.fault_extra = f->fault_armed ? 1u : 0u;
    f->fault_armed = false;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once: the counters are waited on
    at[0].val.cooperative = 1;
    cfg.gridDim = dim3(f->G);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const cudaError_t e = f->q8 ? cudaLaunchKernelEx(&cfg, fused_decode_kernel<true>, p)
                                : cudaLaunchKernelEx(&cfg, fused_decode_kernel<false>, p);
    count_launches(1);
    return e == cudaSuccess ? QW_OK : QW_ECUDA;
}

const int* fused_argmax(const FusedDecode* f) { return f ? f->argmax : nullptr; }

int fused_inject_timeout(FusedDecode* f) {
    if (!f) return QW_EINVAL;
    f->fault_armed = true;
    return QW_OK;
}

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
