// sample() of the article's Step 8 on the GPU, for any nucleus size.
//
// One cluster of 8 CTAs per row; CTA r of the cluster owns an eighth of the vocabulary.
// Greedy rows take the argmax (lowest id on ties), from the per-tile (max, argmax) partials
// the LM-head projection leaves when it has them.  Sampling rows work on
// e_i = exp((l_i - max) / T) and the order "logit descending, id ascending" without sorting:
// a position in that order is a pair (key K, n) -- every entry whose logit is above the one
// with order key K, then the n lowest-id entries with key K -- and each cut is found by a
// radix search over the 32-bit order keys, 8 bits per pass over the row:
//   top-k cut  the k-th entry                         (search by count)
//   top-p cut  the first entry where the cumulative
//              mass reaches top_p * Z                 (search by mass, Z = sum of e_i)
//   kept       the earlier of the two cuts; M = kept mass
//   draw       the first kept entry where the cumulative mass exceeds u * M
//              (u from Philox4x32-10, key = seed, counter = (rng_counter, 0, 0))
// Every pass builds per-warp histograms of the CTA's slice, adds them per CTA, and sums the
// 8 CTAs' histograms through distributed shared memory, so all 8 CTAs take the same bucket
// decisions.  Masses are summed in fp32 per bucket; the result equals the sorted-cumsum
// definition except when a cumulative sum lies within rounding of a cut, which the parity
// tests exempt.
#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace smp {

constexpr int CL = 8;            // CTAs per row (one cluster)
constexpr int THREADS = 256;
constexpr int NW = THREADS / 32;
constexpr int NB = 256;          // buckets per digit
constexpr int NH = 3;            // histograms per pass: count of search 0, count and mass of search 1

QW_DEV uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
QW_DEV float key_value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }

constexpr int FT = 1024, FNW = FT / 32, FNB = 2048, FCAP = 2048, FKMAX = 1024, FCL = 4;
constexpr int FUN = 4;   // float4 loads each thread keeps in flight in a pass over its part

struct FShared {
    uint32_t hist[FNB];
    float stats[3];   // this CTA's (max, min, Z relative to its max), read by the peers
    unsigned long long cand[FCAP];
    float e[FKMAX];
    float fred[FNW];
    float fred2[FNW];
    uint32_t ured[FNW];
    uint32_t ncand, bstar, cnt_star;
    int pick;
};

QW_DEV bool topk_row(const qw_sample_params& P, int vocab) {
    return P.temperature > 0.f && P.top_k >= 1 && P.top_k <= FKMAX && P.top_k < vocab && P.top_p > 0.f &&
           P.top_p <= 1.f;
}

struct Shared {
    uint32_t wcnt[NW][2][NB];     // per-warp counts of both searches
    float wmass[NW][NB];          // per-warp mass of the mass search
    float cta[NH][NB];            // this CTA's histograms (count as float, exact below 2^24)
    float sum[NH][NB];            // the cluster's histograms
    float scal[4], scal_sum[4];   // scalars summed over the cluster
    float red[NW];
    unsigned long long ured[NW];
    int ired[NW];
    uint32_t prefix[2], pmask[2], rem_c[2], cnt_key[2];
    float rem_m[2];
};

QW_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
QW_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
QW_DEV float ld_peer(const float* local, int rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

// Reduction over the CTA; `identity` fills the lanes past the number of warps.
template <typename T, typename Op>
QW_DEV T block_reduce(T v, Op op, T* scratch, T identity) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = lane < NW ? scratch[lane] : identity;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    return v;
}

// Histogram update by every lane of a warp (warp-uniform call) into the warp's own
// histograms: lanes with the same bucket combine their count first (one atomic per group);
// the mass takes one atomic per lane, or one per warp when all lanes share the bucket.
QW_DEV void hist_add(Shared& sh, int s, uint32_t b, float e, bool valid) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? b : NB);
    if (!valid) return;
    if (lane == __ffs(grp) - 1) atomicAdd(&sh.wcnt[w][s][b], (uint32_t)__popc(grp));
    if (s == 1) {
        if (grp == 0xffffffffu) {
            e = warp_sum(e);
            if (lane == 0) atomicAdd(&sh.wmass[w][b], e);
        } else {
            atomicAdd(&sh.wmass[w][b], e);
        }
    }
}

// Per-warp histograms -> this CTA's -> the cluster's (sh.sum), together with the scalars
// sh.scal; then the per-warp histograms are cleared for the next pass.  Cluster barriers inside.
QW_DEV void cluster_histograms(Shared& sh, int rank) {
    __syncthreads();
    for (int b = threadIdx.x; b < NB; b += THREADS) {
        uint32_t c0 = 0, c1 = 0;
        float m1 = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            c0 += sh.wcnt[w][0][b];
            c1 += sh.wcnt[w][1][b];
            m1 += sh.wmass[w][b];
            sh.wcnt[w][0][b] = sh.wcnt[w][1][b] = 0;
            sh.wmass[w][b] = 0.f;
        }
        sh.cta[0][b] = (float)c0;
        sh.cta[1][b] = (float)c1;
        sh.cta[2][b] = m1;
    }
    cluster_sync();   // every CTA's histograms are complete
    // bucket b of histogram h is summed over the 8 CTAs in a fixed order by every CTA (no
    // second exchange): NH * NB * 8 distributed loads per CTA
    for (int i = threadIdx.x; i < NH * NB + 4; i += THREADS) {
        const float* src = i < NH * NB ? &sh.cta[0][0] + i : sh.scal + (i - NH * NB);
        float t = 0.f;
#pragma unroll
        for (int r = 0; r < CL; ++r) t += ld_peer(src, r);
        if (i < NH * NB) (&sh.sum[0][0])[i] = t;
        else sh.scal_sum[i - NH * NB] = t;
    }
    cluster_sync();   // the peers' histograms may be overwritten from here on
}

// Choose the bucket of search s at this digit from the cluster's histograms (thread 0 of each
// CTA, the same decision in all): by count (rem_c-th entry), or by mass (first bucket where
// the cumulative mass reaches rem_m; strict: exceeds it).
QW_DEV void select_bucket(Shared& sh, int s, bool by_mass, bool strict, int shift) {
    const float* cnt = sh.sum[s == 0 ? 0 : 1];
    const float* mass = sh.sum[2];
    int sel = -1;
    if (!by_mass) {
        uint32_t c = 0;
        for (int b = NB - 1; b >= 0; --b) {
            const uint32_t n = (uint32_t)cnt[b];
            if (c + n >= sh.rem_c[s]) {
                sel = b;
                break;
            }
            c += n;
        }
        if (sel >= 0) sh.rem_c[s] -= c;
    } else {
        float acc = 0.f;
        for (int b = NB - 1; b >= 0; --b) {
            const float nxt = acc + mass[b];
            if (cnt[b] > 0.f && (strict ? nxt > sh.rem_m[s] : nxt >= sh.rem_m[s])) {
                sel = b;
                break;
            }
            acc = nxt;
        }
        if (sel >= 0) sh.rem_m[s] -= acc;
    }
    if (sel < 0) {   // rounding left the target past the last entry: take the last nonempty bucket whole
        for (int b = 0; b < NB && sel < 0; ++b)
            if (cnt[b] > 0.f) sel = b;
        sel = sel < 0 ? 0 : sel;
        sh.rem_c[s] = (uint32_t)cnt[sel];
        sh.rem_m[s] = mass[sel];
    }
    sh.prefix[s] |= (uint32_t)sel << shift;
    sh.pmask[s] |= 255u << shift;
    if (shift == 0) sh.cnt_key[s] = (uint32_t)cnt[sel];
}

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS)
    sample_kernel(const float* __restrict__ logits, int vocab, const qw_sample_params* __restrict__ params,
                  uint64_t rng_counter, int32_t* __restrict__ out, const float2* __restrict__ part, int n_part,
                  const int* __restrict__ argmax_hint, int* err) {
    __shared__ Shared sh;
    pdl_wait();   // launched with pdl_launch: the LM head may still be running
    pdl_trigger();
    const int row = blockIdx.x / CL, rank = (int)cluster_rank(), tid = threadIdx.x;
    const float* lg = logits + (size_t)row * vocab;
    const qw_sample_params P = params[row];
    const bool greedy = !(P.temperature > 0.f);
    // rows the top-k kernel (launched just before) sampled: it wrote an id; -1 hands the row over
    if (topk_row(P, vocab) && out[row] >= 0) return;
    // this CTA's ids [j_lo, j_hi): whole float4s, the last CTA takes the ragged end
    const int span = ((vocab + CL - 1) / CL + 3) & ~3;
    const int j_lo = min(vocab, rank * span), j_hi = min(vocab, j_lo + span);
    for (int i = tid; i < NW * 2 * NB; i += THREADS) (&sh.wcnt[0][0][0])[i] = 0;
    for (int i = tid; i < NW * NB; i += THREADS) (&sh.wmass[0][0])[i] = 0.f;
    if (tid < 4) sh.scal[tid] = 0.f;

    // ---- row maximum and its lowest id: pack (order key, ~id) so one max picks both.  Every
    // CTA of the cluster scans the partials (or the whole row) and gets the same answer.
    if (greedy && argmax_hint) {
        if (rank == 0 && tid == 0) out[row] = argmax_hint[row];
        cluster_sync();
        return;
    }
    unsigned long long best = 0ull;
    if (part) {
        const float2* pr = part + (size_t)row * n_part;
        for (int t = tid; t < n_part; t += THREADS) {
            const float2 v = pr[t];
            const unsigned long long k = ((unsigned long long)order_key(v.x) << 32) |
                                         (unsigned long long)(0xFFFFFFFFu - (uint32_t)__float_as_int(v.y));
            best = k > best ? k : best;
        }
    } else {
        for (int j = tid; j < vocab; j += THREADS) {
            const unsigned long long k =
                ((unsigned long long)order_key(lg[j]) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
            best = k > best ? k : best;
        }
    }
    best = block_reduce(best, [](unsigned long long a, unsigned long long b) { return a > b ? a : b; }, sh.ured, 0ull);
    if (greedy) {
        if (rank == 0 && tid == 0) out[row] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
        cluster_sync();
        return;
    }
    const float mx = key_value((uint32_t)(best >> 32));
    int top_k = P.top_k;
    float top_p = P.top_p;
    if (top_k < 0 || !(top_p > 0.f) || top_p > 1.f) {
        if (rank == 0 && tid == 0) set_error(err, QW_EINVAL);
        top_k = max(top_k, 0);
        top_p = fminf(fmaxf(top_p, 1e-6f), 1.f);   // NaN -> 1e-6
    }
    const bool use_k = top_k > 0 && top_k < vocab;
    const bool use_p = top_p < 1.f;
    const float c = 1.4426950408889634f / P.temperature;   // e_i = 2^((l_i - max) * c)
    if (tid < 2) {
        sh.prefix[tid] = sh.pmask[tid] = 0;
        sh.rem_c[tid] = (uint32_t)top_k;
    }

    // ---- a pass over this CTA's slice: histograms of both searches at digit `shift` of the
    // entries matching each search's prefix (pass 1: every entry), plus the sum of e_i of the
    // entries with key > above_k when sum_above (pass 1 and the kept-mass pass)
    auto pass = [&](int shift, bool s0, bool s1, bool all, bool sum_above, uint32_t above_k) {
        __syncthreads();
        const uint32_t pf0 = sh.prefix[0], pm0 = sh.pmask[0], pf1 = sh.prefix[1], pm1 = sh.pmask[1];
        float acc = 0.f;
        const int n_iter = (j_hi - j_lo + 4 * THREADS - 1) / (4 * THREADS);   // the same for every thread:
        for (int it = 0; it < n_iter; ++it) {                                 // the warp intrinsics below
            const int j0 = j_lo + it * 4 * THREADS + 4 * tid;                 // need every lane
            float v[4];
            if (j0 + 3 < j_hi) {
                const float4 q = __ldg((const float4*)(lg + j0));
                v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = j0 + i < j_hi ? lg[j0 + i] : -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool in = j0 + i < j_hi;
                const uint32_t k = order_key(v[i]);
                const bool m0 = in && s0 && (all || (k & pm0) == pf0);
                const bool m1 = in && s1 && (all || (k & pm1) == pf1);
                const float e = (m1 || (sum_above && in && k > above_k)) ? exp2f((v[i] - mx) * c) : 0.f;
                if (sum_above && in && k > above_k) acc += e;
                const uint32_t b = (k >> shift) & 255u;
                if (__any_sync(0xffffffffu, m0)) hist_add(sh, 0, b, 0.f, m0);
                if (__any_sync(0xffffffffu, m1)) hist_add(sh, 1, b, e, m1);
            }
        }
        if (sum_above) acc = block_reduce(acc, [](float a, float b) { return a + b; }, sh.red, 0.f);
        if (tid == 0) sh.scal[0] = acc;
        cluster_histograms(sh, rank);
    };

    // passes 1..4: both cut searches (pass 1 also sums Z: every key is above key 0)
    float z = 0.f;
    for (int shift = 24; shift >= 0; shift -= 8) {
        const bool first = shift == 24;
        if (!first && !use_k && !use_p) break;
        pass(shift, use_k, use_p, first, first, 0u);
        if (first) {
            z = sh.scal_sum[0];
            if (tid == 0) sh.rem_m[1] = top_p * z;
        }
        if (tid == 0) {
            if (use_k) select_bucket(sh, 0, false, false, shift);
            if (use_p) select_bucket(sh, 1, true, false, shift);
        }
        __syncthreads();
    }
    // ---- the kept prefix: the earlier cut; n entries of key K
    uint32_t K = 0;   // order key 0 is below every float: no cut keeps everything
    uint32_t n = 0;
    if (use_p) {
        K = sh.prefix[1];
        const float eK = exp2f((key_value(K) - mx) * c);
        const uint32_t np = eK > 0.f ? (uint32_t)ceilf(sh.rem_m[1] / eK) : 1u;
        n = min(max(np, 1u), sh.cnt_key[1]);
    }
    if (use_k) {
        const uint32_t Kk = sh.prefix[0], nk = sh.rem_c[0];
        if (!use_p || Kk > K || (Kk == K && nk < n)) {
            K = Kk;
            n = nk;
        }
    }
    const bool cut = use_k || use_p;
    const float eK = cut ? exp2f((key_value(K) - mx) * c) : 0.f;
    uint32_t c4[4] = {(uint32_t)rng_counter, (uint32_t)(rng_counter >> 32), 0u, 0u};
    philox4x32_10(c4, (uint32_t)P.seed, (uint32_t)(P.seed >> 32));
    const float u = (float)(c4[0] >> 8) * (1.0f / 16777216.0f);
    // ---- pass 5: the kept mass (entries above K, plus n at K) and the top digit of the draw;
    // passes 6..8: the lower digits of the draw (search 1 by mass, strict)
    __syncthreads();
    if (tid == 0) sh.prefix[1] = sh.pmask[1] = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        const bool first = shift == 24;
        pass(shift, false, true, first, first && cut, K);
        if (tid == 0) {
            if (first) sh.rem_m[1] = u * (cut ? sh.scal_sum[0] + (float)n * eK : z);
            select_bucket(sh, 1, true, true, shift);
        }
        __syncthreads();
    }
    // ---- the drawn entry: the t-th lowest id with key Kd, t = 1 + floor(remaining mass / e)
    uint32_t Kd = sh.prefix[1];
    const float ed = exp2f((key_value(Kd) - mx) * c);
    uint32_t t = ed > 0.f ? (uint32_t)floorf(sh.rem_m[1] / ed) + 1u : 1u;
    t = min(max(t, 1u), sh.cnt_key[1]);
    if (cut && (Kd < K || (Kd == K && t > n))) {   // rounding past the kept prefix: its last entry
        Kd = K;
        t = n;
    }
    // matches of Kd in this CTA's slice, counted in id order: thread i scans
    // [j_lo + i * sub, j_lo + (i + 1) * sub); prefix sums over threads and CTAs locate the t-th
    const int sub = (j_hi - j_lo + THREADS - 1) / THREADS;
    const int s_lo = min(j_hi, j_lo + tid * sub), s_hi = min(j_hi, s_lo + sub);
    uint32_t mine = 0;
    for (int j = s_lo; j < s_hi; ++j) mine += order_key(lg[j]) == Kd;
    uint32_t incl = mine;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    __syncthreads();
    if (lane == 31) sh.ired[warp] = (int)incl;
    __syncthreads();
    uint32_t base = 0, cta_total = 0;
    for (int w = 0; w < NW; ++w) {
        base += w < warp ? (uint32_t)sh.ired[w] : 0u;
        cta_total += (uint32_t)sh.ired[w];
    }
    if (tid == 0) sh.scal[1] = (float)cta_total;   // exact below 2^24
    cluster_sync();
    uint32_t cta_base = 0;
    for (int r = 0; r < rank; ++r) cta_base += (uint32_t)ld_peer(&sh.scal[1], r);
    const uint32_t before = cta_base + base + incl - mine;
    if (before < t && t <= before + mine) {
        uint32_t seen = before;
        for (int j = s_lo; j < s_hi; ++j)
            if (order_key(lg[j]) == Kd && ++seen == t) {
                out[row] = j;
                break;
            }
    }
    cluster_sync();   // no peer reads this CTA's shared memory after it exits
}

// ---------------------------------------------------------------- top-k rows (1 <= top_k <= 1024)
// A row whose kept set is capped by a small top_k needs only its top_k best entries, plus the
// full-vocabulary normaliser Z of the article's softmax.  One cluster of FCL CTAs (1024 threads
// each) per row, CTA r streaming the r-th part of the row (one SM alone pulls a 608 KB row too
// slowly); the CTAs exchange through distributed shared memory:
//   pass 1  max, min and Z = sum of 2^((l - max) c) (online, c = log2(e) / T), merged
//   pass 2  histogram of 2048 equal-width buckets of (max - l) over [0, max - min], summed over
//           the cluster; the first bucket where the count from the top reaches top_k bounds the
//           k-th entry from below
//   pass 3  every entry at or above that bucket (at most FCAP, else the row is handed to the
//           general kernel by writing -1) goes to rank 0 as (order key, ~id), which sorts them
//           (bitonic, descending)
// then, over the sorted candidates: p_i = e_i / Z, cutoff = min(top_k, 1 + #(cumsum < top_p)),
// the draw is the first kept entry whose cumulative e exceeds u * (kept e), u from Philox as in
// the general kernel.  Rows this kernel does not take (greedy, top_k outside [1, 1024], invalid
// parameters) are left untouched for the general kernel that runs after it.  Every decision to
// end early is taken from cluster-wide values, so all CTAs of a row take it together.
QW_DEV void st_peer_u64(unsigned long long* local, int rank, unsigned long long v) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
QW_DEV uint32_t atom_add_peer(uint32_t* local, int rank, uint32_t v) {
    uint32_t a, old;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
    return old;
}
QW_DEV uint32_t ld_peer_u32(const uint32_t* local, int rank) {
    uint32_t a, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

// two CTAs per SM (at most 32 registers a thread), so the 64 clusters of a 64-row batch are
// resident at once
__global__ void __cluster_dims__(FCL, 1, 1) __launch_bounds__(FT, 2)
    sample_topk_kernel(const float* __restrict__ logits, int vocab, const qw_sample_params* __restrict__ params,
                       uint64_t rng_counter, int32_t* __restrict__ out) {
    __shared__ FShared sh;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x / FCL, rank = (int)cluster_rank(), tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const qw_sample_params P = params[row];
    if (!topk_row(P, vocab)) return;   // the same for every CTA of the row
    const float* lg = logits + (size_t)row * vocab;
    const float c = 1.4426950408889634f / P.temperature;
    const int k = P.top_k;
    const int n4 = vocab / 4;   // vocab is a multiple of 32: whole float4s, and n4 a multiple of FCL
    const int i_lo = rank * (n4 / FCL), i_hi = (rank + 1) * (n4 / FCL);
    // a pass over the part: f(i, float4 i) for i = i_lo + tid (mod FT), FUN loads in flight
    auto sweep = [&](auto&& f) {
        for (int i0 = i_lo + tid; i0 < i_hi; i0 += FUN * FT) {
            float4 qs[FUN];
#pragma unroll
            for (int j = 0; j < FUN; ++j)
                if (i0 + j * FT < i_hi) qs[j] = __ldg((const float4*)lg + i0 + j * FT);
#pragma unroll
            for (int j = 0; j < FUN; ++j)
                if (i0 + j * FT < i_hi) f(i0 + j * FT, qs[j]);
        }
    };
    for (int b = tid; b < FNB; b += FT) sh.hist[b] = 0;
    if (tid == 0) sh.ncand = 0;

    // ---- pass 1: max, min, Z of this CTA's part, then of the row
    float m = -INFINITY, mn = INFINITY, z = 0.f;
    sweep([&](int, float4 q) {
        const float v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (v[t] > m) {
                z = z * exp2f((m - v[t]) * c) + 1.f;
                m = v[t];
            } else {
                z += exp2f((v[t] - m) * c);
            }
            mn = fminf(mn, v[t]);
        }
    });
    const float M = warp_max(m);
    float zr = m == -INFINITY ? 0.f : z * exp2f((m - M) * c);
    zr = warp_sum(zr);
    const float mnw = -warp_max(-mn);
    if (lane == 0) {
        sh.fred[warp] = M;
        sh.fred2[warp] = mnw;
    }
    __syncthreads();
    float cM = -INFINITY, cmn = INFINITY;
#pragma unroll 4
    for (int w = 0; w < FNW; ++w) {
        cM = fmaxf(cM, sh.fred[w]);
        cmn = fminf(cmn, sh.fred2[w]);
    }
    __syncthreads();
    if (lane == 0) sh.fred[warp] = M == -INFINITY ? 0.f : zr * exp2f((M - cM) * c);
    __syncthreads();
    if (tid == 0) {
        float cz = 0.f;
        for (int w = 0; w < FNW; ++w) cz += sh.fred[w];
        sh.stats[0] = cM;
        sh.stats[1] = cmn;
        sh.stats[2] = cz;
    }
    cluster_sync();   // every CTA's stats, cleared histogram and candidate count are in place
    float gM = -INFINITY, gmn = INFINITY;
    float pm[FCL], pz[FCL];
#pragma unroll
    for (int r = 0; r < FCL; ++r) {
        pm[r] = ld_peer(&sh.stats[0], r);
        gmn = fminf(gmn, ld_peer(&sh.stats[1], r));
        pz[r] = ld_peer(&sh.stats[2], r);
        gM = fmaxf(gM, pm[r]);
    }
    float Z = 0.f;
#pragma unroll
    for (int r = 0; r < FCL; ++r) Z += pm[r] == -INFINITY ? 0.f : pz[r] * exp2f((pm[r] - gM) * c);
    const bool degenerate = !(gM > gmn) || !(Z > 0.f);   // a constant row (ties everywhere) or non-finite values
    // ---- pass 2: bucket histogram of this CTA's part
    const float inv_w = degenerate ? 0.f : (float)FNB / (gM - gmn);
    auto bucket = [&](float v) {   // monotone in v; NaN lands in the last bucket
        const float d = (gM - v) * inv_w;
        return d < (float)(FNB - 1) ? (int)d : FNB - 1;
    };
    if (!degenerate)
        sweep([&](int, float4 q) {
            atomicAdd(&sh.hist[bucket(q.x)], 1u);
            atomicAdd(&sh.hist[bucket(q.y)], 1u);
            atomicAdd(&sh.hist[bucket(q.z)], 1u);
            atomicAdd(&sh.hist[bucket(q.w)], 1u);
        });
    cluster_sync();   // every part's histogram is complete
    // the row's counts of buckets 2 tid, 2 tid + 1, and an inclusive prefix over the buckets: the
    // first bucket reaching k (every CTA of the cluster finds the same one)
    {
        uint32_t h0 = 0, h1 = 0;
#pragma unroll
        for (int r = 0; r < FCL; ++r) {
            h0 += ld_peer_u32(&sh.hist[2 * tid], r);
            h1 += ld_peer_u32(&sh.hist[2 * tid + 1], r);
        }
        uint32_t incl = h0 + h1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) sh.ured[warp] = incl;
        __syncthreads();
        uint32_t base = 0;
        for (int w = 0; w < warp; ++w) base += sh.ured[w];
        const uint32_t before = base + incl - (h0 + h1);
        if (before < (uint32_t)k && before + h0 >= (uint32_t)k) {
            sh.bstar = 2 * tid;
            sh.cnt_star = before + h0;
        } else if (before + h0 < (uint32_t)k && before + h0 + h1 >= (uint32_t)k) {
            sh.bstar = 2 * tid + 1;
            sh.cnt_star = before + h0 + h1;
        }
    }
    __syncthreads();
    const int bstar = (int)sh.bstar;
    const uint32_t ncand = sh.cnt_star;
    if (degenerate || ncand > FCAP) {   // the general kernel takes the row
        cluster_sync();   // the peers have read this CTA's histogram
        if (rank == 0 && tid == 0) out[row] = -1;
        return;
    }
    // ---- pass 3: the candidates of this part into rank 0's buffer
    sweep([&](int i, float4 q) {
        const float v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (bucket(v[t]) <= bstar) {
                const uint32_t slot = atom_add_peer(&sh.ncand, 0, 1u);
                if (slot < FCAP)
                    st_peer_u64(&sh.cand[slot], 0,
                                ((unsigned long long)order_key(v[t]) << 32) | (0xFFFFFFFFu - (uint32_t)(4 * i + t)));
            }
    });
    cluster_sync();   // rank 0 holds every candidate, and the peers are done with every exchange
    if (rank != 0) return;
    int np2 = 1;
    while (np2 < (int)ncand) np2 <<= 1;
    for (int i = (int)ncand + tid; i < np2; i += FT) sh.cand[i] = 0ull;   // below every entry
    __syncthreads();
    for (int size = 2; size <= np2; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < np2; i += FT) {
                const int j = i ^ stride;
                if (j > i) {
                    const unsigned long long a = sh.cand[i], b = sh.cand[j];
                    const bool desc = (i & size) == 0;   // descending runs, merged into one descending order
                    if (desc ? a < b : a > b) {
                        sh.cand[i] = b;
                        sh.cand[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    // ---- top-k, top-p and the draw over the first k candidates (k <= FT)
    const bool mine = tid < k;
    const float ei = mine ? exp2f((key_value((uint32_t)(sh.cand[tid] >> 32)) - gM) * c) : 0.f;
    float incl = ei;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) sh.fred[warp] = incl;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; ++w) base += sh.fred[w];
    const float cum = base + incl;
    if (mine) sh.e[tid] = cum;
    // cutoff = min(k, 1 + #(cumsum of p < top_p))
    const bool below = mine && cum / Z < P.top_p;
    const uint32_t nb = __popc(__ballot_sync(0xffffffffu, below));
    if (lane == 0) sh.ured[warp] = nb;
    if (tid == 0) sh.pick = k;
    __syncthreads();
    uint32_t nbelow = 0;
    for (int w = 0; w < FNW; ++w) nbelow += sh.ured[w];
    const int cutoff = min(k, (int)nbelow + 1);
    const float kept = sh.e[cutoff - 1];
    uint32_t c4[4] = {(uint32_t)rng_counter, (uint32_t)(rng_counter >> 32), 0u, 0u};
    philox4x32_10(c4, (uint32_t)P.seed, (uint32_t)(P.seed >> 32));
    const float u = (float)(c4[0] >> 8) * (1.0f / 16777216.0f);
    if (tid < cutoff && cum > u * kept) atomicMin(&sh.pick, tid);
    __syncthreads();
    if (tid == 0) {
        const int i = min(sh.pick, cutoff - 1);   // rounding past the kept prefix: its last entry
        out[row] = (int32_t)(0xFFFFFFFFu - (uint32_t)(sh.cand[i] & 0xFFFFFFFFull));
    }
}

}  // namespace smp

int launch_sample(const float* logits, int batch, int vocab, const qw_sample_params* params, uint64_t rng_counter,
                  int32_t* out_ids, const float2* tile_part, int n_part, const int* argmax_hint, int* err,
                  cudaStream_t st) {
    if (batch <= 0) return QW_OK;
    if (pdl_launch(smp::sample_topk_kernel, dim3(batch * smp::FCL), dim3(smp::FT), 0, st, logits, vocab, params,
                   rng_counter, out_ids) != cudaSuccess)
        return QW_ECUDA;
    count_launches(1);
    const cudaError_t e = pdl_launch(smp::sample_kernel, dim3(batch * smp::CL), dim3(smp::THREADS), 0, st, logits, vocab,
                                     params, rng_counter, out_ids, tile_part, n_part, argmax_hint, err);
    count_launches(1);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QW_OK : QW_ECUDA;
}

}  // namespace qw
