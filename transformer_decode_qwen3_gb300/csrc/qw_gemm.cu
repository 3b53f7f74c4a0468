// Y = X W^T on the 5th-generation tensor core: bf16 operands, fp32 accumulation
// in tensor memory (TMEM), operands staged by TMA with 128-byte swizzling.
//
// Used for the projections of the article's Step 5 (q/k/v/o_proj), Step 6
// (gate/up/down_proj) and Step 8 (LM head) whenever a call carries more than a
// few rows (prefill, batched decode).
//
// Persistent: one CTA per SM walks 128 x BN output tiles.  Warp 0 (one lane)
// issues TMA loads into a STAGES-deep shared-memory ring, warp 1 (one lane)
// issues tcgen05.mma (K = 16 per instruction, 4 per 64-wide K block) into one of
// two TMEM accumulators and commits each stage back to the producer; warps 4..7
// read the other accumulator with tcgen05.ld (thread t owns output row t) and
// apply the fused epilogue, so a tile's epilogue overlaps the next tile's MMAs.
//
// Multicast mode (large M): CTAs run in clusters of two that take vertically adjacent
// output tiles with the same weight tile; each CTA fetches half of that B tile and TMA
// multicasts it into both CTAs' shared memory, so each CTA pulls 32 KB instead of 48 KB
// from L2 per 64-wide K block.  A stage is refilled only once both CTAs' MMAs are done
// with it (their commits arrive on both CTAs' empty barriers).
//
// Residual add (large M): each epilogue warp stages its 32 x 32 fp32 block in shared
// memory and adds it into the output with a TMA reduce-add, so the SM never reads the
// residual stream and writes it only in bulk.
//
// Split-operand mode (small M, e.g. decode batches): every activation row a is
// stored as two bf16 rows, hi = bf16(a) in tile rows 0..63 and lo = bf16(a - hi)
// in rows 64..127, so one M=128 MMA yields hi.W and lo.W side by side and the
// epilogue adds them: the activation enters with ~16 mantissa bits instead of 8,
// at no extra tensor-core work (the tile would otherwise be half empty).
#include <cudaTypedefs.h>

#include <string.h>

#include <mutex>
#include <vector>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {

template <int BN>
struct GemmCfg {
    static constexpr int BM = 128;
    static constexpr int BK = 64;                       // 64 bf16 = one 128-byte swizzle row
    static constexpr int STAGES = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;            // two accumulators; power of two >= 32
    // split mode: hand-over of the lo rows (64 x 33 floats); residual add: one 4 KB staging
    // block (32 rows x 32 fp32, 128-byte swizzled) per epilogue warp for the TMA reduce-add
    static constexpr int XCH_BYTES = 4 * 4096;
    static constexpr int SMEM = STAGES * STAGE_BYTES + XCH_BYTES + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr int THREADS = 256;                 // warps 0-3: TMA, MMA, TMEM owner, idle; 4-7: epilogue
};

// SiLU on the special-function unit (2^x and 1/x approximations, relative error ~1e-6; the
// result is rounded to bf16 next).  Large negative g: 2^x overflows to +inf and 1/inf = 0.
QW_DEV float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Destination row of activation row m in the split layout (hi copy; lo is 64 rows further).
QW_DEV int split_row(int m) { return (m >> 6) * 128 + (m & 63); }

template <int BN, int EPI>
QW_DEV void epilogue_chunk(const float (&v)[32], int m, int n, const GemmEpilogue& ep) {
    if (EPI == EPI_STORE_F32) {
        float4* dst = (float4*)(ep.out + (size_t)m * ep.ldo + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else if (EPI == EPI_ADD_ATOMIC) {  // one K-slice of a split-K product: out += partial
        float4* dst = (float4*)(ep.out + (size_t)m * ep.ldo + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) atomicAdd(dst + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
    } else if (EPI == EPI_RESID_ADD) {
        float4* dst = (float4*)(ep.out + (size_t)m * ep.ldo + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 r = dst[i];
            r.x += v[4 * i];
            r.y += v[4 * i + 1];
            r.z += v[4 * i + 2];
            r.w += v[4 * i + 3];
            dst[i] = r;
        }
    } else {  // EPI_SWIGLU: columns alternate gate, up
        float a[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = silu_f(v[2 * i]) * v[2 * i + 1];
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            hi[i] = pack_bf16x2(a[2 * i], a[2 * i + 1]);
            lo[i] = pack_bf16x2(a[2 * i] - bf16_lo(hi[i]), a[2 * i + 1] - bf16_hi(hi[i]));
        }
        const int row = ep.split ? split_row(m) : m;
        uint4* dst = (uint4*)(ep.act + (size_t)row * ep.ldo + (n >> 1));
        dst[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        dst[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        if (ep.split) {
            uint4* dl = (uint4*)((uint16_t*)dst + (size_t)64 * ep.ldo);
            dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        }
    }
}

QW_DEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// global[tile at (x, y)] += shared tile, element-wise in L2 (the tensor map's fp32 type).
QW_DEV void tma_reduce_add_2d(const CUtensorMap* m, const void* smem_src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     (uint64_t)m),
                 "r"(x), "r"(y), "r"(smem_u32(smem_src))
                 : "memory");
}
QW_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
QW_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
QW_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

QW_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
QW_DEV uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
QW_DEV uint32_t n_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// All threads of both CTAs of the cluster.
QW_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA load delivered to the same shared-memory offset (data and mbarrier) in every CTA of mask.
QW_DEV void tma_load_2d_mc(void* smem_dst, const CUtensorMap* m, int x, int y, uint64_t* bar, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
        : "memory");
}
// Arrive on the mbarrier at this offset in every CTA of mask once this thread's MMAs are done.
QW_DEV void umma_commit_mc(uint64_t* bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(smem_u32(bar)),
                 "h"(mask)
                 : "memory");
}

// Store 32 values as bf16 (four 16-byte stores).
QW_DEV void store_bf16x32(uint16_t* dst, const float (&y)[32]) {
    uint4* d = (uint4*)dst;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = make_uint4(pack_bf16x2(y[8 * i], y[8 * i + 1]), pack_bf16x2(y[8 * i + 2], y[8 * i + 3]),
                          pack_bf16x2(y[8 * i + 4], y[8 * i + 5]), pack_bf16x2(y[8 * i + 6], y[8 * i + 7]));
}

// EPI_QKV_ROPE on one accumulator tile: this thread's row m, columns n0 .. n0 + BN - 1 = BN / 128
// whole heads of the fused q|k|v output (Steps 4-5 of the article).  q and k heads: RMS-normalised
// over their 128 values (QK-Norm), scaled by the norm weight, rotated by RoPE with pairs
// (d, d + 64) at angle float32(pos * inv_freq[d]) (cos and sin from a per-row table, read once
// for all heads of the tile); q goes out as bf16, k and v enter the cache page of (tok_seq[m],
// pos) as bf16.  nw: the q and k norm weights in shared memory (nw[0..127] q, nw[128..255] k).
// TMEM loads are warp-collective, so every thread loads even when its row is past M; only the
// stores are per row.
template <int BN>
QW_DEV void qkv_rope_tile(uint32_t trow, int m, int M, int n0, int N, const GemmEpilogue& ep, const float* nw) {
    constexpr int NH = BN / 128;
    const QkvRope& r = ep.rope;
    const bool live = m < M;
    uint16_t* kv_row = nullptr;  // this row's slot in its cache page (k of head 0)
    if (live && n0 + BN > r.Hq * 128) {  // the tile holds k or v heads
        const int pos = r.positions[m];
        const int seq = r.tok_seq[m];
        const int page = pos >= 0 && pos < r.kv.bt_stride * QW_PAGE_SIZE
                             ? r.kv.block_tables[(size_t)seq * r.kv.bt_stride + pos / QW_PAGE_SIZE]
                             : -1;
        if (page < 0 || page >= r.kv.n_pages)
            set_error(ep.err, QW_ERANGE);
        else
            kv_row = r.kv.base + (size_t)page * r.kv.page_stride + (size_t)(pos % QW_PAGE_SIZE) * QW_HEAD_DIM;
    }
    uint16_t* dst[NH];
    bool rope[NH], valid[NH];
    float sc[NH];
#pragma unroll
    for (int hd = 0; hd < NH; ++hd) {
        const int col = n0 + 128 * hd;
        const int head = col / 128;
        valid[hd] = col < N;
        rope[hd] = valid[hd] && head < r.Hq + r.Hkv;
        dst[hd] = nullptr;
        if (valid[hd] && head < r.Hq)
            dst[hd] = live ? r.q_bf16 + (size_t)m * r.Hq * 128 + (size_t)head * 128 : nullptr;
        else if (valid[hd] && kv_row)  // k heads Hq .. Hq+Hkv-1, then v heads: (K/V, head) rows of 16 slots
            dst[hd] = kv_row + (size_t)(head - r.Hq) * QW_PAGE_SIZE * QW_HEAD_DIM;
        sc[hd] = 1.f;
    }
    // v heads: plain bf16 copy; q and k heads: sum of squares
#pragma unroll
    for (int hd = 0; hd < NH; ++hd) {
        if (!valid[hd]) continue;  // uniform
        const uint32_t t0 = trow + (uint32_t)(128 * hd);
        float ss = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(t0 + 32 * c, v);
            if (rope[hd]) {
#pragma unroll
                for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
            } else if (dst[hd]) {
                store_bf16x32(dst[hd] + 32 * c, v);
            }
        }
        sc[hd] = 1.0f / sqrtf(ss / (float)QW_HEAD_DIM + r.eps);
    }
    if (!(rope[0] || (NH > 1 && rope[NH - 1]))) return;  // uniform
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {  // dims 32 j .. 32 j + 31 pair with 32 j + 64 ..
        float4 t[16];              // (cos, sin) of pairs 32 j + 2 i and + 1
        const float4* cs4 = (const float4*)(r.rope + (size_t)(live ? m : 0) * 64 + 32 * j);
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] = __ldg(cs4 + i);
#pragma unroll
        for (int hd = 0; hd < NH; ++hd) {
            if (!rope[hd]) continue;  // uniform
            const int head = (n0 + 128 * hd) / 128;
            const float* w = nw + (head < r.Hq ? 0 : 128);
            const uint32_t t0 = trow + (uint32_t)(128 * hd);
            float a[32], b[32];
            tmem_ld32_nowait(t0 + 32 * j, a);
            tmem_ld32_nowait(t0 + 32 * j + 64, b);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float4 tt = t[i / 2];
                const int d = 32 * j + i;
                const float x1 = a[i] * sc[hd] * w[d], x2 = b[i] * sc[hd] * w[d + 64];
                const float y1 = a[i + 1] * sc[hd] * w[d + 1], y2 = b[i + 1] * sc[hd] * w[d + 65];
                a[i] = x1 * tt.x - x2 * tt.y;
                b[i] = x1 * tt.y + x2 * tt.x;
                a[i + 1] = y1 * tt.z - y2 * tt.w;
                b[i + 1] = y1 * tt.w + y2 * tt.z;
            }
            if (dst[hd]) {
                store_bf16x32(dst[hd] + 32 * j, a);
                store_bf16x32(dst[hd] + 32 * j + 64, b);
            }
        }
    }
}

template <int BN, int EPI, bool SPLIT, bool MC>
__global__ void __launch_bounds__(256, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, int M, int N, int K, int tiles_m, int tiles_n,
                        int ksplit, int share_a, GemmEpilogue ep) {
    // tmC (residual add, not split): ep.out as fp32 [M][N], boxes of 32 x 32, 128-byte swizzle
    // MC: tmB has boxes of BN / 2 rows (each CTA of the pair loads one half)
    using C = GemmCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    float* xch = (float*)(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES + C::XCH_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;   // [2] accumulator ready for the epilogue
    uint64_t* tempty = tfull + 2;          // [2] accumulator drained by the epilogue
    uint32_t* tmem_slot = (uint32_t*)(tempty + 2);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    // a CTA of this launch already gave up on a wait: end quickly instead of timing out again
    // (in a cluster the CTA still meets its peer at the cluster barriers, with no work)
    const bool gave_up = ep.err && *(volatile int*)ep.err == QW_ETIMEOUT;
    if (!MC && gave_up) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = K / C::BK;
    const uint32_t crank = MC ? cluster_ctarank() : 0u;
    const int tiles_mu = MC ? (tiles_m + 1) / 2 : tiles_m;   // m units (pairs of m tiles in MC)
    const int n_tiles = tiles_mu * tiles_n * ksplit;           // work units: (m unit, n tile, K slice)
    const int first = MC ? (int)cluster_id_x() : (int)blockIdx.x;
    const int stride = MC ? (int)n_clusters_x() : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], MC ? 2 : 1);   // MC: both CTAs' MMAs release a stage
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);      // one arrival per epilogue warp
        }
        *abort_flag = gave_up ? 1u : 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    if (MC) cluster_sync();   // the peer's barriers are initialised before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (!(warp == 0 && lane == 0)) {   // the producer waits after starting its weight loads
        pdl_wait();
        pdl_trigger();
    }

    // unit t -> (m tile, n tile, K blocks [kb0, kb1)).  Consecutive CTAs share the A tile
    // (share_a: n tile fastest; the whole B fits in L2) or the B tile (m tile fastest).
    auto unit = [&](int t, int& tm, int& tn, int& kb0, int& kb1) {
        const int ks = t % ksplit, rest = t / ksplit;
        tn = share_a ? rest % tiles_n : rest / tiles_mu;
        tm = share_a ? rest / tiles_n : rest % tiles_mu;
        if (MC) tm = 2 * tm + (int)crank;   // past the last m tile for an odd count: zero rows, no stores
        kb0 = ks * nk / ksplit;
        kb1 = (ks + 1) * nk / ksplit;
    };

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            // The weight tiles of the first stages do not depend on earlier kernels: they start
            // streaming before pdl_wait (launched with pdl_launch, the previous kernel may still run).
            int n_pre = 0;
            if (!MC && first < n_tiles) {
                int tm, tn, kb0, kb1;
                unit(first, tm, tn, kb0, kb1);
                n_pre = min(C::STAGES, kb1 - kb0);
                for (int i = 0; i < n_pre; ++i) {
                    mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
                    tma_load_2d(sB + i * C::B_BYTES, &tmB, (kb0 + i) * C::BK, tn * BN, &full[i]);
                }
            }
            pdl_wait();
            pdl_trigger();
            uint32_t kb_all = 0;
            for (int t = first; t < n_tiles && !*abort_flag; t += stride) {
                int tm, tn, kb0, kb1;
                unit(t, tm, tn, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++kb_all) {
                    const int s = kb_all % C::STAGES;
                    const uint32_t ph = (kb_all / C::STAGES) & 1;
                    if (kb_all < (uint32_t)n_pre) {   // weights already on their way: the activations only
                        tma_load_2d(sA + s * C::A_BYTES, &tmA, kb * C::BK, tm * C::BM, &full[s]);
                        continue;
                    }
                    if (!mbar_wait(&empty[s], ph ^ 1, ep.err) || *abort_flag) {
                        *abort_flag = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);   // MC: half of B comes from the peer
                    tma_load_2d(sA + s * C::A_BYTES, &tmA, kb * C::BK, tm * C::BM, &full[s]);
                    if (MC)
                        tma_load_2d_mc(sB + s * C::B_BYTES + crank * (C::B_BYTES / 2), &tmB, kb * C::BK,
                                       tn * BN + (int)crank * (BN / 2), &full[s], (uint16_t)0x3);
                    else
                        tma_load_2d(sB + s * C::B_BYTES, &tmB, kb * C::BK, tn * BN, &full[s]);
                }
            }
            if (MC) {
                // every commit of both CTAs aimed at this CTA's empty barriers has landed before the exit
                const uint32_t from = kb_all > (uint32_t)C::STAGES ? kb_all - C::STAGES : 0u;
                for (uint32_t i = from; i < kb_all; ++i) mbar_wait(&empty[i % C::STAGES], (i / C::STAGES) & 1, ep.err);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            constexpr uint32_t idesc = umma_idesc_bf16(C::BM, BN);
            uint32_t kb_all = 0;
            int local = 0;
            for (int t = first; t < n_tiles; t += stride, ++local) {
                const int acc = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                bool ok = !*abort_flag && mbar_wait(&tempty[acc], (use & 1) ^ 1, ep.err);
                tc_fence_after();
                const uint32_t dtm = tmem + (uint32_t)(acc * BN);
                int tm, tn, kb0, kb1;
                unit(t, tm, tn, kb0, kb1);
                for (int kb = kb0; kb < kb1 && ok; ++kb, ++kb_all) {
                    const int s = kb_all % C::STAGES;
                    const uint32_t ph = (kb_all / C::STAGES) & 1;
                    if (!mbar_wait(&full[s], ph, ep.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + s * C::A_BYTES), b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < C::BK / 16; ++k)
                        umma_bf16(dtm, umma_desc_sw128(a0 + k * 32), umma_desc_sw128(b0 + k * 32), idesc,
                                  (kb != kb0) || k != 0);
                    if (MC)
                        umma_commit_mc(&empty[s], (uint16_t)0x3);
                    else
                        umma_commit(&empty[s]);
                }
                if (!ok) {
                    *abort_flag = 1;
                    mbar_arrive(&tfull[acc]);  // release the epilogue, which sees the abort flag
                    break;
                }
                umma_commit(&tfull[acc]);
            }
        }
    } else if (warp >= 4) {
        // Epilogue warpgroup: warp 4 + i reads TMEM lanes 32 i .. 32 i + 31.
        const int ew = warp - 4;
        const int et = threadIdx.x - 128;
        if constexpr (EPI == EPI_QKV_ROPE) {  // q and k norm weights into shared memory
            xch[et] = ep.rope.q_norm[et];
            xch[128 + et] = ep.rope.k_norm[et];
            epi_bar();
        }
        int local = 0;
        for (int t = first; t < n_tiles; t += stride, ++local) {
            int tm, tn, kb0, kb1;
            unit(t, tm, tn, kb0, kb1);
            const int acc = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            const bool ok = mbar_wait(&tfull[acc], use & 1, ep.err) && !*abort_flag;
            tc_fence_after();
            if (!ok) break;
            const uint32_t trow = tmem + (uint32_t)(acc * BN) + ((uint32_t)(ew * 32) << 16);
            const int n0 = tn * BN;
            if constexpr (EPI == EPI_QKV_ROPE) qkv_rope_tile<BN>(trow, tm * C::BM + et, M, n0, N, ep, xch);
            if constexpr (EPI == EPI_RESID_ADD && !SPLIT) {
                // Each warp stages its 32 rows x 32 columns in shared memory (row = lane, 16-byte
                // units swizzled by row & 7) and one lane adds the block into the output with a
                // TMA reduce-add: the residual is never read by the SM, and rows past M are
                // clipped by the tensor map.
                uint8_t* xw = (uint8_t*)xch + ew * 4096;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    if (n0 + c0 >= N) break;  // uniform
                    float v[32];
                    tmem_ld32(trow + c0, v);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *(float4*)(xw + lane * 128 + ((u ^ (lane & 7)) << 4)) =
                            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                    fence_proxy_async();  // the TMA reads the block through the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_2d(&tmC, xw, n0 + c0, tm * C::BM + ew * 32);
                        bulk_commit();
                        bulk_wait_read0();  // the block may be overwritten once the TMA has read it
                    }
                    __syncwarp();
                }
            }
            // LM head (fp32 store with ep.tile_max): this row's maximum over the tile and its
            // lowest column, the partial the sampler's argmax and softmax start from
            float tmax = -INFINITY;
            int targ = n0;
            const int mrow = SPLIT ? tm * 64 + ew * 32 + lane : tm * C::BM + et;
#pragma unroll 1
            for (int c0 = 0; c0 < BN && EPI != EPI_QKV_ROPE && !(EPI == EPI_RESID_ADD && !SPLIT); c0 += 32) {
                if (n0 + c0 >= N) break;  // uniform over the warpgroup
                float v[32];
                tmem_ld32(trow + c0, v);
                if (SPLIT) {
                    if (ew >= 2) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) xch[((ew - 2) * 32 + lane) * 33 + i] = v[i];
                    }
                    epi_bar();
                    if (ew < 2) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] += xch[(ew * 32 + lane) * 33 + i];
                        if (mrow < M) epilogue_chunk<BN, EPI>(v, mrow, n0 + c0, ep);
                    }
                    epi_bar();
                } else {
                    if (mrow < M) epilogue_chunk<BN, EPI>(v, mrow, n0 + c0, ep);
                }
                if (EPI == EPI_STORE_F32 && ep.tile_max) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (n0 + c0 + i < N && v[i] > tmax) {
                            tmax = v[i];
                            targ = n0 + c0 + i;
                        }
                }
            }
            if (EPI == EPI_STORE_F32 && ep.tile_max && (!SPLIT || ew < 2) && mrow < M)
                ep.tile_max[(size_t)mrow * ep.tile_ld + tn] = make_float2(tmax, __int_as_float(targ));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        if (EPI == EPI_RESID_ADD && !SPLIT && lane == 0) bulk_wait0();  // the reduce-adds are done
    }
    tc_fence_before();
    __syncthreads();
    if (MC) cluster_sync();   // no multicast or remote arrive can still target this CTA
    if (warp == 2) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool load_encode_fn() {
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    return true;
}

int make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_rows) {
    if (!load_encode_fn()) return QW_ECUDA;
    if (((uintptr_t)base & 15) || (row_stride_bytes & 15)) return QW_EINVAL;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QW_OK : QW_ECUDA;
}

// fp32 [rows][inner] with 32 x 32 boxes and 128-byte swizzling (the reduce-add target).
static int make_tmap_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t row_stride_bytes) {
    if (!load_encode_fn()) return QW_ECUDA;
    if (((uintptr_t)base & 15) || (row_stride_bytes & 15)) return QW_EINVAL;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QW_OK : QW_ECUDA;
}

template <int BN, int EPI, bool SPLIT, bool MC>
static int launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, const GemmEpilogue& ep,
                     cudaStream_t st) {
    CUtensorMap tc;
    memset(&tc, 0, sizeof(tc));
    if (EPI == EPI_RESID_ADD && !SPLIT) {
        const int rc = make_tmap_f32(&tc, ep.out, (uint64_t)N, (uint64_t)M, (uint64_t)ep.ldo * 4);
        if (rc) return rc;
    }
    using C = GemmCfg<BN>;
    auto kern = gemm_bf16_tc_kernel<BN, EPI, SPLIT, MC>;
    // per device (function attributes and occupancy belong to the device), set up once under a lock
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static bool attr_set[kMaxDevices] = {};
    static int n_sm_dev[kMaxDevices] = {}, max_clusters_dev[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QW_ECUDA;
    int n_sm = 0, max_clusters = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            cudaDeviceGetAttribute(&n_sm_dev[dev], cudaDevAttrMultiProcessorCount, dev);
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
                return QW_ECUDA;
            if (MC) {
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeClusterDimension;
                at[0].val.clusterDim.x = 2;
                at[0].val.clusterDim.y = 1;
                at[0].val.clusterDim.z = 1;
                cfg.gridDim = dim3(2 * (n_sm_dev[dev] / 2));
                cfg.blockDim = dim3(C::THREADS);
                cfg.dynamicSmemBytes = C::SMEM;
                cfg.attrs = at;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&max_clusters_dev[dev], kern, &cfg) != cudaSuccess ||
                    max_clusters_dev[dev] < 1)
                    return QW_ECUDA;
            }
            attr_set[dev] = true;
        }
        n_sm = n_sm_dev[dev];
        max_clusters = max_clusters_dev[dev];
    }
    const int tiles_m = SPLIT ? (M + 63) / 64 : (M + C::BM - 1) / C::BM;
    const int tiles_n = (N + BN - 1) / BN;
    // split-K (atomic epilogue only): enough K slices to give every SM a unit
    int ksplit = 1;
    if (EPI == EPI_ADD_ATOMIC) {
        const int nk = K / C::BK, units = tiles_m * tiles_n;
        ksplit = units < n_sm ? n_sm / units : 1;
        if (ksplit > nk) ksplit = nk;
        if (ksplit < 1) ksplit = 1;
    }
    // A streams from HBM once when the CTAs running together share its tiles; that needs the
    // weight matrix B to stay L2-resident (projection weights are 4..13 MB; the LM head is not).
    const int share_a = (int64_t)N * K * 2 <= (int64_t)32 << 20 && tiles_m > 1;
    if (MC) {
        const int units = (tiles_m + 1) / 2 * tiles_n;
        const int nc = units < max_clusters ? units : max_clusters;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * nc);
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, M, N, K, tiles_m, tiles_n, 1, share_a, ep);
        count_launches(1);
        return e == cudaSuccess ? QW_OK : QW_ECUDA;
    }
    const int work = tiles_m * tiles_n * ksplit;
    const int grid = work < n_sm ? work : n_sm;
    const cudaError_t e = pdl_launch(kern, dim3(grid), dim3(C::THREADS), C::SMEM, st, ta, tb, tc, M, N, K, tiles_m,
                                     tiles_n, ksplit, share_a, ep);
    count_launches(1);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QW_OK : QW_ECUDA;
}

template <bool SPLIT>
static int launch_split(const CUtensorMap& ta, const CUtensorMap& tb, int bn, int M, int N, int K, int epi,
                        const GemmEpilogue& ep, cudaStream_t st) {
    if constexpr (SPLIT) {
        // narrow tiles for decode batches: a 4096-wide q|k|v on 32-wide tiles covers 128 SMs
        if (bn == 32 || bn == 64) {
            if (epi == EPI_QKV_ROPE || epi == EPI_RESID_ADD) return QW_EINVAL;
            if (bn == 32) {
                if (epi == EPI_STORE_F32) return launch_bn<32, EPI_STORE_F32, true, false>(ta, tb, M, N, K, ep, st);
                if (epi == EPI_ADD_ATOMIC) return launch_bn<32, EPI_ADD_ATOMIC, true, false>(ta, tb, M, N, K, ep, st);
                return launch_bn<32, EPI_SWIGLU, true, false>(ta, tb, M, N, K, ep, st);
            }
            if (epi == EPI_STORE_F32) return launch_bn<64, EPI_STORE_F32, true, false>(ta, tb, M, N, K, ep, st);
            if (epi == EPI_ADD_ATOMIC) return launch_bn<64, EPI_ADD_ATOMIC, true, false>(ta, tb, M, N, K, ep, st);
            return launch_bn<64, EPI_SWIGLU, true, false>(ta, tb, M, N, K, ep, st);
        }
    }
    if (bn == 256) {
        if (epi == EPI_STORE_F32) return launch_bn<256, EPI_STORE_F32, SPLIT, false>(ta, tb, M, N, K, ep, st);
        if (epi == EPI_RESID_ADD) return launch_bn<256, EPI_RESID_ADD, SPLIT, false>(ta, tb, M, N, K, ep, st);
        if (epi == EPI_ADD_ATOMIC) return launch_bn<256, EPI_ADD_ATOMIC, SPLIT, false>(ta, tb, M, N, K, ep, st);
        if (epi == EPI_QKV_ROPE) {
            if constexpr (SPLIT) return QW_EINVAL;
            else return launch_bn<256, EPI_QKV_ROPE, false, false>(ta, tb, M, N, K, ep, st);
        }
        return launch_bn<256, EPI_SWIGLU, SPLIT, false>(ta, tb, M, N, K, ep, st);
    }
    if (bn != 128) return QW_EINVAL;
    if (epi == EPI_STORE_F32) return launch_bn<128, EPI_STORE_F32, SPLIT, false>(ta, tb, M, N, K, ep, st);
    if (epi == EPI_RESID_ADD) return launch_bn<128, EPI_RESID_ADD, SPLIT, false>(ta, tb, M, N, K, ep, st);
    if (epi == EPI_ADD_ATOMIC) return launch_bn<128, EPI_ADD_ATOMIC, SPLIT, false>(ta, tb, M, N, K, ep, st);
    if (epi == EPI_QKV_ROPE) {
        if constexpr (SPLIT) return QW_EINVAL;
        else return launch_bn<128, EPI_QKV_ROPE, false, false>(ta, tb, M, N, K, ep, st);
    }
    return launch_bn<128, EPI_SWIGLU, SPLIT, false>(ta, tb, M, N, K, ep, st);
}

// Large-M products on 256-wide tiles in CTA pairs sharing the weight tile (tb_half: the same
// weight with 128-row boxes).
static int launch_mc(const CUtensorMap& ta, const CUtensorMap& tb_half, int M, int N, int K, int epi,
                     const GemmEpilogue& ep, cudaStream_t st) {
    if (epi == EPI_STORE_F32) return launch_bn<256, EPI_STORE_F32, false, true>(ta, tb_half, M, N, K, ep, st);
    if (epi == EPI_RESID_ADD) return launch_bn<256, EPI_RESID_ADD, false, true>(ta, tb_half, M, N, K, ep, st);
    if (epi == EPI_QKV_ROPE) return launch_bn<256, EPI_QKV_ROPE, false, true>(ta, tb_half, M, N, K, ep, st);
    if (epi == EPI_SWIGLU) return launch_bn<256, EPI_SWIGLU, false, true>(ta, tb_half, M, N, K, ep, st);
    return QW_EINVAL;
}

int gemm_bf16(const void* A, int lda_elems, const CUtensorMap& tmB, int bn, int M, int N, int K, int epi,
              const GemmEpilogue& ep, cudaStream_t st, const CUtensorMap* tmB_half) {
    if (M <= 0) return QW_OK;
    if (K % 64 || N % 32 || (bn != 128 && bn != 256 && !(ep.split && (bn == 32 || bn == 64)))) return QW_EINVAL;
    // split layout: ceil(M/64) tiles of 128 rows (64 hi rows, then their 64 lo rows)
    const uint64_t rows = ep.split ? (uint64_t)((M + 63) / 64) * 128 : (uint64_t)M;
    CUtensorMap ta;
    int rc = make_tmap_bf16(&ta, A, (uint64_t)K, rows, (uint64_t)lda_elems * 2, 64, 128);
    if (rc) return rc;
    if (tmB_half && !ep.split && bn == 256 && M > 128 && epi != EPI_ADD_ATOMIC)
        return launch_mc(ta, *tmB_half, M, N, K, epi, ep, st);
    return ep.split ? launch_split<true>(ta, tmB, bn, M, N, K, epi, ep, st)
                    : launch_split<false>(ta, tmB, bn, M, N, K, epi, ep, st);
}

}  // namespace qw
