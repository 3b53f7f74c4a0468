// Causal prefill attention of the article's Step 5 on the 5th-generation tensor core.
//
// One CTA takes 128 / G consecutive query positions of one sequence and one KV head g,
// G = Hq / Hkv query heads per KV head (1, 2, 4, 8 or 16): its 128 MMA rows are those
// positions for each query head G g + hh of the group (rows hh * 128 / G ..), which share the
// KV head (grouped-query attention; G = 2 for Qwen3-0.6B: 64 positions x 2 heads).  Keys and
// values stream from the paged cache in tiles of 64 positions (4 pages), loaded by
// TMA through a 4-D view of the pool ([page][K/V, head][slot][dim], 16-slot boxes,
// 128-byte swizzle) into a 2-deep ring; two CTAs share an SM so that one's softmax
// overlaps the other's loads and MMAs.
//
//   warp 0      TMA producer (Q once, then K/V tiles)
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers, then
//               O += P_j V_j (V as an MN-major operand) into a TMEM accumulator
//   warps 2..5  softmax: thread = row; reads S_j from TMEM, masks keys beyond the
//               row's position, keeps the running max m and sum l, rescales O in
//               TMEM when m grows, writes P_j (bf16) to shared memory
// Scores are in log2 units (scale 1/sqrt(128) * log2 e); the output is O / l.
#include <cudaTypedefs.h>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {
namespace fa {

constexpr int BM = 128, BN = 64, HD = 128;
constexpr int CHUNK = 128 * 64 * 2;           // 128 rows x 64 bf16, one 128-byte-swizzle column block
constexpr int KCHUNK = BN * 64 * 2;           // 64 keys x 64 dims: one column block of a K or V tile
constexpr int Q_BYTES = 2 * CHUNK;            // 32 KB
constexpr int KV_STAGES = 2;                  // two CTAs per SM: their softmax warps interleave
constexpr int KV_STAGE = 4 * KCHUNK;          // K (2 blocks) + V (2 blocks) = 32 KB
constexpr int P_BYTES = BM * BN * 2;          // 16 KB: one 64-key block
// The dynamic shared-memory window starts 1024-byte aligned (checked at run time), so no
// alignment slack is reserved: two CTAs (2 x (112.25 + 1) KB) fit in one SM.
constexpr int SMEM = Q_BYTES + KV_STAGES * KV_STAGE + P_BYTES + 256;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;           // S0 [0,64), S1 [64,128), O [128,256)

// Instruction descriptor: bf16 x bf16 -> f32, M = 128, N = 128, A K-major, B K-major
// (S = Q K^T) or B MN-major (bit 16: O += P V with V stored [key][dim]).
constexpr uint32_t IDESC_S = umma_idesc_bf16(BM, BN);
constexpr uint32_t IDESC_PV = umma_idesc_bf16(BM, HD) | (1u << 16);

// MN-major operand with 128-byte swizzle: 8 K-rows of 128 bytes (64 MN elements) per
// atom; LBO = byte stride between atoms along MN, SBO = between 8-row groups along K.
QW_DEV uint64_t desc_mn_sw128(uint32_t smem_addr, uint32_t lbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

QW_DEV void tma_load_4d(void* smem_dst, const CUtensorMap* m, int c0, int c1, int c2, int c3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

QW_DEV int split_dst(int m) { return (m >> 6) * 128 + (m & 63); }

// 2^x on the special-function unit (relative error ~2^-22; P is rounded to bf16 next)
QW_DEV float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(THREADS, 2)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                           const int* __restrict__ positions, const int4* __restrict__ tiles,
                           const int* __restrict__ block_tables, int bt_stride, int n_pages, int Hq, int Hkv,
                           int lg, uint16_t* __restrict__ out, float scale_log2, int split, int* err) {
    // lg = log2(G): the tile holds 128 >> lg positions of each of the group's G query heads
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw;
    // 128-byte-swizzled tiles need 1024-byte aligned shared memory
    if (smem_u32(sm) & 1023) {
        if (threadIdx.x == 0) set_error(err, QW_EINVAL);
        return;
    }
    uint8_t* sQ = sm;
    uint8_t* sKV = sm + Q_BYTES;                       // stage s: K blocks at s*KV_STAGE, V blocks at +2*KCHUNK
    uint8_t* sP = sm + Q_BYTES + KV_STAGES * KV_STAGE;
    uint64_t* bars = (uint64_t*)(sP + P_BYTES);
    uint64_t* q_full = bars;
    // K and V of a stage are filled and released separately: a K slot frees as soon as its
    // S = Q K^T is done, so the next K loads start well before their tile is needed
    uint64_t* k_full = bars + 1;                   // [KV_STAGES]
    uint64_t* v_full = k_full + KV_STAGES;         // [KV_STAGES]
    uint64_t* k_empty = v_full + KV_STAGES;        // [KV_STAGES]
    uint64_t* v_empty = k_empty + KV_STAGES;       // [KV_STAGES]
    uint64_t* s_full = v_empty + KV_STAGES;        // [2]
    uint64_t* p_full = s_full + 2;
    uint64_t* o_done = p_full + 1;
    uint32_t* tmem_slot = (uint32_t*)(o_done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    // a CTA of this launch already gave up on a wait: end quickly instead of timing out again
    if (err && *(volatile int*)err == QW_ETIMEOUT) return;
    const int4 tile = tiles[blockIdx.x];
    const int seq = tile.x, row0 = tile.y, nrows = tile.z;
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pmax = positions[row0 + nrows - 1];
    const int nt = pmax < 0 ? 0 : pmax / BN + 1;
    const int* bt = block_tables + (size_t)seq * bt_stride;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) mbar_init(&s_full[s], 1);
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmKV);
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (nt > 0) {
            // the whole warp runs the producer loop: lanes look up one page id each, lane 0 issues
            constexpr int PPT = BN / QW_PAGE_SIZE;  // pages per key tile
            auto page_of = [&](int j) {
                const int pidx = j * PPT + (lane & (PPT - 1));
                int page = pidx < bt_stride ? __ldg(bt + pidx) : -1;
                if (page < 0 || page >= n_pages) {
                    if (lane < PPT && pidx * QW_PAGE_SIZE <= pmax) set_error(err, QW_ERANGE);
                    page = n_pages;  // out of the tensor map: TMA fills zeros
                }
                return page;
            };
            if (lane == 0) {
                // Q: rows hh * (128 >> lg) .. = head (g << lg) + hh, two 64-dim blocks each
                mbar_arrive_expect_tx(q_full, Q_BYTES);
                for (int hh = 0; hh < (1 << lg); ++hh)
                    for (int c = 0; c < 2; ++c)
                        tma_load_2d(sQ + c * CHUNK + hh * ((128 >> lg) * 128), &tmQ, ((g << lg) + hh) * HD + 64 * c,
                                    row0, q_full);
            }
            // issue order K_0, then K_{j+1}, V_j for j = 0, 1, ...: K runs one tile ahead of V
            auto issue = [&](int j, int page_lane, bool is_v) -> bool {
                const int st_i = j % KV_STAGES;
                uint64_t* emp = is_v ? &v_empty[st_i] : &k_empty[st_i];
                uint64_t* ful = is_v ? &v_full[st_i] : &k_full[st_i];
                bool ok = true;
                if (lane == 0) ok = mbar_wait(emp, ((j / KV_STAGES) & 1) ^ 1, err) && !*abort_flag;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) *abort_flag = 1;
                    return false;
                }
                uint8_t* st = sKV + st_i * KV_STAGE + (is_v ? 2 * KCHUNK : 0);
                if (lane == 0) mbar_arrive_expect_tx(ful, 2 * KCHUNK);
                for (int pi = 0; pi < PPT; ++pi) {
                    const int page = __shfl_sync(0xffffffffu, page_lane, pi);
                    if (lane == 0)
                        for (int c = 0; c < 2; ++c)
                            tma_load_4d(st + c * KCHUNK + pi * QW_PAGE_SIZE * 128, &tmKV, 64 * c, 0,
                                        is_v ? Hkv + g : g, page, ful);
                }
                return true;
            };
            int page_j = page_of(0);
            bool go = issue(0, page_j, false);
            for (int j = 0; j < nt && go; ++j) {
                const int page_next = j + 1 < nt ? page_of(j + 1) : 0;
                if (j + 1 < nt) go = issue(j + 1, page_next, false);
                if (go) go = issue(j, page_j, true);
                page_j = page_next;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && nt > 0) {
            const uint32_t aq = smem_u32(sQ), ap = smem_u32(sP);
            bool ok = mbar_wait(q_full, 0, err);
            auto issue_s = [&](int j) {
                const uint32_t k0 = smem_u32(sKV + (j % KV_STAGES) * KV_STAGE);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t qoff = (kk >> 2) * CHUNK + (kk & 3) * 32;
                    const uint32_t koff = (kk >> 2) * KCHUNK + (kk & 3) * 32;
                    umma_bf16(tmem + (j & 1) * BN, umma_desc_sw128(aq + qoff), umma_desc_sw128(k0 + koff), IDESC_S,
                              kk != 0);
                }
                umma_commit(&s_full[j & 1]);
                umma_commit(&k_empty[j % KV_STAGES]);   // the K slot is free once S_j is computed
            };
            if (ok) ok = mbar_wait(&k_full[0], 0, err);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int j = 0; j < nt && ok; ++j) {
                if (j + 1 < nt) {
                    if (!mbar_wait(&k_full[(j + 1) % KV_STAGES], ((j + 1) / KV_STAGES) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(j + 1);
                }
                if (!mbar_wait(p_full, j & 1, err) || !mbar_wait(&v_full[j % KV_STAGES], (j / KV_STAGES) & 1, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t v0 = smem_u32(sKV + (j % KV_STAGES) * KV_STAGE + 2 * KCHUNK);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // A = P (K-major, keys 16 kk ..), B = V (MN-major: keys 16 kk .. are rows 16 kk ..)
                    umma_bf16(tmem + 2 * BN, umma_desc_sw128(ap + kk * 32), desc_mn_sw128(v0 + kk * 16 * 128, KCHUNK),
                              IDESC_PV, (j | kk) != 0);
                }
                umma_commit(o_done);
                umma_commit(&v_empty[j % KV_STAGES]);
            }
            if (!ok) {
                *abort_flag = 1;
                // release the softmax warps
                for (int s = 0; s < 2; ++s) mbar_arrive(&s_full[s]);
                mbar_arrive(o_done);
            }
        }
    } else {
        // softmax warps 2..5: TMEM lane group (warp % 4), thread = row
        const int r = 32 * (warp & 3) + lane;
        const int hh = r >> (7 - lg), ri = r & ((128 >> lg) - 1);
        const int qp = ri < nrows ? positions[row0 + ri] : -1;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < nt; ++j) {
            if (!mbar_wait(&s_full[j & 1], (j >> 1) & 1, err) || *abort_flag) break;
            tc_fence_after();
            // S row: four 32-column TMEM loads in flight, one wait
            const uint32_t sbase = tmem + (j & 1) * BN + lane_off;
            const int kbase = j * BN;
            const bool full_tile = kbase + BN - 1 <= qp;     // no key of this tile is masked for this row
            float sv[BN];
            tmem_ld32_nowait(sbase + 0, sv + 0);
            tmem_ld32_nowait(sbase + 32, sv + 32);
            tmem_wait_ld();
            // row max over 8 independent chains (the loop is latency-bound: one or two warps per SMSP)
            float mx[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mx[c] = -INFINITY;
            if (full_tile) {
#pragma unroll
                for (int i = 0; i < BN; ++i) mx[i & 7] = fmaxf(mx[i & 7], sv[i]);
            } else {
#pragma unroll
                for (int i = 0; i < BN; ++i) {
                    if (kbase + i > qp) sv[i] = -INFINITY;
                    mx[i & 7] = fmaxf(mx[i & 7], sv[i]);
                }
            }
            const float rmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            // Lazy reference max: m moves (and O is rescaled) only when the tile's max exceeds it by
            // more than 8 (log2 units), so P <= 2^8; O and l share the reference, so O / l is exact.
            const float cand = rmax * scale_log2;
            float alpha = 1.f;
            if (cand > m + 8.f) {
                alpha = m == -INFINITY ? 0.f : ex2_approx(m - cand);
                m = cand;
            }
            const float neg = m == -INFINITY ? 0.f : -m;
            // p = 2^(s * scale - m) (masked keys: 2^-inf = 0), row sum, P row r packed as bf16;
            // all before waiting for the previous P V, which this work overlaps
            float sums[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) sums[c] = 0.f;
            uint32_t pk[BN / 2];
#pragma unroll
            for (int i = 0; i < BN; i += 2) {
                const float p0 = ex2_approx(fmaf(sv[i], scale_log2, neg));
                const float p1 = ex2_approx(fmaf(sv[i + 1], scale_log2, neg));
                sums[(i >> 1) & 7] += p0 + p1;
                pk[i >> 1] = pack_bf16x2(p0, p1);
            }
            const float sum = ((sums[0] + sums[1]) + (sums[2] + sums[3])) + ((sums[4] + sums[5]) + (sums[6] + sums[7]));
            // P_j may overwrite P_{j-1} and O may be rescaled once P_{j-1} V_{j-1} is done
            if (j > 0) {
                if (!mbar_wait(o_done, (j - 1) & 1, err) || *abort_flag) break;
                tc_fence_after();
                // tcgen05.ld/st are warp-collective: rescale when any row of the warp needs it
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {  // 64 columns at a time
                        float o[64];
                        const uint32_t ob = tmem + 2 * BN + lane_off + 64 * half;
                        tmem_ld32_nowait(ob + 0, o + 0);
                        tmem_ld32_nowait(ob + 32, o + 32);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 64; ++i) o[i] *= alpha;
                        tmem_st32_nowait(ob + 0, o + 0);
                        tmem_st32_nowait(ob + 32, o + 32);
                        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    }
                }
            }
#pragma unroll
            for (int unit = 0; unit < BN / 8; ++unit)   // 16-byte units of the row's 128 bytes
                *(uint4*)(sP + r * 128 + ((unit ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * unit], pk[4 * unit + 1], pk[4 * unit + 2], pk[4 * unit + 3]);
            l = l * alpha + sum;
            fence_proxy_async();   // the MMA reads P through the async proxy
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (nt > 0 && !*abort_flag && mbar_wait(o_done, (nt - 1) & 1, err)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t ld = (size_t)Hq * HD;
            const int h = (g << lg) + hh;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                float o[32];
                tmem_ld32(tmem + 2 * BN + lane_off + 32 * c, o);
                if (ri < nrows) {
                    const int row = row0 + ri;
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        hi[i] = pack_bf16x2(o[2 * i] * inv, o[2 * i + 1] * inv);
                        lo[i] = pack_bf16x2(o[2 * i] * inv - bf16_lo(hi[i]), o[2 * i + 1] * inv - bf16_hi(hi[i]));
                    }
                    const int dst_row = split ? split_dst(row) : row;
                    uint4* dst = (uint4*)(out + (size_t)dst_row * ld + h * HD + 32 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
                    if (split) {
                        uint4* dl = (uint4*)(out + (size_t)(dst_row + 64) * ld + h * HD + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dl[i] = make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace fa

static PFN_cuTensorMapEncodeTiled_v12000 g_encode_fa = nullptr;

static int encode(CUtensorMap* map, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                  const cuuint32_t* box) {
    if (!g_encode_fa) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return QW_ECUDA;
        g_encode_fa = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode_fa(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? QW_OK
               : QW_ECUDA;
}

int launch_attn_prefill_tc(const uint16_t* q_bf16, int n_tok, const int* positions, const int4* tiles, int n_tiles,
                           int Hq, int Hkv, const KvView& kv, uint16_t* out, int split, int* err, cudaStream_t st) {
    if (n_tiles <= 0) return QW_OK;
    if (!group_size_ok(Hq, Hkv)) return QW_EINVAL;
    const int G = Hq / Hkv, lg = 31 - __builtin_clz((unsigned)G);
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(fa::attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::SMEM) !=
            cudaSuccess)
            return QW_ECUDA;
        attr = true;
    }
    CUtensorMap tq, tkv;
    {   // q as [tokens][Hq * 128] bf16, boxes of 64 dims x (128 / G) tokens
        cuuint64_t dims[2] = {(cuuint64_t)Hq * 128, (cuuint64_t)n_tok};
        cuuint64_t strides[1] = {(cuuint64_t)Hq * 128 * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)(128 / G)};
        if (encode(&tq, const_cast<uint16_t*>(q_bf16), 2, dims, strides, box)) return QW_ECUDA;
    }
    {   // this layer's pool as [page][K/V x head][slot][dim], boxes of 64 dims x 16 slots
        cuuint64_t dims[4] = {128, QW_PAGE_SIZE, (cuuint64_t)2 * Hkv, (cuuint64_t)kv.n_pages};
        cuuint64_t strides[3] = {128 * 2, (cuuint64_t)QW_PAGE_SIZE * 128 * 2, (cuuint64_t)kv.page_stride * 2};
        cuuint32_t box[4] = {64, QW_PAGE_SIZE, 1, 1};
        if (encode(&tkv, kv.base, 4, dims, strides, box)) return QW_ECUDA;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf(128.f);
    fa::attn_prefill_tc_kernel<<<dim3(n_tiles, Hkv), fa::THREADS, fa::SMEM, st>>>(
        tq, tkv, positions, tiles, kv.block_tables, kv.bt_stride, kv.n_pages, Hq, Hkv, lg, out, scale_log2, split, err);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ECUDA;
}

}  // namespace qw
