// Y = X W^T on the 5th-generation tensor core: bf16 operands, fp32 accumulation
// in tensor memory (TMEM), operands staged by TMA with 128-byte swizzling.
//
// Used for the projections of the article's Step 5 (q/k/v/o_proj), Step 6
// (gate/up/down_proj) and Step 8 (LM head) whenever a call carries more than a
// few rows (prefill, batched decode).
//
// One CTA computes a 128 x BN output tile.  Warp 0 (one lane) issues TMA loads
// into a STAGES-deep shared-memory ring, warp 1 (one lane) issues tcgen05.mma
// (K = 16 per instruction, 4 per 64-wide K block) and commits each stage back
// to the producer; all four warps then read the accumulator with tcgen05.ld
// (thread t owns output row t) and apply the fused epilogue.
//
// Split-operand mode (small M, e.g. decode batches): every activation row a is
// stored as two bf16 rows, hi = bf16(a) in tile rows 0..63 and lo = bf16(a - hi)
// in rows 64..127, so one M=128 MMA yields hi.W and lo.W side by side and the
// epilogue adds them: the activation enters with ~16 mantissa bits instead of 8,
// at no extra tensor-core work (the tile would otherwise be half empty).
#include <cudaTypedefs.h>

#include <vector>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {

template <int BN>
struct GemmCfg {
    static constexpr int BM = 128;
    static constexpr int BK = 64;                       // 64 bf16 = one 128-byte swizzle row
    static constexpr int STAGES = BN >= 256 ? 4 : 6;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = BN;                // power of two >= 32
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

QW_DEV float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Destination row of activation row m in the split layout (hi copy; lo is 64 rows further).
QW_DEV int split_row(int m) { return (m >> 6) * 128 + (m & 63); }

template <int BN, int EPI>
QW_DEV void epilogue_chunk(const float (&v)[32], int m, int n, const GemmEpilogue& ep) {
    if (EPI == EPI_STORE_F32) {
        float4* dst = (float4*)(ep.out + (size_t)m * ep.ldo + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
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

template <int BN, int EPI, bool SPLIT>
__global__ void __launch_bounds__(128, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        int M, int N, int K, GemmEpilogue ep) {
    using C = GemmCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* done = empty + C::STAGES;
    uint32_t* tmem_slot = (uint32_t*)(done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * C::BM;
    const int nk = K / C::BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // TMA producer
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::STAGES;
            const uint32_t ph = (kb / C::STAGES) & 1;
            if (!mbar_wait(&empty[s], ph ^ 1, ep.err)) break;
            if (*abort_flag) break;
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
            tma_load_2d(sA + s * C::A_BYTES, &tmA, kb * C::BK, m0, &full[s]);
            tma_load_2d(sB + s * C::B_BYTES, &tmB, kb * C::BK, n0, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = umma_idesc_bf16(C::BM, BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::STAGES;
            const uint32_t ph = (kb / C::STAGES) & 1;
            if (!mbar_wait(&full[s], ph, ep.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * C::A_BYTES), b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
            for (int k = 0; k < C::BK / 16; ++k) {
                umma_bf16(tmem, umma_desc_sw128(a0 + k * 32), umma_desc_sw128(b0 + k * 32), idesc,
                          (kb | k) != 0);
            }
            umma_commit(&empty[s]);
        }
        if (ok) {
            umma_commit(done);
        } else {
            *abort_flag = 1;
            mbar_arrive(done);
        }
    }
    __syncwarp();

    // Epilogue: thread t of the CTA owns accumulator row t.
    const bool ok = mbar_wait(done, 0, ep.err) && !*abort_flag;
    tc_fence_after();
    if (ok) {
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        float* xch = (float*)smem;  // split mode: lo rows handed to the hi rows (stages are idle now)
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            if (n0 + c0 >= N) break;  // CTA-uniform
            float v[32];
            tmem_ld32(trow + c0, v);
            if (SPLIT) {
                if (warp >= 2) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) xch[((warp - 2) * 32 + lane) * 33 + i] = v[i];
                }
                __syncthreads();
                if (warp < 2) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] += xch[(warp * 32 + lane) * 33 + i];
                    const int m = blockIdx.y * 64 + warp * 32 + lane;
                    if (m < M) epilogue_chunk<BN, EPI>(v, m, n0 + c0, ep);
                }
                __syncthreads();
            } else {
                const int m = m0 + warp * 32 + lane;
                if (m < M) epilogue_chunk<BN, EPI>(v, m, n0 + c0, ep);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
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

template <int BN, int EPI, bool SPLIT>
static int launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, const GemmEpilogue& ep,
                     cudaStream_t st) {
    using C = GemmCfg<BN>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemm_bf16_tc_kernel<BN, EPI, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM) != cudaSuccess)
            return QW_ECUDA;
        attr_set = true;
    }
    const int m_tiles = SPLIT ? (M + 63) / 64 : (M + C::BM - 1) / C::BM;
    dim3 grid((N + BN - 1) / BN, m_tiles);
    gemm_bf16_tc_kernel<BN, EPI, SPLIT><<<grid, 128, C::SMEM, st>>>(ta, tb, M, N, K, ep);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ECUDA;
}

template <bool SPLIT>
static int launch_split(const CUtensorMap& ta, const CUtensorMap& tb, int bn, int M, int N, int K, int epi,
                        const GemmEpilogue& ep, cudaStream_t st) {
    if (bn == 256) {
        if (epi == EPI_STORE_F32) return launch_bn<256, EPI_STORE_F32, SPLIT>(ta, tb, M, N, K, ep, st);
        if (epi == EPI_RESID_ADD) return launch_bn<256, EPI_RESID_ADD, SPLIT>(ta, tb, M, N, K, ep, st);
        return launch_bn<256, EPI_SWIGLU, SPLIT>(ta, tb, M, N, K, ep, st);
    }
    if (epi == EPI_STORE_F32) return launch_bn<128, EPI_STORE_F32, SPLIT>(ta, tb, M, N, K, ep, st);
    if (epi == EPI_RESID_ADD) return launch_bn<128, EPI_RESID_ADD, SPLIT>(ta, tb, M, N, K, ep, st);
    return launch_bn<128, EPI_SWIGLU, SPLIT>(ta, tb, M, N, K, ep, st);
}

int gemm_bf16(const void* A, int lda_elems, const CUtensorMap& tmB, int bn, int M, int N, int K, int epi,
              const GemmEpilogue& ep, cudaStream_t st) {
    if (M <= 0) return QW_OK;
    if (K % 64 || N % 32 || (bn != 128 && bn != 256)) return QW_EINVAL;
    // split layout: ceil(M/64) tiles of 128 rows (64 hi rows, then their 64 lo rows)
    const uint64_t rows = ep.split ? (uint64_t)((M + 63) / 64) * 128 : (uint64_t)M;
    CUtensorMap ta;
    int rc = make_tmap_bf16(&ta, A, (uint64_t)K, rows, (uint64_t)lda_elems * 2, 64, 128);
    if (rc) return rc;
    return ep.split ? launch_split<true>(ta, tmB, bn, M, N, K, epi, ep, st)
                    : launch_split<false>(ta, tmB, bn, M, N, K, epi, ep, st);
}

}  // namespace qw
