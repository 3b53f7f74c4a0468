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

template <int BN, int EPI>
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

    // Epilogue: thread t of the CTA owns output row m0 + t.
    const bool ok = mbar_wait(done, 0, ep.err) && !*abort_flag;
    tc_fence_after();
    const int m = m0 + warp * 32 + lane;
    if (ok) {
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            if (n0 + c0 >= N) break;  // warp-uniform
            float v[32];
            tmem_ld32(trow + c0, v);
            if (m >= M) continue;
            const int n = n0 + c0;
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
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float a0 = silu_f(v[4 * i]) * v[4 * i + 1];
                    const float a1 = silu_f(v[4 * i + 2]) * v[4 * i + 3];
                    pk[i] = pack_bf16x2(a0, a1);
                }
                uint4* dst = (uint4*)(ep.act + (size_t)m * ep.ldo + (n >> 1));
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
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

template <int BN, int EPI>
static int launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, const GemmEpilogue& ep,
                     cudaStream_t st) {
    using C = GemmCfg<BN>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemm_bf16_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM) != cudaSuccess)
            return QW_ECUDA;
        attr_set = true;
    }
    dim3 grid((N + BN - 1) / BN, (M + C::BM - 1) / C::BM);
    gemm_bf16_tc_kernel<BN, EPI><<<grid, 128, C::SMEM, st>>>(ta, tb, M, N, K, ep);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ECUDA;
}

int gemm_bf16(const void* A, int lda_elems, const CUtensorMap& tmB, int bn, int M, int N, int K, int epi,
              const GemmEpilogue& ep, cudaStream_t st) {
    if (M <= 0) return QW_OK;
    if (K % 64 || N % 32 || (bn != 128 && bn != 256)) return QW_EINVAL;
    CUtensorMap ta;
    int rc = make_tmap_bf16(&ta, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda_elems * 2, 64, 128);
    if (rc) return rc;
    if (bn == 256) {
        if (epi == EPI_STORE_F32) return launch_bn<256, EPI_STORE_F32>(ta, tmB, M, N, K, ep, st);
        if (epi == EPI_RESID_ADD) return launch_bn<256, EPI_RESID_ADD>(ta, tmB, M, N, K, ep, st);
        return launch_bn<256, EPI_SWIGLU>(ta, tmB, M, N, K, ep, st);
    }
    if (epi == EPI_STORE_F32) return launch_bn<128, EPI_STORE_F32>(ta, tmB, M, N, K, ep, st);
    if (epi == EPI_RESID_ADD) return launch_bn<128, EPI_RESID_ADD>(ta, tmB, M, N, K, ep, st);
    return launch_bn<128, EPI_SWIGLU>(ta, tmB, M, N, K, ep, st);
}

}  // namespace qw
