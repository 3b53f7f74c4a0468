// Per-op kernels of the decoder pass (everything except the tensor-core GEMM).
// Step numbers refer to "Inside an LLM: Pure Python Inference for Qwen3-0.6B on MLX".
#include <float.h>

#include "qw_common.cuh"
#include "qw_internal.h"

namespace qw {

static unsigned long long g_launches = 0;
void count_launches(int n) { __atomic_fetch_add(&g_launches, (unsigned long long)n, __ATOMIC_RELAXED); }
unsigned long long launches_so_far() { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

static inline int check_launch() {
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? QW_OK : QW_ECUDA;
}

// Activation rows feeding a small-M projection are written as bf16 hi/lo pairs:
// row m goes to row split_dst(m) (hi) and split_dst(m) + 64 (lo = bf16(a - hi)).
QW_DEV int split_dst(int m) { return (m >> 6) * 128 + (m & 63); }
QW_DEV void store_bf16x2(uint16_t* base, size_t ld, int row, int col, float a, float b, int split) {
    const uint32_t hi = pack_bf16x2(a, b);
    if (!split) {
        *(uint32_t*)(base + (size_t)row * ld + col) = hi;
        return;
    }
    const int r = split_dst(row);
    *(uint32_t*)(base + (size_t)r * ld + col) = hi;
    *(uint32_t*)(base + (size_t)(r + 64) * ld + col) = pack_bf16x2(a - bf16_lo(hi), b - bf16_hi(hi));
}

// ---------------------------------------------------------------- Step 2: embedding
// x[t][:] = E[ids[t]][:] widened to fp32.  An id outside [0, vocab) gives a zero row
// and QW_ERANGE in the error word.
__global__ void embed_kernel(const int* __restrict__ ids, const uint16_t* __restrict__ E, int vocab, int D,
                             float* __restrict__ x, int* err) {
    pdl_wait();   // launched with pdl_launch: earlier kernels may still be running
    pdl_trigger();
    const int t = blockIdx.x;
    const int id = ids[t];
    const bool bad = id < 0 || id >= vocab;
    if (bad && threadIdx.x == 0) set_error(err, QW_ERANGE);
    float* xr = x + (size_t)t * D;
    for (int c = threadIdx.x * 8; c < D; c += blockDim.x * 8) {
        uint4 v = bad ? make_uint4(0, 0, 0, 0) : *(const uint4*)(E + (size_t)id * D + c);
        float4 lo = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
        float4 hi = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
        *(float4*)(xr + c) = lo;
        *(float4*)(xr + c + 4) = hi;
    }
}

int launch_embed(const int* ids, int n, const uint16_t* E, int vocab, int D, float* x, int* err, cudaStream_t st) {
    if (n <= 0) return QW_OK;
    if (pdl_launch(embed_kernel, dim3(n), dim3(128), 0, st, ids, E, vocab, D, x, err) != cudaSuccess) return QW_ECUDA;
    return check_launch();
}

// ---------------------------------------------------------------- Step 3: RMSNorm
// out[r] = bf16(x[src] / sqrt(mean(x[src]^2) + eps) * w), one warp per row.
__global__ void rmsnorm_bf16_kernel(const float* __restrict__ x, const int* __restrict__ rows, int n, int D,
                                    const float* __restrict__ w, float eps, uint16_t* __restrict__ out, int split) {
    pdl_wait();   // launched with pdl_launch: earlier kernels may still be running
    pdl_trigger();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= n) return;
    const int src = rows ? rows[r] : r;
    const float* xr = x + (size_t)src * D;
    float ss = 0.f;
    for (int c = lane * 4; c < D; c += 128) {
        float4 v = *(const float4*)(xr + c);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    const float s = 1.0f / sqrtf(ss / (float)D + eps);
    for (int c = lane * 4; c < D; c += 128) {
        float4 v = *(const float4*)(xr + c);
        float4 wv = *(const float4*)(w + c);
        store_bf16x2(out, D, r, c, v.x * s * wv.x, v.y * s * wv.y, split);
        store_bf16x2(out, D, r, c + 2, v.z * s * wv.z, v.w * s * wv.w, split);
    }
}

int launch_rmsnorm_bf16(const float* x, const int* rows, int n, int D, const float* w, float eps, uint16_t* out,
                        int split, cudaStream_t st) {
    if (n <= 0) return QW_OK;
    if (pdl_launch(rmsnorm_bf16_kernel, dim3((n + 7) / 8), dim3(256), 0, st, x, rows, n, D, w, eps, out, split) !=
        cudaSuccess)
        return QW_ECUDA;
    return check_launch();
}

// ------------------------------------- Step 5: QK-Norm, Step 4: RoPE, KV cache append
// One warp per (token, head) of the fused q|k|v projection output.  Lane l holds
// dims l, l+32, l+64, l+96, so both halves of every RoPE pair (i, i+64) sit in one
// lane.  q goes to q_out (fp32); k and v go, as bf16, to slot pos % 16 of page
// block_tables[seq][pos / 16].
__global__ void qkv_post_kernel(const float* __restrict__ qkv, const int* __restrict__ positions,
                                const int* __restrict__ tok_seq, int Hq, int Hkv, const float* __restrict__ q_norm,
                                const float* __restrict__ k_norm, const float* __restrict__ inv_freq, float eps,
                                float* __restrict__ q_out, uint16_t* __restrict__ q_bf16, KvView kv, int* err) {
    pdl_wait();   // launched with pdl_launch: earlier kernels may still be running
    pdl_trigger();
    const int t = blockIdx.x;
    const int hh = blockIdx.y * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int nh = Hq + 2 * Hkv;
    if (hh >= nh) return;
    const float* row = qkv + ((size_t)t * nh + hh) * QW_HEAD_DIM;
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = row[lane + 32 * i];
    const int pos = positions[t];
    if (hh < Hq + Hkv) {
        float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
        const float s = 1.0f / sqrtf(ss / (float)QW_HEAD_DIM + eps);
        const float* w = hh < Hq ? q_norm : k_norm;
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = y[i] * s * w[lane + 32 * i];
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // pairs (lane + 32j, lane + 32j + 64)
            const float ang = __fmul_rn((float)pos, inv_freq[lane + 32 * j]);
            float sn, cs;
            sincosf(ang, &sn, &cs);
            const float a = y[j], b = y[j + 2];
            y[j] = a * cs - b * sn;
            y[j + 2] = a * sn + b * cs;
        }
    }
    if (hh < Hq) {
        if (q_out) {
            float* dst = q_out + ((size_t)t * Hq + hh) * QW_HEAD_DIM;
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = y[i];
        }
        if (q_bf16) {
            uint16_t* qb = q_bf16 + ((size_t)t * Hq + hh) * QW_HEAD_DIM;
#pragma unroll
            for (int i = 0; i < 4; ++i) qb[lane + 32 * i] = f2bf(y[i]);
        }
        return;
    }
    const int seq = tok_seq[t];
    if (pos < 0 || pos >= kv.bt_stride * QW_PAGE_SIZE) {
        if (lane == 0) set_error(err, QW_ERANGE);
        return;
    }
    const int page = kv.block_tables[(size_t)seq * kv.bt_stride + pos / QW_PAGE_SIZE];
    if (page < 0 || page >= kv.n_pages) {
        if (lane == 0) set_error(err, QW_ERANGE);
        return;
    }
    const int which = hh < Hq + Hkv ? 0 : 1;
    const int g = (hh - Hq) - which * Hkv;
    uint16_t* dst = kv.base + (size_t)page * kv.page_stride + ((size_t)(which * Hkv + g) * QW_PAGE_SIZE +
                                                               (pos % QW_PAGE_SIZE)) * QW_HEAD_DIM;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = f2bf(y[i]);
}

__global__ void positions_kernel(int* __restrict__ out, int start, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = start + i;
}

int launch_positions(int* out, int start, int n, cudaStream_t st) {
    if (n <= 0) return QW_OK;
    positions_kernel<<<(n + 255) / 256, 256, 0, st>>>(out, start, n);
    return check_launch();
}

__global__ void rope_table_kernel(const int* __restrict__ positions, int n, const float* __restrict__ inv_freq,
                                  float2* __restrict__ tab) {
    pdl_wait();   // launched with pdl_launch: earlier kernels may still be running
    pdl_trigger();
    const int t = blockIdx.x, i = threadIdx.x;
    float sn, cs;
    sincosf(__fmul_rn((float)positions[t], inv_freq[i]), &sn, &cs);
    tab[(size_t)t * 64 + i] = make_float2(cs, sn);
}

int launch_rope_table(const int* positions, int n, const float* inv_freq, float2* tab, cudaStream_t st) {
    if (n <= 0) return QW_OK;
    if (pdl_launch(rope_table_kernel, dim3(n), dim3(64), 0, st, positions, n, inv_freq, tab) != cudaSuccess)
        return QW_ECUDA;
    return check_launch();
}

int launch_qkv_post(const float* qkv, int n_tok, const int* positions, const int* tok_seq, int Hq, int Hkv,
                    const float* q_norm, const float* k_norm, const float* inv_freq, float eps, float* q_out,
                    uint16_t* q_bf16, const KvView& kv, int* err, cudaStream_t st) {
    if (n_tok <= 0) return QW_OK;
    dim3 grid(n_tok, (Hq + 2 * Hkv + 3) / 4);
    if (pdl_launch(qkv_post_kernel, grid, dim3(128), 0, st, qkv, positions, tok_seq, Hq, Hkv, q_norm, k_norm, inv_freq,
                   eps, q_out, q_bf16, kv, err) != cudaSuccess)
        return QW_ECUDA;
    return check_launch();
}

// ---------------------------------------------------------------- mma.sync helpers
QW_DEV void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
QW_DEV void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
QW_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
QW_DEV void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
QW_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QW_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------- Step 5: causal attention over the cache
// Flash-style prefill attention.  A CTA takes one tile of up to 64 query rows of
// one sequence and one KV head; warps 0-3 serve query head 2g, warps 4-7 query
// head 2g+1 (the grouped-query sharing of Step 5), 16 rows each.  Keys and values
// stream from the paged cache in tiles of 64 positions (double-buffered cp.async,
// XOR-swizzled rows), S = QK^T and PV run on mma.sync m16n8k16 with an online
// softmax in fp32.  Key position j is visible to a query at position p iff j <= p.
constexpr int AP_KEYS = 64;
constexpr int AP_SMEM = 2 * 2 * AP_KEYS * QW_HEAD_DIM * 2;  // 2 buffers x (K, V) x 64 x 128 bf16

__global__ void __launch_bounds__(256) attn_prefill_kernel(const float* __restrict__ q,
                                                           const int* __restrict__ positions,
                                                           const int4* __restrict__ tiles, int Hq, int Hkv,
                                                           KvView kv, uint16_t* __restrict__ out, float scale_log2,
                                                           int split, int* err) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int4 tile = tiles[blockIdx.x];
    const int seq = tile.x, row0 = tile.y, nrows = tile.z;
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int h = g * 2 + (warp >> 2);
    const int r0 = (warp & 3) * 16;
    const int ra = r0 + gq, rb = ra + 8;
    const int pa = ra < nrows ? positions[row0 + ra] : -1;
    const int pb = rb < nrows ? positions[row0 + rb] : -1;
    const int pmax = positions[row0 + nrows - 1];

    uint32_t qf[8][4];
    {
        const float* qa = q + ((size_t)(row0 + ra) * Hq + h) * QW_HEAD_DIM;
        const float* qb = q + ((size_t)(row0 + rb) * Hq + h) * QW_HEAD_DIM;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int d0 = kk * 16 + 2 * tq;
            qf[kk][0] = pa >= 0 ? pack_bf16x2(qa[d0], qa[d0 + 1]) : 0u;
            qf[kk][1] = pb >= 0 ? pack_bf16x2(qb[d0], qb[d0 + 1]) : 0u;
            qf[kk][2] = pa >= 0 ? pack_bf16x2(qa[d0 + 8], qa[d0 + 9]) : 0u;
            qf[kk][3] = pb >= 0 ? pack_bf16x2(qb[d0 + 8], qb[d0 + 9]) : 0u;
        }
    }
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    const int nkt = pmax / AP_KEYS + 1;
    const int64_t head_off = (int64_t)g * QW_PAGE_SIZE * QW_HEAD_DIM;
    const int64_t v_off = (int64_t)Hkv * QW_PAGE_SIZE * QW_HEAD_DIM;
    const int* bt = kv.block_tables + (size_t)seq * kv.bt_stride;

    auto load_tile = [&](int kt, int buf) {
        uint8_t* sK = sm + buf * (2 * AP_KEYS * 256);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = threadIdx.x + i * 256;
            const int which = idx >> 10, r = (idx >> 4) & 63, c = idx & 15;
            const int pos = kt * AP_KEYS + r;
            const uint16_t* src = kv.base;
            int bytes = 0;
            if (pos <= pmax) {
                const int pidx = pos / QW_PAGE_SIZE;
                const int page = pidx < kv.bt_stride ? bt[pidx] : -1;
                if (page >= 0 && page < kv.n_pages) {
                    src = kv.base + (int64_t)page * kv.page_stride + which * v_off + head_off +
                          (pos % QW_PAGE_SIZE) * QW_HEAD_DIM + c * 8;
                    bytes = 16;
                } else if (c == 0) {
                    set_error(err, QW_ERANGE);
                }
            }
            uint8_t* dst = sK + which * (AP_KEYS * 256) + r * 256 + ((c ^ (r & 7)) << 4);
            cp_async16(smem_u32(dst), src, bytes);
        }
        cp_async_commit();
    };

    load_tile(0, 0);
    for (int kt = 0; kt < nkt; ++kt) {
        if (kt + 1 < nkt)
            load_tile(kt + 1, (kt + 1) & 1);
        else
            cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint8_t* sK = sm + (kt & 1) * (2 * AP_KEYS * 256);
        const uint8_t* sV = sK + AP_KEYS * 256;

        float s[8][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) {
                const int key = nb * 8 + (lane & 7);
                const int ch = kk2 * 4 + (lane >> 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3, smem_u32(sK + key * 256 + ((ch ^ (key & 7)) << 4)));
                mma16816(s[nb], qf[2 * kk2], b0, b1);
                mma16816(s[nb], qf[2 * kk2 + 1], b2, b3);
            }
        }
        const int kv0 = kt * AP_KEYS;
        float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int kp = kv0 + nb * 8 + 2 * tq + j;
                s[nb][j] = kp <= pa ? s[nb][j] * scale_log2 : -INFINITY;
                s[nb][2 + j] = kp <= pb ? s[nb][2 + j] * scale_log2 : -INFINITY;
                mx_a = fmaxf(mx_a, s[nb][j]);
                mx_b = fmaxf(mx_b, s[nb][2 + j]);
            }
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float al_a = mn_a == -INFINITY ? 1.f : exp2f(m_a - mn_a);
        const float al_b = mn_b == -INFINITY ? 1.f : exp2f(m_b - mn_b);
        m_a = mn_a;
        m_b = mn_b;
        float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                s[nb][j] = mn_a == -INFINITY ? 0.f : exp2f(s[nb][j] - mn_a);
                s[nb][2 + j] = mn_b == -INFINITY ? 0.f : exp2f(s[nb][2 + j] - mn_b);
                sum_a += s[nb][j];
                sum_b += s[nb][2 + j];
            }
        }
        l_a = l_a * al_a + sum_a;
        l_b = l_b * al_b + sum_b;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            o[nd][0] *= al_a;
            o[nd][1] *= al_a;
            o[nd][2] *= al_b;
            o[nd][3] *= al_b;
        }
#pragma unroll
        for (int kk2 = 0; kk2 < 4; ++kk2) {
            uint32_t a[4];
            a[0] = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
            a[1] = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
            a[2] = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
            a[3] = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
            for (int nd = 0; nd < 16; nd += 2) {
                const int mi = lane >> 3;
                const int key = kk2 * 16 + (mi & 1) * 8 + (lane & 7);
                const int ch = nd + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3, smem_u32(sV + key * 256 + ((ch ^ (key & 7)) << 4)));
                mma16816(o[nd], a, b0, b1);
                mma16816(o[nd + 1], a, b2, b3);
            }
        }
        __syncthreads();
    }
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
    const size_t ld = (size_t)Hq * QW_HEAD_DIM;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        const int d = h * QW_HEAD_DIM + nd * 8 + 2 * tq;
        if (ra < nrows) store_bf16x2(out, ld, row0 + ra, d, o[nd][0] * ia, o[nd][1] * ia, split);
        if (rb < nrows) store_bf16x2(out, ld, row0 + rb, d, o[nd][2] * ib, o[nd][3] * ib, split);
    }
}

int launch_attn_prefill(const float* q, const int* positions, const int4* tiles, int n_tiles, int Hq, int Hkv,
                        const KvView& kv, uint16_t* out, int split, int* err, cudaStream_t st) {
    if (n_tiles <= 0) return QW_OK;
    if (Hq != 2 * Hkv) return QW_EINVAL;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AP_SMEM) !=
            cudaSuccess)
            return QW_ECUDA;
        attr = true;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)QW_HEAD_DIM);
    attn_prefill_kernel<<<dim3(n_tiles, Hkv), 256, AP_SMEM, st>>>(q, positions, tiles, Hq, Hkv, kv, out,
                                                                  scale_log2, split, err);
    return check_launch();
}

// ---------------------------------------------- Step 5: decode attention, split over the cache
// One CTA per (split of the cached positions, slice of HPC query heads of one KV group,
// sequence): those query heads against up to chunk_pages pages of the group's KV head g
// (grouped-query sharing of Step 5: query head h reads KV head h / (Hq / Hkv)).  A group of
// G = Hq / Hkv heads is one slice when G <= 4, else G / 4 slices of 4 (each reads the group's
// pages).  Each warp walks pages; lane l covers keys (l >> 4) + 2i of the page and dims
// 8 (l & 15) .. +8.  The CTA writes an unnormalised partial (o[128], running max m in log2
// units, sum l) per query head; attn_combine_kernel merges the splits.
constexpr int AD_WARPS = 4;
constexpr int AD_PART = QW_HEAD_DIM + 2;

QW_DEV uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
QW_DEV float dot8(const float (&q)[8], uint4 k) {
    return q[0] * bf16_lo(k.x) + q[1] * bf16_hi(k.x) + q[2] * bf16_lo(k.y) + q[3] * bf16_hi(k.y) +
           q[4] * bf16_lo(k.z) + q[5] * bf16_hi(k.z) + q[6] * bf16_lo(k.w) + q[7] * bf16_hi(k.w);
}

template <int HPC>
__global__ void __launch_bounds__(AD_WARPS * 32) attn_decode_kernel(const float* __restrict__ q,
                                                                    const int* __restrict__ positions, int Hq,
                                                                    int Hkv, KvView kv, int chunk_pages,
                                                                    int n_splits, float* __restrict__ part,
                                                                    float scale_log2, int* err) {
    pdl_wait();   // launched with pdl_launch: earlier kernels may still be running
    pdl_trigger();
    const int G = Hq / Hkv, slices = G / HPC;
    const int split = blockIdx.x, g = blockIdx.y / slices, b = blockIdx.z;
    const int h0 = g * G + (blockIdx.y % slices) * HPC;   // first query head of this CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, dc = lane & 15;
    const int pos = positions[b];
    int L = pos + 1;
    if (pos < 0 || pos >= kv.bt_stride * QW_PAGE_SIZE) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) set_error(err, QW_ERANGE);
        L = 0;
    }
    const int np = (L + QW_PAGE_SIZE - 1) / QW_PAGE_SIZE;
    const int p_lo = split * chunk_pages, p_hi = min(np, p_lo + chunk_pages);
    float* pbase = part + (((size_t)b * Hq + h0) * n_splits + split) * AD_PART;   // head hh: + hh * n_splits * AD_PART
    if (p_lo >= p_hi) {
        if (threadIdx.x < HPC) {
            pbase[(size_t)threadIdx.x * n_splits * AD_PART + QW_HEAD_DIM] = -INFINITY;
            pbase[(size_t)threadIdx.x * n_splits * AD_PART + QW_HEAD_DIM + 1] = 0.f;
        }
        return;
    }
    float qh[HPC][8];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
        const float* q0 = q + ((size_t)b * Hq + h0 + hh) * QW_HEAD_DIM + dc * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) qh[hh][i] = q0[i] * scale_log2;
    }
    float m[HPC], l[HPC], o[HPC][8];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[hh][i] = 0.f;
    }
    const int* bt = kv.block_tables + (size_t)b * kv.bt_stride;
    const int64_t v_off = (int64_t)Hkv * QW_PAGE_SIZE * QW_HEAD_DIM;

    int next_page = p_lo + warp < p_hi ? __ldg(bt + p_lo + warp) : 0;
    for (int pi = p_lo + warp; pi < p_hi; pi += AD_WARPS) {
        const int page = next_page;  // the next lookup is in flight while this page is processed
        if (pi + AD_WARPS < p_hi) next_page = __ldg(bt + pi + AD_WARPS);
        if (page < 0 || page >= kv.n_pages) {
            if (lane == 0) set_error(err, QW_ERANGE);
            continue;
        }
        const uint16_t* kp = kv.base + (int64_t)page * kv.page_stride + (int64_t)g * QW_PAGE_SIZE * QW_HEAD_DIM +
                             half * QW_HEAD_DIM + dc * 8;
        uint4 kr[8], vr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) kr[i] = ldg_stream(kp + i * 2 * QW_HEAD_DIM);
#pragma unroll
        for (int i = 0; i < 8; ++i) vr[i] = ldg_stream(kp + v_off + i * 2 * QW_HEAD_DIM);
        float sc[HPC][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int hh = 0; hh < HPC; ++hh) sc[hh][i] = dot8(qh[hh], kr[i]);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int hh = 0; hh < HPC; ++hh) sc[hh][i] += __shfl_xor_sync(0xffffffffu, sc[hh][i], off);
        float nm[HPC];
#pragma unroll
        for (int hh = 0; hh < HPC; ++hh) {
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (pi * QW_PAGE_SIZE + half + 2 * i >= L) sc[hh][i] = -INFINITY;
                mx = fmaxf(mx, sc[hh][i]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            nm[hh] = fmaxf(m[hh], mx);   // finite: key pi*16 is always visible
            const float al = exp2f(m[hh] - nm[hh]);
            m[hh] = nm[hh];
            l[hh] *= al;
#pragma unroll
            for (int d = 0; d < 8; ++d) o[hh][d] *= al;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float v[8] = {bf16_lo(vr[i].x), bf16_hi(vr[i].x), bf16_lo(vr[i].y), bf16_hi(vr[i].y),
                                bf16_lo(vr[i].z), bf16_hi(vr[i].z), bf16_lo(vr[i].w), bf16_hi(vr[i].w)};
#pragma unroll
            for (int hh = 0; hh < HPC; ++hh) {
                const float e = exp2f(sc[hh][i] - nm[hh]);
                l[hh] += e;
#pragma unroll
                for (int d = 0; d < 8; ++d) o[hh][d] += e * v[d];
            }
        }
    }
    // the two key halves of a warp share m: add them
    __shared__ float s_o[AD_WARPS][HPC][QW_HEAD_DIM];
    __shared__ float s_m[AD_WARPS][HPC], s_l[AD_WARPS][HPC];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
        l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 16);
#pragma unroll
        for (int d = 0; d < 8; ++d) o[hh][d] += __shfl_xor_sync(0xffffffffu, o[hh][d], 16);
        if (half == 0) {
#pragma unroll
            for (int d = 0; d < 8; ++d) s_o[warp][hh][dc * 8 + d] = o[hh][d];
        }
        if (lane == 0) {
            s_m[warp][hh] = m[hh];
            s_l[warp][hh] = l[hh];
        }
    }
    __syncthreads();
    const int d = threadIdx.x;  // 128 threads = head_dim
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
        float M = -INFINITY;
        for (int w = 0; w < AD_WARPS; ++w)
            if (s_l[w][hh] > 0.f) M = fmaxf(M, s_m[w][hh]);
        float Ls = 0.f, O = 0.f;
        for (int w = 0; w < AD_WARPS; ++w) {
            if (s_l[w][hh] > 0.f) {
                const float sc = exp2f(s_m[w][hh] - M);
                Ls += s_l[w][hh] * sc;
                O += s_o[w][hh][d] * sc;
            }
        }
        float* dst = pbase + (size_t)hh * n_splits * AD_PART;
        dst[d] = O;
        if (d == 0) {
            dst[QW_HEAD_DIM] = M;
            dst[QW_HEAD_DIM + 1] = Ls;
        }
    }
}

__global__ void attn_combine_kernel(const float* __restrict__ part, int n_splits, int Hq,
                                    uint16_t* __restrict__ out, int split) {
    pdl_wait();   // launched with pdl_launch: earlier kernels may still be running
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x * 2;
    const float* base = part + ((size_t)b * Hq + h) * n_splits * AD_PART;
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s)
        if (base[s * AD_PART + QW_HEAD_DIM + 1] > 0.f) M = fmaxf(M, base[s * AD_PART + QW_HEAD_DIM]);
    float Ls = 0.f, O0 = 0.f, O1 = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float l = base[s * AD_PART + QW_HEAD_DIM + 1];
        if (l > 0.f) {
            const float sc = exp2f(base[s * AD_PART + QW_HEAD_DIM] - M);
            Ls += l * sc;
            O0 += base[s * AD_PART + d] * sc;
            O1 += base[s * AD_PART + d + 1] * sc;
        }
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    store_bf16x2(out, (size_t)Hq * QW_HEAD_DIM, b, h * QW_HEAD_DIM + d, O0 * inv, O1 * inv, split);
}

int launch_attn_decode(const float* q, const int* positions, int batch, int Hq, int Hkv, const KvView& kv,
                       float* part, int max_splits, uint16_t* out, int split, int* err, int n_sm, cudaStream_t st) {
    if (batch <= 0) return QW_OK;
    if (!group_size_ok(Hq, Hkv)) return QW_EINVAL;
    const int G = Hq / Hkv, hpc = G < 4 ? G : 4, slices = G / hpc;
    // pages per split: aim for ~8 CTAs per SM when every sequence is at full capacity
    long want = ((long)kv.bt_stride * batch * Hkv * slices + 8L * n_sm - 1) / (8L * n_sm);
    int chunk = 2;
    while (chunk < want && chunk < 32) chunk <<= 1;
    int n_splits = (kv.bt_stride + chunk - 1) / chunk;
    while (n_splits > max_splits) {
        chunk <<= 1;
        n_splits = (kv.bt_stride + chunk - 1) / chunk;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)QW_HEAD_DIM);
    const dim3 grid(n_splits, Hkv * slices, batch), block(AD_WARPS * 32);
    cudaError_t e;
    if (hpc == 1) e = pdl_launch(attn_decode_kernel<1>, grid, block, 0, st, q, positions, Hq, Hkv, kv, chunk, n_splits, part, scale_log2, err);
    else if (hpc == 2) e = pdl_launch(attn_decode_kernel<2>, grid, block, 0, st, q, positions, Hq, Hkv, kv, chunk, n_splits, part, scale_log2, err);
    else e = pdl_launch(attn_decode_kernel<4>, grid, block, 0, st, q, positions, Hq, Hkv, kv, chunk, n_splits, part, scale_log2, err);
    if (e != cudaSuccess) return QW_ECUDA;
    if (check_launch()) return QW_ECUDA;
    if (pdl_launch(attn_combine_kernel, dim3(Hq, batch), dim3(QW_HEAD_DIM / 2), 0, st, part, n_splits, Hq, out, split) !=
        cudaSuccess)
        return QW_ECUDA;
    return check_launch();
}

// ---------------------------------------------------------------- weight staging
__global__ void bf16_to_f32_kernel(const uint16_t* __restrict__ src, float* __restrict__ dst, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = __uint_as_float((uint32_t)src[i] << 16);
}

int launch_bf16_to_f32(const uint16_t* src, float* dst, int n, cudaStream_t st) {
    if (n <= 0) return QW_OK;
    bf16_to_f32_kernel<<<(n + 255) / 256, 256, 0, st>>>(src, dst, n);
    return check_launch();
}

// Weight-only int8 per output channel, one warp per row r of a bf16 matrix W (row stride ldw):
// S[r] = the smallest power of two >= max_c |W[r][c]| / 127 (that quotient in IEEE float32) and
// Q[r][c] = W[r][c] / S[r] rounded half to even (exact: a division by a power of two), within
// +-127; a zero row gets S = 0 and codes 0.  W[r][c] is replaced by bf16(Q[r][c] * S[r]), which
// is exact (seven magnitude bits times a power of two), so the paths that stream bf16 compute
// with exactly the weights the int8 path streams.
QW_DEV float pow2_ceil(float t) {
    const uint32_t b = __float_as_uint(t);
    if (!(t > 0.f)) return 0.f;
    if (b >= 0x00800000u) return (b & 0x007FFFFFu) ? __uint_as_float((b & 0x7F800000u) + 0x00800000u) : t;
    // subnormal: the next power of two of the integer significand, on the same 2^-149 grid
    return (b & (b - 1)) ? __uint_as_float(1u << (32 - __clz(b))) : t;
}

__global__ void quantize_rows_kernel(uint16_t* __restrict__ W, int rows, int cols, int ldw, int8_t* __restrict__ Q,
                                     float* __restrict__ S) {
    const int r = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (r >= rows) return;
    uint16_t* w = W + (size_t)r * ldw;
    float m = 0.f;
    for (int c = lane; c < cols; c += 32) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)w[c] << 16)));
    m = warp_max(m);
    const float sc = pow2_ceil(__fdiv_rn(m, 127.0f));
    if (lane == 0) S[r] = sc;
    int8_t* q = Q + (size_t)r * cols;
    for (int c = lane; c < cols; c += 32) {
        int v = 0;
        if (sc > 0.f) v = max(-127, min(127, __float2int_rn(__fdiv_rn(__uint_as_float((uint32_t)w[c] << 16), sc))));
        q[c] = (int8_t)v;
        w[c] = f2bf((float)v * sc);
    }
}

int launch_quantize_rows(uint16_t* W, int rows, int cols, int ldw, int8_t* Q, float* S, cudaStream_t st) {
    if (rows <= 0) return QW_OK;
    quantize_rows_kernel<<<(unsigned)(((size_t)rows * 32 + 255) / 256), 256, 0, st>>>(W, rows, cols, ldw, Q, S);
    return check_launch();
}

}  // namespace qw
