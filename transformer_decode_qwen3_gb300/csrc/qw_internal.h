// Declarations shared by the translation units of libqwdecode (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qwdecode.h"

namespace qw {

// Counts every kernel launch the library makes (read by qw_kernel_launches).
void count_launches(int n);

// Launch `kern` on `st` with programmatic stream serialization: it may begin while the previous
// kernel of the stream finishes, so it must call pdl_wait() before touching dependent data.
template <typename... KArgs, typename... Args>
cudaError_t pdl_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Query heads per KV head (grouped-query attention of Step 5) the attention kernels take:
// 1 (MHA), 2, 4, 8 or 16 (MQA for 16 heads), with n_heads a multiple of n_kv_heads.
inline bool group_size_ok(int Hq, int Hkv) {
    if (Hkv < 1 || Hq < Hkv || Hq % Hkv) return false;
    const int G = Hq / Hkv;
    return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

// Record `msg` for qw_last_error_message() on this thread and return `code`.
int report_error(int code, const char* msg);

// EPI_ADD_ATOMIC: out += acc with fp32 atomics; the launch splits K so that every SM gets
// work (small-M products: decode batches).
// EPI_QKV_ROPE: the q|k|v projection of a prefill with everything that follows it up to the
// attention: QK-Norm and half-split RoPE of the q and k heads, q stored as bf16, k and v
// written into their cache pages (non-split products; output columns = whole heads).
enum { EPI_STORE_F32 = 0, EPI_RESID_ADD = 1, EPI_SWIGLU = 2, EPI_ADD_ATOMIC = 3, EPI_QKV_ROPE = 4 };

struct KvView {
    uint16_t* base;        // this layer's pages: [n_pages][2][n_kv][16][128]
    int64_t page_stride;   // elements per page (2 * n_kv * 16 * 128)
    int n_pages;
    const int* block_tables;
    int bt_stride;
};

struct QkvRope {
    const int* positions;   // [M] position of each row
    const int* tok_seq;     // [M] sequence (block-table row) of each row
    KvView kv;
    const float* q_norm;    // [128] fp32
    const float* k_norm;    // [128] fp32
    const float2* rope;     // [M][64] (cos, sin) of float32(pos * inv_freq[i]) (launch_rope_table)
    float eps;
    uint16_t* q_bf16;       // [M][Hq * 128]
    int Hq, Hkv;
};

struct GemmEpilogue {
    float* out;      // EPI_STORE_F32: out[m][n]; EPI_RESID_ADD: out[m][n] += acc
    uint16_t* act;   // EPI_SWIGLU: act[m][n/2] = bf16(silu(acc[2j]) * acc[2j+1])
    int ldo;         // row stride (elements) of out / act
    int* err;        // device error word
    int split;       // A holds hi/lo row pairs (see split_rows); SwiGLU output is written the same way
    QkvRope rope;    // EPI_QKV_ROPE only
    float2* tile_max = nullptr;  // EPI_STORE_F32 (nullable): [m][tile_ld] (max, argmax as int bits) per BN-column tile
    int tile_ld = 0;
};

// Rows an M-row activation occupies in the split (hi/lo) layout.
inline int split_rows(int M) { return (M + 63) / 64 * 128; }
// Small-M GEMMs (decode batches) take their activations as hi/lo bf16 pairs.
constexpr int SPLIT_MAX_M = 256;
// qw_generate writes the positions of this many steps at a time.
constexpr int GEN_CHUNK = 4096;

// Tensor map of a row-major bf16 matrix [rows][inner] with a (box_rows x box_inner)
// box and 128-byte swizzling (box_inner * 2 must be 128).
int make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_rows);

// C[M][N] (epilogue) = A[M][K] . B[N][K]^T; tmB must have box {64, bn}.  tmB_half (nullable):
// the same B with box {64, 128}; given with bn = 256 and M > 128 (not split, not split-K), the
// product runs in CTA pairs that multicast the shared weight tile.
int gemm_bf16(const void* A, int lda_elems, const CUtensorMap& tmB, int bn, int M, int N, int K, int epi,
              const GemmEpilogue& ep, cudaStream_t st, const CUtensorMap* tmB_half = nullptr);

// ---------------------------------------------------------------- per-op kernels
// out[i] = start + i, i < n.
int launch_positions(int* out, int start, int n, cudaStream_t st);
// (cos, sin) of the RoPE angles float32(positions[t] * inv_freq[i]), i < 64, for n rows.
int launch_rope_table(const int* positions, int n, const float* inv_freq, float2* tab, cudaStream_t st);
int launch_embed(const int* ids, int n, const uint16_t* E, int vocab, int D, float* x, int* err, cudaStream_t st);
int launch_rmsnorm_bf16(const float* x, const int* rows /*nullable*/, int n, int D, const float* w, float eps,
                        uint16_t* out, int split, cudaStream_t st);
int launch_qkv_post(const float* qkv, int n_tok, const int* positions, const int* tok_seq, int Hq, int Hkv,
                    const float* q_norm, const float* k_norm, const float* inv_freq, float eps, float* q_out /*nullable*/,
                    uint16_t* q_bf16 /*nullable*/, const KvView& kv, int* err, cudaStream_t st);
int launch_attn_prefill(const float* q, const int* positions, const int4* tiles, int n_tiles, int Hq, int Hkv,
                        const KvView& kv, uint16_t* out, int split, int* err, cudaStream_t st);
// Prefill attention on tcgen05 (q as bf16 [n_tok][Hq * 128]).
int launch_attn_prefill_tc(const uint16_t* q_bf16, int n_tok, const int* positions, const int4* tiles, int n_tiles,
                           int Hq, int Hkv, const KvView& kv, uint16_t* out, int split, int* err, cudaStream_t st);
int launch_attn_decode(const float* q, const int* positions, int batch, int Hq, int Hkv, const KvView& kv,
                       float* part, int max_splits, uint16_t* out, int split, int* err, int n_sm, cudaStream_t st);
// tile_part (nullable): [batch][n_part] per-tile (max, argmax) of the logits rows, left by the
// LM-head projection; argmax_hint (nullable, batch 1): the argmax of the logits row, already
// computed by the fused decode.  Greedy rows then skip the scan.
int launch_sample(const float* logits, int batch, int vocab, const qw_sample_params* params, uint64_t rng_counter,
                  int32_t* out_ids, const float2* tile_part, int n_part, const int* argmax_hint, int* err,
                  cudaStream_t st);
int launch_bf16_to_f32(const uint16_t* src, float* dst, int n, cudaStream_t st);
// Per-row int8 codes Q [rows][cols] (dense) and fp32 scales S [rows] of the bf16 matrix W (row
// stride ldw); W is overwritten with the dequantised bf16 values.
int launch_quantize_rows(uint16_t* W, int rows, int cols, int ldw, int8_t* Q, float* S, cudaStream_t st);

}  // namespace qw
