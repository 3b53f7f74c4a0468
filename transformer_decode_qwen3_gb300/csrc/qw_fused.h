// Fused persistent decode for one sequence (declared here, used by qw_api.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace qw {

struct FusedDecode;

// Device pointers into the context's packed weights.
struct FusedWeights {
    const uint16_t* E;
    const float* final_norm;
    const float* inv_freq;
    std::vector<const uint16_t*> wqkv, wo, wgu, wd;   // wo: [hidden][n_heads*128], wd: [hidden][intermediate]
    std::vector<const float*> in_norm, post_norm, q_norm, k_norm;
    // Weight-only int8 (q8): the same matrices as int8 codes in the same layouts, with one fp32
    // scale per output channel (row of E, wqkv, wo, wgu, wd); the bf16 matrices above then hold
    // the dequantised values.
    bool q8 = false;
    const int8_t* Eq = nullptr;
    const float* sE = nullptr;
    std::vector<const int8_t*> wqkv_q, wo_q, wgu_q, wd_q;
    std::vector<const float*> s_qkv, s_o, s_gu, s_d;
};

// nullptr when the shape or the device does not fit the fused kernel.
FusedDecode* fused_create(const FusedWeights& w, int n_layers, int V, float eps, int hidden, int n_heads,
                          int n_kv_heads, int intermediate);
// The fused kernel takes batch 1 with block tables of at most 4088 pages (65408 positions).
bool fused_supported(const FusedDecode* f, int batch, int bt_stride);
int fused_decode(FusedDecode* f, const int* tokens, const int* positions, int batch, uint16_t* kv_base,
                 int64_t layer_elems, int64_t page_elems, int n_pages, const int* block_tables, int bt_stride,
                 float* logits, int* err, cudaStream_t st);
// Clear the step counters and accumulators (after a device error left them mid-step).
int fused_reset(FusedDecode* f, cudaStream_t st);
// Test hook: the next fused step waits at one place for an arrival that never comes, with a
// 2 ms limit, so that step ends in QW_ETIMEOUT (reported by qw_check) without a device fault.
int fused_inject_timeout(FusedDecode* f);
// Device int holding the argmax of the last fused step's logits.
const int* fused_argmax(const FusedDecode* f);
// Phase timestamps of the following fused steps (enable), copied out to host_out.
int fused_trace(FusedDecode* f, int enable, uint64_t* host_out, int64_t n, int64_t* n_needed);
void fused_destroy(FusedDecode* f);

}  // namespace qw
