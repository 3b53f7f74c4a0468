// Fused persistent decode for small batches (declared here, used by qw_api.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace qw {

struct FusedDecode;

bool fused_supported(const FusedDecode* f, int batch);
int fused_decode(FusedDecode* f, const int* tokens, const int* positions, int batch, uint16_t* kv_base,
                 int64_t layer_elems, int64_t page_elems, int n_pages, const int* block_tables, int bt_stride,
                 float* logits, int* err, cudaStream_t st);
void fused_destroy(FusedDecode* f);

}  // namespace qw
