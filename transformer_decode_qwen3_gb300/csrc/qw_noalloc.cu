// Decode attention for callers that cannot allocate device memory.
//
// Same kernels as qw_attn_decode; the only difference is where the split
// partials live: a fixed array in this library's device image instead of a
// context workspace, so the call needs no context and performs no allocation.
#include "qw_common.cuh"
#include "qw_internal.h"

// Partials of the split-KV decode attention, [batch][n_heads][splits][128 + 2] floats.
// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) float g_attn_scratch[QW_NOALLOC_SCRATCH_FLOATS];

namespace {
// Device address of g_attn_scratch in the current device's current context.  In host code
// the array's name is only a stand-in: kernels must get this address.  It is looked up on
// every call rather than cached, because it belongs to a context: after cudaDeviceReset, or
// with another context current on the same device, a cached address would be stale.  The
// lookup allocates nothing.
int scratch_on_current_device(float** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return QW_ECUDA;
    *out = (float*)p;
    return QW_OK;
}
}  // namespace

extern "C" int qw_attn_decode_noalloc(const float* q, const int32_t* positions, int32_t batch, int32_t n_heads,
                                      int32_t n_kv_heads, const uint16_t* kv_layer, int32_t n_pages,
                                      const int32_t* block_tables, int32_t bt_stride, uint16_t* out, void* stream) {
    if (!q || !positions || !kv_layer || !block_tables || !out)
        return qw::report_error(QW_EINVAL, "qw_attn_decode_noalloc: null argument");
    if (batch < 1 || !qw::group_size_ok(n_heads, n_kv_heads) || n_pages < 1 || bt_stride < 1)
        return qw::report_error(QW_EINVAL,
                                "qw_attn_decode_noalloc: bad size (n_heads must be n_kv_heads times 1, 2, 4, 8 or 16)");
    const long per_split = (long)batch * n_heads * (QW_HEAD_DIM + 2);
    const long max_splits = QW_NOALLOC_SCRATCH_FLOATS / per_split;
    if (max_splits < 1)
        return qw::report_error(QW_EINVAL, "qw_attn_decode_noalloc: batch * n_heads exceeds the fixed scratch");
    float* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != QW_OK)
        return qw::report_error(QW_ECUDA, "qw_attn_decode_noalloc: cudaGetSymbolAddress failed");
    int dev = 0, n_sm = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return qw::report_error(QW_ECUDA, "qw_attn_decode_noalloc: device query failed");
    qw::KvView kv{const_cast<uint16_t*>(kv_layer), (int64_t)2 * n_kv_heads * QW_PAGE_SIZE * QW_HEAD_DIM, n_pages,
                  block_tables, bt_stride};
    const int rc = qw::launch_attn_decode(q, positions, batch, n_heads, n_kv_heads, kv, scratch,
                                          (int)(max_splits < 4096 ? max_splits : 4096), out, 0, nullptr, n_sm,
                                          (cudaStream_t)stream);
    return rc == QW_OK ? QW_OK : qw::report_error(rc, "qw_attn_decode_noalloc: launch failed");
}
