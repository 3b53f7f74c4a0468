// Fused persistent decode for small batches: not built yet; every call reports
// "unsupported" so qw_decode_step takes the per-op path.
#include "../../include/qwdecode.h"
#include "qw_fused.h"

namespace qw {

bool fused_supported(const FusedDecode* f, int batch) { return f != nullptr && batch <= 8; }

int fused_decode(FusedDecode*, const int*, const int*, int, uint16_t*, int64_t, int64_t, int, const int*, int,
                 float*, int*, cudaStream_t) {
    return QW_EINVAL;
}

void fused_destroy(FusedDecode*) {}

}  // namespace qw
