// One-kernel MiTA forward for short sequences (placeholder: no shape yet).
#include "fused.cuh"

namespace mita {
bool fused_supported(const Shape&, mita_dtype_t) { return false; }
cudaError_t run_fused(mita_plan_s*, const void*, const void*, const void*, void*, int32_t*, int32_t*, int,
                      cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace mita
