// small-M kernel: not built yet.
#include "mmq_internal.h"
namespace mmq {
cudaError_t launch_gemm_small_m(mmq_q8_1_t, const uint8_t*, float*, int64_t, int64_t, int64_t,
                                int*, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace mmq
