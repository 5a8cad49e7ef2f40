// gemm_bf16.cu -- bf16 GEMM for linear_dx.
#include "gemm.h"

namespace gbq {
int launch_bf16_gemm_nn(const void *, const void *, void *, int64_t, int64_t, int64_t, unsigned int *, int,
                        cudaStream_t) {
    return gbq_fail(GBQ_ENOTSUP, "gbq_linear_dx: not built yet");
}
}  // namespace gbq
