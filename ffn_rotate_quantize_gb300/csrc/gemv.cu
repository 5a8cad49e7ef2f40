// gemv.cu -- decode GEMV path (M <= 8).
#include "gemm.h"

namespace gbq {
int launch_gemv(const void *, const int8_t *, const float *, const void *, void *, int64_t, int64_t, int64_t, int,
                int, int, cudaStream_t) {
    return GBQ_ENOTSUP;
}
}  // namespace gbq
