// rotate_q.cu -- quantizing instantiations of the fused rotate+quantize kernel.
#include "rotate_launch.cuh"

namespace gbq {

cudaError_t launch_rotq(int logn, int in_kind, int out_kind, RotArgs a, cudaStream_t st) {
    if (out_kind == OUT_S8) {
        switch (in_kind) {
            case IN_BF16: return launch_rotq_logn<IN_BF16, OUT_S8>(logn, a, st);
            case IN_GLU_BF16: return launch_rotq_logn<IN_GLU_BF16, OUT_S8>(logn, a, st);
            case IN_ACC_GLU: return launch_rotq_logn<IN_ACC_GLU, OUT_S8>(logn, a, st);
            default: return cudaErrorNotSupported;
        }
    } else if (out_kind == OUT_F16Q) {
        switch (in_kind) {
            case IN_BF16: return launch_rotq_logn<IN_BF16, OUT_F16Q>(logn, a, st);
            case IN_GLU_BF16: return launch_rotq_logn<IN_GLU_BF16, OUT_F16Q>(logn, a, st);
            default: return cudaErrorNotSupported;
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace gbq
