// rotate_launch.cuh -- launch helper for rotq_kernel instantiations.
#pragma once

#include "kernels.h"

namespace gbq {

template <int LOGN, int IN, int OUT>
cudaError_t launch_rotq_t(RotArgs a, cudaStream_t st) {
    const int rt = rotq_row_threads(LOGN, a.G);
    if (rt > RotqMaxThreads<LOGN>::value) return cudaErrorNotSupported;
    a.rows_per_cta = rt >= 128 ? 1 : 128 / rt;
    const size_t smem = rotq_smem_bytes(LOGN, a.G, a.rows_per_cta);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    static bool attr_set = false;  // one attribute per instantiation
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(rotq_kernel<LOGN, IN, OUT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t grid = (a.M + a.rows_per_cta - 1) / a.rows_per_cta;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    prof_begin(0, st);
    rotq_kernel<LOGN, IN, OUT><<<(unsigned)grid, rt * a.rows_per_cta, smem, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

template <int IN, int OUT>
cudaError_t launch_rotq_logn(int logn, RotArgs a, cudaStream_t st) {
    switch (logn) {
        case 4: return launch_rotq_t<4, IN, OUT>(a, st);
        case 5: return launch_rotq_t<5, IN, OUT>(a, st);
        case 6: return launch_rotq_t<6, IN, OUT>(a, st);
        case 7: return launch_rotq_t<7, IN, OUT>(a, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace gbq
