// misc.cu -- memory-bound elementwise kernels of libgbq and workspace sizing.
#include <algorithm>

#include "common.cuh"
#include "gemm.h"

namespace gbq {
namespace {

// y[m, n] = bf16(fmaf(fp32(acc[m, n]) * xs[m], ws[n], bias[n]))  (the page's dequant epilogue,
// "API": out = acc * x_scale[m] * w_scale[n] + bias[n]).  Blocks tile (column groups) x (rows): a thread
// owns 8 consecutive columns and strides over rows, two rows per step (four 16-byte accumulator loads in
// flight, two 16-byte stores) when the rows and pointers are 16-byte aligned (vec), else element by
// element.
__device__ __forceinline__ float dq_one(int32_t a, float x, float w, float b) {
    return __fmaf_rn(__fmul_rn(__int2float_rn(a), x), w, b);
}

__global__ void dequant_kernel(const int32_t *__restrict__ acc, int64_t ld_acc, const float *__restrict__ xs,
                               const float *__restrict__ ws, const __nv_bfloat16 *__restrict__ bias,
                               __nv_bfloat16 *__restrict__ y, int64_t ld_y, int64_t M, int64_t N, int vec,
                               unsigned int *status) {
    const int64_t n0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (n0 >= N) return;
    const int cols = (int)min((int64_t)8, N - n0);
    // Column operands, loaded once for all the thread's rows.
    float w[8], b[8];
    if (vec && cols == 8) {
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(ws + n0));
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(ws + n0) + 1);
        w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
        w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
        if (bias) {
            const uint4 bb = __ldg(reinterpret_cast<const uint4 *>(bias + n0));
            const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                b[2 * k] = __uint_as_float(bw[k] << 16);
                b[2 * k + 1] = __uint_as_float(bw[k] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) b[k] = 0.0f;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            w[k] = k < cols ? __ldg(ws + n0 + k) : 0.0f;
            b[k] = (k < cols && bias) ? __bfloat162float(bias[n0 + k]) : 0.0f;
        }
    }
    if (vec && cols == 8) {
        // Two rows per step: four 16-byte loads in flight per thread.
        for (int64_t m = blockIdx.y; m < M; m += 2 * (int64_t)gridDim.y) {
            const int64_t m2 = m + gridDim.y;
            const bool two = m2 < M;
            if (!(GBQ_IN_RANGE(status, m, 1, M) && GBQ_IN_RANGE(status, n0, 8, N))) continue;
            const int4 *ar = reinterpret_cast<const int4 *>(acc + m * ld_acc + n0);
            const int4 *ar2 = reinterpret_cast<const int4 *>(acc + (two ? m2 : m) * ld_acc + n0);
            const int4 a0 = __ldcs(ar), a1 = __ldcs(ar + 1);
            const int4 c0 = __ldcs(ar2), c1 = __ldcs(ar2 + 1);
            const float x = __ldg(xs + m), x2 = __ldg(xs + (two ? m2 : m));
            const int a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const int c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t o[4], o2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                __nv_bfloat162 h = __floats2bfloat162_rn(dq_one(a[2 * k], x, w[2 * k], b[2 * k]),
                                                         dq_one(a[2 * k + 1], x, w[2 * k + 1], b[2 * k + 1]));
                __nv_bfloat162 h2 = __floats2bfloat162_rn(dq_one(c[2 * k], x2, w[2 * k], b[2 * k]),
                                                          dq_one(c[2 * k + 1], x2, w[2 * k + 1], b[2 * k + 1]));
                o[k] = *reinterpret_cast<uint32_t *>(&h);
                o2[k] = *reinterpret_cast<uint32_t *>(&h2);
            }
            *reinterpret_cast<uint4 *>(y + m * ld_y + n0) = make_uint4(o[0], o[1], o[2], o[3]);
            if (two && GBQ_IN_RANGE(status, m2, 1, M))
                *reinterpret_cast<uint4 *>(y + m2 * ld_y + n0) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        }
        return;
    }
    for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
        if (!(GBQ_IN_RANGE(status, m, 1, M) && GBQ_IN_RANGE(status, n0, cols, N))) continue;
        const float x = __ldg(xs + m);
        const int32_t *ar = acc + m * ld_acc + n0;
        __nv_bfloat16 *yr = y + m * ld_y + n0;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < cols) yr[k] = __float2bfloat16_rn(dq_one(ar[k], x, w[k], b[k]));
    }
}

// Exact int8 -> fp16 (the tensor-core coding of quantized activations), 16 per thread-step.
__global__ void s8_to_f16_kernel(const int8_t *__restrict__ q, __half *__restrict__ out, int64_t n16,
                                 unsigned int *status) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
        if (!GBQ_IN_RANGE(status, 16 * i, 16, 16 * n16)) continue;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(q) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            o[2 * k] = s8pair_to_f16x2(__byte_perm(w[k], 0, 0x4140));      // bytes 0,1 -> 0x00B100B0
            o[2 * k + 1] = s8pair_to_f16x2(__byte_perm(w[k], 0, 0x4342));  // bytes 2,3
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out) + 2 * i;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// w[n, k] = bf16(fp32(w8[n, k]) * s[n]): dequant_weight with an identity rotation.
__global__ void scale_rows_s8_kernel(const int8_t *__restrict__ w8, const float *__restrict__ s,
                                     __nv_bfloat16 *__restrict__ w, int64_t N, int64_t K, unsigned int *status) {
    const int64_t per_row = K / 16;
    const int64_t total = N * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / per_row;
        if (!(GBQ_IN_RANGE(status, n, 1, N) && GBQ_IN_RANGE(status, 16 * i, 16, N * K))) continue;
        const float sc = __ldg(s + n);
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(w8) + i);
        const int8_t *b = reinterpret_cast<const int8_t *>(&v);
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn((float)b[2 * k], sc), __fmul_rn((float)b[2 * k + 1], sc));
            o[k] = *reinterpret_cast<uint32_t *>(&h);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(w) + 2 * i;
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g > 152 * 16) g = 152 * 16;
    return (int)(g < 1 ? 1 : g);
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

cudaError_t launch_dequant(const int32_t *acc, int64_t ld_acc, const float *xs, const float *ws, const void *bias,
                           void *y, int64_t ld_y, int64_t M, int64_t N, cudaStream_t st, unsigned int *status) {
    if (M == 0 || N == 0) return cudaSuccess;
    // 16-byte accesses: accumulator rows (4-byte elements) and output / bias rows (2-byte elements)
    // start on 16-byte boundaries.
    const int vec = (ld_acc % 4 == 0 && ld_y % 8 == 0 && ((uintptr_t)acc & 15) == 0 && ((uintptr_t)y & 15) == 0 &&
                     ((uintptr_t)ws & 15) == 0 && ((uintptr_t)bias & 15) == 0)
                        ? 1
                        : 0;
    constexpr int kThreads = 128;
    const int64_t col_groups = (N + 7) / 8;
    const unsigned gx = (unsigned)((col_groups + kThreads - 1) / kThreads);
    // One wave of 16 resident 128-thread blocks per SM; each thread then strides over rows (its column
    // operands loaded once).
    const int64_t want_rows = ((int64_t)152 * 16 + gx - 1) / gx;
    const unsigned gy = (unsigned)std::min<int64_t>(std::min<int64_t>(M, 65535), std::max<int64_t>(want_rows, 1));
    prof_begin(4, st);
    dequant_kernel<<<dim3(gx, gy), kThreads, 0, st>>>(acc, ld_acc, xs, ws, reinterpret_cast<const __nv_bfloat16 *>(bias),
                                                      reinterpret_cast<__nv_bfloat16 *>(y), ld_y, M, N, vec, status);
    prof_end(st);
    return cudaGetLastError();
}

cudaError_t launch_s8_to_f16(const int8_t *q, void *out, int64_t n, cudaStream_t st, unsigned int *status) {
    if (n % 16) return cudaErrorInvalidValue;
    prof_begin(4, st);
    s8_to_f16_kernel<<<grid_for(n / 16, 256), 256, 0, st>>>(q, reinterpret_cast<__half *>(out), n / 16, status);
    prof_end(st);
    return cudaGetLastError();
}

cudaError_t launch_scale_rows_s8(const int8_t *w8, const float *s, void *w, int64_t N, int64_t K, cudaStream_t st,
                                 unsigned int *status) {
    if (K % 16) return cudaErrorInvalidValue;
    prof_begin(4, st);
    scale_rows_s8_kernel<<<grid_for(N * K / 16, 256), 256, 0, st>>>(w8, s, reinterpret_cast<__nv_bfloat16 *>(w), N, K, status);
    prof_end(st);
    return cudaGetLastError();
}

// Workspace layouts (each region 256-byte aligned):
//   LINEAR / INT8_GEMM : q f16 [M][K], x_scale f32 [M]
//   FFN                : qx f16 [M][d], x_scale [M], g|u bf16 [M][2H], qh f16 [M][H], h_scale [M]
//   LINEAR_DX_INT8     : qd f16 [M][N], t f32 [M], dx_rot f32 [M][K]
// Preferred size: the minimum plus, for each quantized GEMM operand, the sums of |code| over each
// 1024-long block of every token row (int32 [M][ceil(K/1024)]), which let the int8 GEMM accumulate
// longer exact chunks when they are small.
size_t gemm_workspace_size_pref(int op, int64_t M, int64_t N, int64_t K, int64_t H) {
    const size_t base = gemm_workspace_size(op, M, N, K, H);
    if (M < 0 || base == 0) return base;
    const auto blocks = [](int64_t k) { return (size_t)((k + 1023) / 1024); };
    switch (op) {
        case GBQ_OP_LINEAR:
            return base + align256((size_t)M * 4 * blocks(K));
        case GBQ_OP_FFN:
            return base + align256((size_t)M * 4 * blocks(K)) + align256((size_t)M * 4 * blocks(H));
        case GBQ_OP_LINEAR_DX_INT8:  // the contraction runs over N
            return base + align256((size_t)M * 4 * blocks(N));
        default:
            return base;
    }
}

size_t gemm_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t H) {
    if (M < 0 || N < 0 || K < 0 || H < 0) return 0;
    switch (op) {
        case GBQ_OP_LINEAR:
        case GBQ_OP_INT8_GEMM:
            return align256((size_t)M * K * 2) + align256((size_t)M * 4);
        case GBQ_OP_FFN:
            return align256((size_t)M * K * 2) + align256((size_t)M * 4) + align256((size_t)M * 2 * H * 2) +
                   align256((size_t)M * H * 2) + align256((size_t)M * 4);
        case GBQ_OP_LINEAR_DX_INT8:
            return align256((size_t)M * N * 2) + align256((size_t)M * 4) + align256((size_t)M * K * 4);
        default:
            return 0;
    }
}

}  // namespace gbq
