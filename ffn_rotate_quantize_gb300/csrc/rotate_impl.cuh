// rotate_impl.cuh -- fused Kronecker-Hadamard rotation (+ per-row INT8 quantize).
//
// What it computes (PyPI page "xpu-kernels 0.2.0", sections "Algorithm: fused
// ConvRot rotation" and "API"): for each row x of length K = G*n*n, each of the
// G contiguous groups X[n][n] (x[i*n+j] = X[i][j]) becomes
//     V = (H_n X H_n) / n        (= (H_n (x) H_n) x / sqrt(n*n), H_n symmetric)
// in fp32; then, per row, amax = max|v|, s = amax/127, q = clamp(rne(v/s), +-127).
//
// GB300 design: one group is owned by TPG = n/CPT threads.
//   pass 1  thread t holds CPT whole columns of X (n values each) loaded with
//           coalesced 4-byte loads, applies H_n down each column in registers
//           (H4/2 butterflies on base-4 digits; an unnormalised H2 on the top bit
//           when log2 n is odd);
//   swap    columns are written to a padded fp32 tile in shared memory and read
//           back as rows (float4 reads, padding makes both sides conflict-free);
//   pass 2  thread t holds CPT whole rows, applies H_n along each row;
//   quant   row amax by shuffles + one shared atomicMax per warp-group, then
//           IEEE division and round-half-even, and 16-byte vector stores of the
//           thread's contiguous output rows.
// Input variants fuse the producer: bf16 / fp32 activations, SiLU-GLU of two
// bf16 tensors, SiLU-GLU of two int32 accumulators through the dequant
// epilogue, and int8 weight rows times their fp32 scale (dequant_weight).
#pragma once

#include "common.cuh"

namespace gbq {

enum InKind { IN_BF16 = 0, IN_F32 = 1, IN_GLU_BF16 = 2, IN_S8_ROWSCALE = 3, IN_ACC_GLU = 4 };
enum OutKind { OUT_S8 = 0, OUT_F16Q = 1, OUT_BF16 = 2 };

struct RotArgs {
    const void *in0;        // x / g / W8 / acc_g
    const void *in1;        // u / acc_u (GLU inputs), else unused
    const float *in_scale;  // IN_S8_ROWSCALE: s[row]; IN_ACC_GLU: x_scale[row]
    const float *col_scale0;  // IN_ACC_GLU: s_gate[col]
    const float *col_scale1;  // IN_ACC_GLU: s_up[col]
    int64_t ld_in;          // elements between consecutive input rows
    void *out;              // int8 / f16-coded int / bf16, row stride K
    float *out_scale;       // per-row scale (quantizing outputs)
    int64_t M, K;
    int G;                  // groups per row
    int rows_per_cta;
};

__device__ __forceinline__ float bf16_to_float(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// SiLU(g) * u in fp32: g / (1 + exp(-g)) * u, IEEE operations throughout.
__device__ __forceinline__ float silu_mul(float g, float u) {
    float e = expf(-g);
    float d = __fadd_rn(1.0f, e);
    float sg = __fdiv_rn(g, d);
    return __fmul_rn(sg, u);
}

// Dequant epilogue value rounded to bf16 and widened back (the gate/up outputs).
__device__ __forceinline__ float dequant_bf16_value(int32_t acc, float xs, float ws) {
    float t = __fmul_rn(__int2float_rn(acc), xs);
    float r = __fmaf_rn(t, ws, 0.0f);
    return __bfloat162float(__float2bfloat16_rn(r));
}

// In-register H_n (normalised H4/2 on digits from bit 0; unnormalised H2 on the
// top bit when LOG is odd).
template <int LOG>
__device__ __forceinline__ void hadamard_regs(float (&v)[1 << LOG]) {
    constexpr int N = 1 << LOG;
#pragma unroll
    for (int d = 0; d + 1 < LOG; d += 2) {
#pragma unroll
        for (int base = 0; base < N; ++base) {
            if ((base >> d) & 3) continue;
            const float x0 = v[base], x1 = v[base | (1 << d)], x2 = v[base | (2 << d)], x3 = v[base | (3 << d)];
            const float s = __fadd_rn(__fadd_rn(x0, x1), __fadd_rn(x2, x3));
            v[base] = __fmaf_rn(0.5f, s, -x3);
            v[base | (1 << d)] = __fmaf_rn(0.5f, s, -x2);
            v[base | (2 << d)] = __fmaf_rn(0.5f, s, -x1);
            v[base | (3 << d)] = __fmaf_rn(0.5f, s, -x0);
        }
    }
    if (LOG & 1) {
        constexpr int h = N / 2;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float a = v[i], b = v[i + h];
            v[i] = __fadd_rn(a, b);
            v[i + h] = __fsub_rn(a, b);
        }
    }
}

// Largest CTA of a rotq launch: wide groups keep 128 values per thread in
// registers, so they get fewer threads and up to 255 registers each.
template <int LOGN>
struct RotqMaxThreads {
    static constexpr int value = LOGN >= 6 ? 256 : 512;
};

// The rotation of one group (pass 1, transpose through T, pass 2) for the
// thread (row, g, t); leaves this thread's CPT rows of the rotated group in v.
// Every thread of the CTA must call it (it contains one __syncthreads()).
template <int LOGN, int IN>
__device__ __forceinline__ void rot_group_core(const RotArgs &p, int64_t row, bool active, int g, int t, float *T,
                                               float (&v)[(LOGN >= 7) ? 1 : 2][1 << LOGN]) {
    constexpr int N = 1 << LOGN;
    constexpr int CPT = (LOGN >= 7) ? 1 : 2;
    constexpr int TPG = N / CPT;
    constexpr int P = N + 4;
    (void)TPG;
    // ---------------- pass 1: CPT columns j = CPT*t + e, all N rows i ----------------
    float c[CPT][N];
    const int64_t goff = (int64_t)g * N * N;
    if (active) {
        const int64_t rbase = row * p.ld_in + goff;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const int64_t idx = rbase + (int64_t)i * N + CPT * t;
            if constexpr (IN == IN_BF16) {
                if constexpr (CPT == 2) {
                    const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(p.in0) + idx / 2);
                    c[0][i] = __uint_as_float(w << 16);
                    c[1][i] = __uint_as_float(w & 0xFFFF0000u);
                } else {
                    c[0][i] = bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in0) + idx));
                }
            } else if constexpr (IN == IN_F32) {
                if constexpr (CPT == 2) {
                    const float2 f = __ldg(reinterpret_cast<const float2 *>(p.in0) + idx / 2);
                    c[0][i] = f.x;
                    c[1][i] = f.y;
                } else {
                    c[0][i] = __ldg(reinterpret_cast<const float *>(p.in0) + idx);
                }
            } else if constexpr (IN == IN_GLU_BF16) {
                if constexpr (CPT == 2) {
                    const uint32_t wg = __ldg(reinterpret_cast<const uint32_t *>(p.in0) + idx / 2);
                    const uint32_t wu = __ldg(reinterpret_cast<const uint32_t *>(p.in1) + idx / 2);
                    c[0][i] = silu_mul(__uint_as_float(wg << 16), __uint_as_float(wu << 16));
                    c[1][i] = silu_mul(__uint_as_float(wg & 0xFFFF0000u), __uint_as_float(wu & 0xFFFF0000u));
                } else {
                    c[0][i] = silu_mul(bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in0) + idx)),
                                       bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in1) + idx)));
                }
            } else if constexpr (IN == IN_S8_ROWSCALE) {
                const float sr = __ldg(p.in_scale + row);
                if constexpr (CPT == 2) {
                    const char2 q = __ldg(reinterpret_cast<const char2 *>(p.in0) + idx / 2);
                    c[0][i] = __fmul_rn((float)q.x, sr);
                    c[1][i] = __fmul_rn((float)q.y, sr);
                } else {
                    c[0][i] = __fmul_rn((float)__ldg(reinterpret_cast<const int8_t *>(p.in0) + idx), sr);
                }
            } else {  // IN_ACC_GLU
                const float xs = __ldg(p.in_scale + row);
                const int64_t col = goff + (int64_t)i * N + CPT * t;  // column within the H-wide row
#pragma unroll
                for (int e = 0; e < CPT; ++e) {
                    const int32_t ag = __ldg(reinterpret_cast<const int32_t *>(p.in0) + idx + e);
                    const int32_t au = __ldg(reinterpret_cast<const int32_t *>(p.in1) + idx + e);
                    const float gv = dequant_bf16_value(ag, xs, __ldg(p.col_scale0 + col + e));
                    const float uv = dequant_bf16_value(au, xs, __ldg(p.col_scale1 + col + e));
                    c[e][i] = silu_mul(gv, uv);
                }
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < CPT; ++e)
#pragma unroll
            for (int i = 0; i < N; ++i) c[e][i] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < CPT; ++e) hadamard_regs<LOGN>(c[e]);

    if (active) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if constexpr (CPT == 2) {
                *reinterpret_cast<float2 *>(&T[i * P + 2 * t]) = make_float2(c[0][i], c[1][i]);
            } else {
                T[i * P + t] = c[0][i];
            }
        }
    }
    __syncthreads();

    // ---------------- pass 2: CPT rows r = t + e*TPG, all N columns ----------------
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
        const int r = t + e * TPG;
#pragma unroll
        for (int j4 = 0; j4 < N / 4; ++j4) {
            const float4 f = active ? *reinterpret_cast<const float4 *>(&T[r * P + 4 * j4])
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            v[e][4 * j4 + 0] = f.x;
            v[e][4 * j4 + 1] = f.y;
            v[e][4 * j4 + 2] = f.z;
            v[e][4 * j4 + 3] = f.w;
        }
        hadamard_regs<LOGN>(v[e]);
        if (LOGN & 1) {
#pragma unroll
            for (int j = 0; j < N; ++j) v[e][j] = __fmul_rn(v[e][j], 0.5f);  // the two H2 levels: (1/sqrt2)^2
        }
    }

}

template <int LOGN, int IN, int OUT>
__global__ void __launch_bounds__(RotqMaxThreads<LOGN>::value) rotq_kernel(RotArgs p) {
    constexpr int N = 1 << LOGN;
    constexpr int CPT = (LOGN >= 7) ? 1 : 2;  // columns (pass 1) / rows (pass 2) per thread
    constexpr int TPG = N / CPT;              // threads per group
    constexpr int P = N + 4;                  // padded fp32 row stride in the swap tile
    constexpr int GSTRIDE = N * P + 16;       // floats per group tile
    (void)P;

    extern __shared__ __align__(16) float smem[];
    const int G = p.G;
    const int row_threads = G * TPG;
    const int tid = threadIdx.x;
    const int rloc = tid / row_threads;
    const int rem = tid - rloc * row_threads;
    const int g = rem / TPG;
    const int t = rem - g * TPG;
    const int64_t row = (int64_t)blockIdx.x * p.rows_per_cta + rloc;
    const bool active = row < p.M;
    float *T = smem + (size_t)(rloc * G + g) * GSTRIDE;
    unsigned *s_amax = reinterpret_cast<unsigned *>(smem + (size_t)p.rows_per_cta * G * GSTRIDE);
    if (tid < p.rows_per_cta) s_amax[tid] = 0u;
    const int64_t goff = (int64_t)g * N * N;

    float v[CPT][N];
    rot_group_core<LOGN, IN>(p, row, active, g, t, T, v);

    if constexpr (OUT == OUT_BF16) {
        if (!active) return;
#pragma unroll
        for (int e = 0; e < CPT; ++e) {
            const int r = t + e * TPG;
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + row * p.K + goff +
                                                   (int64_t)r * N);
#pragma unroll
            for (int j8 = 0; j8 < N / 8; ++j8) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(v[e][8 * j8 + 2 * h], v[e][8 * j8 + 2 * h + 1]);
                    w[h] = *reinterpret_cast<uint32_t *>(&b2);
                }
                dst[j8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        return;
    } else {
        // ---------------- row amax ----------------
        float m = 0.0f;
#pragma unroll
        for (int e = 0; e < CPT; ++e)
#pragma unroll
            for (int j = 0; j < N; ++j) m = fmaxf(m, fabsf(v[e][j]));
        constexpr int W = TPG < 32 ? TPG : 32;  // lanes of one group inside a warp
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((t & (W - 1)) == 0) atomicMax(&s_amax[rloc], __float_as_uint(m));
        __syncthreads();
        if (!active) return;
        const float amax = __uint_as_float(s_amax[rloc]);
        const float s = __fdiv_rn(amax, 127.0f);
        if (rem == 0) p.out_scale[row] = s;

#pragma unroll
        for (int e = 0; e < CPT; ++e) {
            const int r = t + e * TPG;
            int qv[N];
#pragma unroll
            for (int j = 0; j < N; ++j) {
                int q = 0;
                if (s != 0.0f) {
                    q = __float2int_rn(__fdiv_rn(v[e][j], s));
                    q = max(-127, min(127, q));
                }
                qv[j] = q;
            }
            if constexpr (OUT == OUT_S8) {
                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<int8_t *>(p.out) + row * p.K + goff +
                                                       (int64_t)r * N);
#pragma unroll
                for (int j16 = 0; j16 < N / 16; ++j16) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int b = 16 * j16 + 4 * h;
                        w[h] = (uint32_t)(qv[b] & 0xFF) | ((uint32_t)(qv[b + 1] & 0xFF) << 8) |
                               ((uint32_t)(qv[b + 2] & 0xFF) << 16) | ((uint32_t)(qv[b + 3] & 0xFF) << 24);
                    }
                    dst[j16] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            } else {  // OUT_F16Q: exact integers coded as fp16 (the tensor-core operand)
                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(p.out) + row * p.K + goff +
                                                       (int64_t)r * N);
#pragma unroll
                for (int j8 = 0; j8 < N / 8; ++j8) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        __half2 h2 = __halves2half2(__int2half_rn(qv[8 * j8 + 2 * h]),
                                                    __int2half_rn(qv[8 * j8 + 2 * h + 1]));
                        w[h] = *reinterpret_cast<uint32_t *>(&h2);
                    }
                    dst[j8] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
}

// Shared memory bytes for one launch of rotq_kernel.
__host__ __device__ inline size_t rotq_smem_bytes(int logn, int G, int rows_per_cta) {
    const int n = 1 << logn;
    return (size_t)rows_per_cta * G * (n * (n + 4) + 16) * sizeof(float) + (size_t)rows_per_cta * sizeof(unsigned) +
           16;
}

}  // namespace gbq
