// rotate_impl.cuh -- fused Kronecker-Hadamard rotation (+ per-row INT8 quantize).
//
// What it computes (PyPI page "xpu-kernels 0.2.0", sections "Algorithm: fused
// ConvRot rotation" and "API"): for each row x of length K = G*n*n, each of the
// G contiguous groups X[n][n] (x[i*n+j] = X[i][j]) becomes
//     V = (H_n X H_n) / n        (= (H_n (x) H_n) x / sqrt(n*n), H_n symmetric)
// in fp32; then, per row, amax = max|v|, s = amax/127, q = clamp(rne(v/s), +-127).
//
// GB300 design.  One group is owned by TPG threads; every value is carried in a
// float2 pair so that each Hadamard level runs on the packed fp32x2 pipe:
//   n <= 64  pass 1: thread t holds columns 2t, 2t+1 (pair = the two columns);
//            pass 2: thread t holds rows t, t+n/2     (pair = the two rows);
//   n == 128 pass 1: thread t holds column t, pair = (row i, row i+64);
//            pass 2: thread t holds row t,    pair = (col j, col j+64).
// Pass 1 applies H_n down the columns, a padded shared tile of float2 pairs
// turns columns into rows (16-byte accesses, conflict-free), pass 2 applies H_n
// along the rows.  Levels run in a fixed order (H4/2 on base-4 digits from the
// low bit up, then the unnormalised H2 on the top bit when log2 n is odd, whose
// two sqrt(2) factors are removed by one final exact halving), so every kernel
// that uses this core produces bit-identical rotated values.
// Quantize: r = 1/s once per row; t = v*r; the code is rint(t) (read out of the
// low byte of t + 1.5*2^23), which equals rne(fl(v/s)) unless t lies within
// 1e-4 of a half-integer (|t - v/s| <= 128*2^-23 and |fl(v/s) - v/s| <= 2^-18
// bound the difference far below that); such threads, and rows with a scale
// too small for a finite reciprocal, are recomputed with IEEE division.
#pragma once

#include "common.cuh"

namespace gbq {

enum InKind { IN_BF16 = 0, IN_F32 = 1, IN_GLU_BF16 = 2, IN_S8_ROWSCALE = 3, IN_ACC_GLU = 4 };
enum OutKind { OUT_S8 = 0, OUT_F16Q = 1, OUT_BF16 = 2 };

struct RotArgs {
    const void *in0;          // x / g / W8 / acc_g
    const void *in1;          // u / acc_u (GLU inputs), else unused
    const float *in_scale;    // IN_S8_ROWSCALE: s[row]; IN_ACC_GLU: x_scale[row]
    const float *col_scale0;  // IN_ACC_GLU: s_gate[col]
    const float *col_scale1;  // IN_ACC_GLU: s_up[col]
    int64_t ld_in;            // elements between consecutive input rows
    void *out;                // int8 / f16-coded int / bf16, row stride K
    float *out_scale;         // per-row scale (quantizing outputs)
    int64_t M, K;
    int G;                    // groups per row
    int rows_per_cta;
};

// Shapes of the packed two-pass rotation of one n x n group.
template <int LOGN>
struct RotGeom {
    static constexpr int N = 1 << LOGN;
    static constexpr bool PAIR_TOP = LOGN >= 7;        // n = 128: pairs across the top index bit
    static constexpr int TPG = PAIR_TOP ? N : N / 2;   // threads per group
    static constexpr int NP = PAIR_TOP ? N / 2 : N;    // float2 pairs per thread per pass
    static constexpr int ROWS = PAIR_TOP ? N : N / 2;  // rows of the swap tile
    static constexpr int COLS = PAIR_TOP ? N / 2 : N;  // float2 columns of the swap tile
    static constexpr int PP = COLS + 2;                // padded row stride (float2)
    static constexpr int TILE = ROWS * PP + 8;         // float2 per group tile
};

// Largest CTA of a rotq launch: wide groups keep 128 values per thread in
// registers, so they get fewer threads and up to 255 registers each.
template <int LOGN>
struct RotqMaxThreads {
    static constexpr int value = LOGN >= 6 ? 256 : 512;
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

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// One H4/2 level on index digit (bits D, D+1) of a pair array: for each group of
// four, s = (x0 + x1) + (x2 + x3), out_i = s/2 - x_(3-i), on both halves at once.
template <int NP, int D>
__device__ __forceinline__ void h4_level(float2 (&v)[NP]) {
    const float2 half2 = f2(0.5f, 0.5f);
    const float2 mone2 = f2(-1.0f, -1.0f);
#pragma unroll
    for (int base = 0; base < NP; ++base) {
        if ((base >> D) & 3) continue;
        const float2 x0 = v[base], x1 = v[base | (1 << D)], x2 = v[base | (2 << D)], x3 = v[base | (3 << D)];
        const float2 s = __fadd2_rn(__fadd2_rn(x0, x1), __fadd2_rn(x2, x3));
        const float2 h = __fmul2_rn(s, half2);  // exact halving
        v[base] = __ffma2_rn(x3, mone2, h);
        v[base | (1 << D)] = __ffma2_rn(x2, mone2, h);
        v[base | (2 << D)] = __ffma2_rn(x1, mone2, h);
        v[base | (3 << D)] = __ffma2_rn(x0, mone2, h);
    }
}

// H_n on the index of a pair array (LOG index bits): H4/2 digits from bit 0 up,
// then (odd LOG) the unnormalised H2 on the top index bit.
template <int LOG>
__device__ __forceinline__ void hadamard_pairs(float2 (&v)[1 << LOG]) {
    constexpr int NP = 1 << LOG;
    if constexpr (LOG >= 2) h4_level<NP, 0>(v);
    if constexpr (LOG >= 4) h4_level<NP, 2>(v);
    if constexpr (LOG >= 6) h4_level<NP, 4>(v);
    if constexpr (LOG & 1) {
        constexpr int h = NP / 2;
        const float2 mone2 = f2(-1.0f, -1.0f);
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float2 a = v[i], b = v[i + h];
            v[i] = __fadd2_rn(a, b);
            v[i + h] = __ffma2_rn(b, mone2, a);
        }
    }
}

// H_n for the pass layout of RotGeom<LOGN>: for n = 128 the pair holds the top
// index bit, so the H4 digits run packed and the H2 combines the two halves.
template <int LOGN>
__device__ __forceinline__ void hadamard_pass(float2 (&v)[RotGeom<LOGN>::NP]) {
    if constexpr (RotGeom<LOGN>::PAIR_TOP) {
        hadamard_pairs<LOGN - 1>(v);
#pragma unroll
        for (int i = 0; i < RotGeom<LOGN>::NP; ++i) {
            const float a = v[i].x, b = v[i].y;
            v[i] = f2(__fadd_rn(a, b), __fsub_rn(a, b));
        }
    } else {
        hadamard_pairs<LOGN>(v);
    }
}

// Load one input element (idx into in0/in1; col = column within the row) as fp32.
template <int IN>
__device__ __forceinline__ float load_in(const RotArgs &p, int64_t row, int64_t idx, int64_t col) {
    if constexpr (IN == IN_BF16) {
        return bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in0) + idx));
    } else if constexpr (IN == IN_F32) {
        return __ldg(reinterpret_cast<const float *>(p.in0) + idx);
    } else if constexpr (IN == IN_GLU_BF16) {
        return silu_mul(bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in0) + idx)),
                        bf16_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in1) + idx)));
    } else if constexpr (IN == IN_S8_ROWSCALE) {
        return __fmul_rn((float)__ldg(reinterpret_cast<const int8_t *>(p.in0) + idx), __ldg(p.in_scale + row));
    } else {  // IN_ACC_GLU
        const float xs = __ldg(p.in_scale + row);
        const float gv = dequant_bf16_value(__ldg(reinterpret_cast<const int32_t *>(p.in0) + idx), xs,
                                            __ldg(p.col_scale0 + col));
        const float uv = dequant_bf16_value(__ldg(reinterpret_cast<const int32_t *>(p.in1) + idx), xs,
                                            __ldg(p.col_scale1 + col));
        return silu_mul(gv, uv);
    }
}

// Load two adjacent input elements (idx even) as an fp32 pair.
template <int IN>
__device__ __forceinline__ float2 load_in2(const RotArgs &p, int64_t row, int64_t idx, int64_t col) {
    if constexpr (IN == IN_BF16) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(p.in0) + idx / 2);
        return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    } else if constexpr (IN == IN_F32) {
        return __ldg(reinterpret_cast<const float2 *>(p.in0) + idx / 2);
    } else if constexpr (IN == IN_GLU_BF16) {
        const uint32_t wg = __ldg(reinterpret_cast<const uint32_t *>(p.in0) + idx / 2);
        const uint32_t wu = __ldg(reinterpret_cast<const uint32_t *>(p.in1) + idx / 2);
        return f2(silu_mul(__uint_as_float(wg << 16), __uint_as_float(wu << 16)),
                  silu_mul(__uint_as_float(wg & 0xFFFF0000u), __uint_as_float(wu & 0xFFFF0000u)));
    } else if constexpr (IN == IN_S8_ROWSCALE) {
        const float sr = __ldg(p.in_scale + row);
        const char2 q = __ldg(reinterpret_cast<const char2 *>(p.in0) + idx / 2);
        return __fmul2_rn(f2((float)q.x, (float)q.y), f2(sr, sr));
    } else {
        return f2(load_in<IN>(p, row, idx, col), load_in<IN>(p, row, idx + 1, col + 1));
    }
}

// The rotation of one group (pass 1, transpose through T, pass 2) for the
// thread (row, g, t); leaves this thread's pass-2 pairs in v.  Every thread of
// the CTA must call it (it contains one __syncthreads()).  Inactive threads
// touch neither global memory nor the tile and return zeros.
template <int LOGN, int IN>
__device__ __forceinline__ void rot_group_core(const RotArgs &p, int64_t row, bool active, int g, int t, float2 *T,
                                               float2 (&v)[RotGeom<LOGN>::NP]) {
    using Geo = RotGeom<LOGN>;
    constexpr int N = Geo::N, NP = Geo::NP, PP = Geo::PP;
    float2 c[NP];
    const int64_t goff = (int64_t)g * N * N;
    // ---------------- pass 1: load columns, H_n down each column ----------------
    if (active) {
        const int64_t rbase = row * p.ld_in + goff;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            if constexpr (Geo::PAIR_TOP) {  // column t, rows i and i + N/2
                c[i] = f2(load_in<IN>(p, row, rbase + (int64_t)i * N + t, goff + (int64_t)i * N + t),
                          load_in<IN>(p, row, rbase + (int64_t)(i + N / 2) * N + t,
                                      goff + (int64_t)(i + N / 2) * N + t));
            } else {  // columns 2t, 2t+1 of row i
                c[i] = load_in2<IN>(p, row, rbase + (int64_t)i * N + 2 * t, goff + (int64_t)i * N + 2 * t);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < NP; ++i) c[i] = f2(0.f, 0.f);
    }
    hadamard_pass<LOGN>(c);
    if (active) {
        if constexpr (Geo::PAIR_TOP) {
            // tile row i, float2 column (t mod N/2), half (t div N/2) <- X[i][t]
            float *Tf = reinterpret_cast<float *>(T);
            const int cc = t & (N / 2 - 1), hh = t >> (LOGN - 1);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                Tf[(i * PP + cc) * 2 + hh] = c[i].x;
                Tf[((i + N / 2) * PP + cc) * 2 + hh] = c[i].y;
            }
        } else {
            // tile row i' holds pairs (X[i'][j], X[i' + N/2][j])
#pragma unroll
            for (int i = 0; i < N / 2; ++i)
                *reinterpret_cast<float4 *>(&T[i * PP + 2 * t]) =
                    make_float4(c[i].x, c[i + N / 2].x, c[i].y, c[i + N / 2].y);
        }
    }
    __syncthreads();
    // ---------------- pass 2: read row pairs, H_n along each row ----------------
#pragma unroll
    for (int j2 = 0; j2 < NP / 2; ++j2) {
        const float4 f =
            active ? *reinterpret_cast<const float4 *>(&T[t * PP + 2 * j2]) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[2 * j2] = f2(f.x, f.y);
        v[2 * j2 + 1] = f2(f.z, f.w);
    }
    hadamard_pass<LOGN>(v);
    if (LOGN & 1) {
        const float2 half2 = f2(0.5f, 0.5f);
#pragma unroll
        for (int j = 0; j < NP; ++j) v[j] = __fmul2_rn(v[j], half2);  // the two H2 levels: (1/sqrt2)^2
    }
}

// Element offset, within the row, of output half h of thread t in group g:
//   n <= 64 : half 0 = row t, half 1 = row t + n/2 (n contiguous values: v[j].x / v[j].y)
//   n == 128: half 0 = row t, first 64 values (v[j].x); half 1 = row t, last 64 (v[j].y)
template <int LOGN>
__device__ __forceinline__ int64_t out_offset(int g, int t, int h) {
    using Geo = RotGeom<LOGN>;
    constexpr int N = Geo::N;
    if constexpr (Geo::PAIR_TOP)
        return (int64_t)g * N * N + (int64_t)t * N + h * (N / 2);
    else
        return (int64_t)g * N * N + (int64_t)(t + h * (N / 2)) * N;
}

__device__ __forceinline__ float pair_max_abs(const float2 a) { return fmaxf(fabsf(a.x), fabsf(a.y)); }

// Codes rint(v * r) of a pair array, four int8 per word per half: words[h][w]
// holds elements 4w..4w+3 of half h.  Returns false if some t = v*r lies within
// 1e-4 of a half-integer, where the code might differ from rne(fl(v/s)).
template <int NP>
__device__ __forceinline__ bool quant_codes_fast(const float2 (&v)[NP], float r, uint32_t (&words)[2][NP / 4]) {
    const float2 r2 = f2(r, r);
    const float2 magic = f2(12582912.0f, 12582912.0f);  // 1.5 * 2^23: t + magic rounds t to an integer (RNE)
    const float2 nmagic = f2(-12582912.0f, -12582912.0f);
    const float2 mone2 = f2(-1.0f, -1.0f);
    float dmax = 0.0f;
#pragma unroll
    for (int w = 0; w < NP / 4; ++w) {
        uint32_t mx[4], my[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 tt = __fmul2_rn(v[4 * w + k], r2);
            const float2 m = __fadd2_rn(tt, magic);     // low mantissa byte = rint(t) mod 256
            const float2 q = __fadd2_rn(m, nmagic);     // rint(t), exact
            const float2 d = __ffma2_rn(q, mone2, tt);  // t - rint(t), exact
            dmax = fmaxf(dmax, pair_max_abs(d));
            mx[k] = __float_as_uint(m.x);
            my[k] = __float_as_uint(m.y);
        }
        words[0][w] = __byte_perm(__byte_perm(mx[0], mx[1], 0x0040), __byte_perm(mx[2], mx[3], 0x0040), 0x5410);
        words[1][w] = __byte_perm(__byte_perm(my[0], my[1], 0x0040), __byte_perm(my[2], my[3], 0x0040), 0x5410);
    }
    return dmax <= 0.4999f;
}

// The codes clamp(rne(fl(v/s)), +-127) through IEEE division.
template <int NP>
__device__ __forceinline__ void quant_codes_exact(const float2 (&v)[NP], float s, uint32_t (&words)[2][NP / 4]) {
#pragma unroll
    for (int w = 0; w < NP / 4; ++w) {
        uint32_t wx = 0, wy = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            int qx = 0, qy = 0;
            if (s != 0.0f) {
                qx = max(-127, min(127, __float2int_rn(__fdiv_rn(v[4 * w + k].x, s))));
                qy = max(-127, min(127, __float2int_rn(__fdiv_rn(v[4 * w + k].y, s))));
            }
            wx |= (uint32_t)(qx & 0xFF) << (8 * k);
            wy |= (uint32_t)(qy & 0xFF) << (8 * k);
        }
        words[0][w] = wx;
        words[1][w] = wy;
    }
}

// Quantize a thread's pairs with the row scale s (|v| <= 127 s): reciprocal
// path unless a tie is near or 1/s is not a safe finite number.
template <int NP>
__device__ __forceinline__ void quant_codes(const float2 (&v)[NP], float s, uint32_t (&words)[2][NP / 4]) {
    bool ok = false;
    if (s >= 1e-30f) ok = quant_codes_fast<NP>(v, __frcp_rn(s), words);
    if (!ok) quant_codes_exact<NP>(v, s, words);
}

// Store the codes of one output half (NW words = 4*NW values) with 16-byte stores.
template <int OUT, int NW>
__device__ __forceinline__ void store_codes(void *out, int64_t off, const uint32_t (&w)[NW]) {
    if constexpr (OUT == OUT_S8) {
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<int8_t *>(out) + off);
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {  // exact integers coded as fp16 (the tensor-core operand)
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(out) + off);
#pragma unroll
        for (int i = 0; i < NW / 2; ++i) {
            const uint32_t a = w[2 * i], b = w[2 * i + 1];
            dst[i] = make_uint4(s8pair_to_f16x2(__byte_perm(a, 0, 0x4140)), s8pair_to_f16x2(__byte_perm(a, 0, 0x4342)),
                                s8pair_to_f16x2(__byte_perm(b, 0, 0x4140)), s8pair_to_f16x2(__byte_perm(b, 0, 0x4342)));
        }
    }
}

template <int LOGN, int IN, int OUT>
__global__ void __launch_bounds__(RotqMaxThreads<LOGN>::value) rotq_kernel(RotArgs p) {
    using Geo = RotGeom<LOGN>;
    constexpr int NP = Geo::NP, TPG = Geo::TPG;
    extern __shared__ __align__(16) float2 smem2[];
    const int G = p.G;
    const int row_threads = G * TPG;
    const int tid = threadIdx.x;
    const int rloc = tid / row_threads;
    const int rem = tid - rloc * row_threads;
    const int g = rem / TPG;
    const int t = rem - g * TPG;
    const int64_t row = (int64_t)blockIdx.x * p.rows_per_cta + rloc;
    const bool active = row < p.M;
    float2 *T = smem2 + (size_t)(rloc * G + g) * Geo::TILE;
    unsigned *s_amax = reinterpret_cast<unsigned *>(smem2 + (size_t)p.rows_per_cta * G * Geo::TILE);
    if (tid < p.rows_per_cta) s_amax[tid] = 0u;

    float2 v[NP];
    rot_group_core<LOGN, IN>(p, row, active, g, t, T, v);

    if constexpr (OUT == OUT_BF16) {
        if (!active) return;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + row * p.K +
                                                   out_offset<LOGN>(g, t, h));
#pragma unroll
            for (int j8 = 0; j8 < NP / 8; ++j8) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = h ? v[8 * j8 + 2 * k].y : v[8 * j8 + 2 * k].x;
                    const float b = h ? v[8 * j8 + 2 * k + 1].y : v[8 * j8 + 2 * k + 1].x;
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(a, b);
                    w[k] = *reinterpret_cast<uint32_t *>(&b2);
                }
                dst[j8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        return;
    } else {
        // ---------------- row amax ----------------
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < NP; ++j) m = fmaxf(m, pair_max_abs(v[j]));
        constexpr int W = TPG < 32 ? TPG : 32;  // lanes of one group inside a warp
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((t & (W - 1)) == 0) atomicMax(&s_amax[rloc], __float_as_uint(m));
        __syncthreads();
        if (!active) return;
        const float amax = __uint_as_float(s_amax[rloc]);
        const float s = __fdiv_rn(amax, 127.0f);
        if (rem == 0) p.out_scale[row] = s;
        uint32_t words[2][NP / 4];
        quant_codes<NP>(v, s, words);
#pragma unroll
        for (int h = 0; h < 2; ++h) store_codes<OUT, NP / 4>(p.out, row * p.K + out_offset<LOGN>(g, t, h), words[h]);
    }
}

// Shared memory bytes for one launch of rotq_kernel.
__host__ __device__ inline size_t rotq_smem_bytes(int logn, int G, int rows_per_cta) {
    const int n = 1 << logn;
    const bool pt = logn >= 7;
    const int rows = pt ? n : n / 2, cols = pt ? n / 2 : n;
    const size_t tile = (size_t)rows * (cols + 2) + 8;
    return (size_t)rows_per_cta * G * tile * sizeof(float2) + (size_t)rows_per_cta * sizeof(unsigned) + 16;
}

}  // namespace gbq
