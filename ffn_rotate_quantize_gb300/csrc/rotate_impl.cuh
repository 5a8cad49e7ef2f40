// rotate_impl.cuh -- fused Kronecker-Hadamard rotation (+ per-row INT8 quantize).
//
// What it computes (PyPI page "xpu-kernels 0.2.0", sections "Algorithm: fused
// ConvRot rotation" and "API"): for each row x of length K = G*n*n, each of the
// G contiguous groups X[n][n] (x[i*n+j] = X[i][j]) becomes
//     V = (H_n X H_n) / n        (= (H_n (x) H_n) x / sqrt(n*n), H_n symmetric)
// in fp32; then, per row, amax = max|v|, s = amax/127, q = clamp(rne(v/s), +-127).
//
// GB300 design.  The kernel is persistent and HBM-streaming: each CTA holds a
// few "teams" (one warp, or the threads of one row when a row needs more), and
// each team loops over rows.  Its leader thread bulk-copies (cp.async.bulk) the
// input rows into a double-buffered shared-memory stage two rows ahead, so the
// HBM stream never waits for arithmetic, and the team writes each finished row
// back with one bulk store from shared memory.  The rotation itself: one group
// is owned by TPG threads and every value is carried in a float2 pair so that
// each Hadamard level runs on the packed fp32x2 pipe:
//   n <= 64  pass 1: thread t holds columns 2t, 2t+1 (pair = the two columns);
//            pass 2: thread t holds rows t, t+n/2     (pair = the two rows);
//   n == 128 pass 1: thread t holds column t, pair = (row i, row i+64);
//            pass 2: thread t holds row t,    pair = (col j, col j+64).
// Pass 1 applies H_n down the columns (reading the staged input), a padded
// shared tile of float2 pairs turns columns into rows (16-byte accesses,
// conflict-free), pass 2 applies H_n along the rows; the tile then holds the
// row's output for the bulk store.  Levels run in a fixed order (H4/2 on base-4
// digits from the low bit up, then the unnormalised H2 on the top bit when
// log2 n is odd, whose two sqrt(2) factors are removed by one final exact
// halving), so every kernel that uses this core produces bit-identical values.
// Quantize: r = 1/s once per row; t = v*r; the code is rint(t) (read out of the
// low byte of t + 1.5*2^23), which equals rne(fl(v/s)) unless t lies within
// 1e-4 of a half-integer (|t - v/s| <= 128*2^-23 and |fl(v/s) - v/s| <= 2^-18
// bound the difference far below that); such threads, and rows with a scale
// too small for a finite reciprocal, are recomputed with IEEE division.
#pragma once

#include "common.cuh"

namespace gbq {

// IN_ACC_ROWSCALE: int32 accumulators times a row scale, fl(fp32(acc) * in_scale[row]) (the dx route's
// rotated gradient, with the same operation as the GEMM's row-scale epilogue).
enum InKind { IN_BF16 = 0, IN_F32 = 1, IN_GLU_BF16 = 2, IN_S8_ROWSCALE = 3, IN_ACC_GLU = 4, IN_ACC_ROWSCALE = 5 };
enum OutKind { OUT_S8 = 0, OUT_F16Q = 1, OUT_BF16 = 2 };

struct RotArgs {
    const void *in0;          // x / g / W8 / acc_g
    const void *in1;          // u / acc_u (GLU inputs), else unused
    const float *in_scale;    // IN_S8_ROWSCALE: s[row]; IN_ACC_GLU: x_scale[row]; IN_ACC_ROWSCALE: t[row]
    const float *col_scale0;  // IN_ACC_GLU: s_gate[col]
    const float *col_scale1;  // IN_ACC_GLU: s_up[col]
    int64_t ld_in;            // elements between consecutive input rows
    void *out;                // int8 / f16-coded int / bf16, row stride K
    float *out_scale;         // per-row scale (quantizing outputs)
    int32_t *out_l1;          // optional [M][K/1024]: sum of |code| over each 1024-long block of a row
                              // (quantizing outputs of the three-pass kernels)
    int64_t M, K;
    int G;                    // groups per row
    unsigned int *status;     // device status word (bounded-wait timeouts)
    int num_sms;
    // Set by the launcher (launch_rotq_t):
    int team_threads;         // threads of one team (a multiple of 32)
    int rows_per_team;        // rows a team rotates at once (several only when a row needs < 32 threads)
    int stages;               // input stages per team (1 or 2)
    uint32_t row_in_bytes;    // bytes of one input row (one of the two GLU inputs)
    uint32_t stage_bytes;     // one stage: rows_per_team x inputs x row_in_bytes (rounded to 128)
    uint32_t tiles_bytes;     // the transpose tiles of one team (rounded to 128)
    uint32_t team_bytes;      // stages + tiles + barriers / scratch
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

// SiLU(g) * u in fp32: g / (1 + exp(-g)) * u with CUDA's accurate expf (a few ulp at most from the
// correctly rounded exponential; not the special-function unit's __expf) and the division through the
// reciprocal (__fdividef, within 2 ulp of the IEEE quotient), so a code can move only where the value sits
// at a rounding boundary.  For g < -88 the exponential overflows to inf and the quotient is -0 (as g e^g).
__device__ __forceinline__ float silu_mul(float g, float u) {
    const float e = expf(-g);
    const float d = __fadd_rn(1.0f, e);
    return __fmul_rn(__fdividef(g, d), u);
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

// Unnormalised H2 across the two halves of every pair: (x, y) -> (x + y, x - y).
template <int NP>
__device__ __forceinline__ void h2_pairs(float2 (&v)[NP]) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const float a = v[i].x, b = v[i].y;
        v[i] = f2(__fadd_rn(a, b), __fsub_rn(a, b));
    }
}

// H_n for the pass layout of RotGeom<LOGN>, in the fixed level order every
// rotation kernel of the library shares (so their rotated values agree bit for
// bit).  COLS selects the first pass (H_n down the columns, index i) or the
// second (along the rows, index j):
//   n = 16, 32 : digits (0,1), (2,3), then H2 on bit 4 for n = 32, both passes;
//   n = 64     : columns (0,1), (2,3), (4,5); rows (4,5), (0,1), (2,3);
//   n = 128    : columns H2 on bit 6, then (0,1), (2,3), (4,5);
//                rows (4,5), H2 on bit 6, (0,1), (2,3).
// (For n = 128 the pair holds bit 6, so its H2 combines the two halves.)
template <int LOGN, bool COLS>
__device__ __forceinline__ void hadamard_pass(float2 (&v)[RotGeom<LOGN>::NP]) {
    constexpr int NP = RotGeom<LOGN>::NP;
    if constexpr (LOGN == 7) {
        if constexpr (COLS) {
            h2_pairs<NP>(v);
            h4_level<NP, 0>(v);
            h4_level<NP, 2>(v);
            h4_level<NP, 4>(v);
        } else {
            h4_level<NP, 4>(v);
            h2_pairs<NP>(v);
            h4_level<NP, 0>(v);
            h4_level<NP, 2>(v);
        }
    } else if constexpr (LOGN == 6) {
        if constexpr (COLS) {
            h4_level<NP, 0>(v);
            h4_level<NP, 2>(v);
            h4_level<NP, 4>(v);
        } else {
            h4_level<NP, 4>(v);
            h4_level<NP, 0>(v);
            h4_level<NP, 2>(v);
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
    } else if constexpr (IN == IN_ACC_ROWSCALE) {
        return __fmul_rn(__int2float_rn(__ldg(reinterpret_cast<const int32_t *>(p.in0) + idx)), __ldg(p.in_scale + row));
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

// Pass-1 tile write: after H_n down the columns (c), write the column pairs of
// this thread into the transpose tile T of its group.
template <int LOGN>
__device__ __forceinline__ void pass1_store_tile(const float2 (&c)[RotGeom<LOGN>::NP], int t, float2 *T) {
    using Geo = RotGeom<LOGN>;
    constexpr int N = Geo::N, NP = Geo::NP, PP = Geo::PP;
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
            *reinterpret_cast<float4 *>(&T[i * PP + 2 * t]) = make_float4(c[i].x, c[i + N / 2].x, c[i].y, c[i + N / 2].y);
    }
}

// Pass 2: read this thread's row pairs from the tile and apply H_n along the rows
// (then the exact halving that normalises the two H2 levels of an odd log2 n).
template <int LOGN>
__device__ __forceinline__ void pass2_from_tile(bool active, int t, const float2 *T, float2 (&v)[RotGeom<LOGN>::NP]) {
    using Geo = RotGeom<LOGN>;
    constexpr int NP = Geo::NP, PP = Geo::PP;
#pragma unroll
    for (int j2 = 0; j2 < NP / 2; ++j2) {
        const float4 f =
            active ? *reinterpret_cast<const float4 *>(&T[t * PP + 2 * j2]) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[2 * j2] = f2(f.x, f.y);
        v[2 * j2 + 1] = f2(f.z, f.w);
    }
    hadamard_pass<LOGN, false>(v);
    if (LOGN & 1) {
        const float2 half2 = f2(0.5f, 0.5f);
#pragma unroll
        for (int j = 0; j < NP; ++j) v[j] = __fmul2_rn(v[j], half2);  // the two H2 levels: (1/sqrt2)^2
    }
}

// The rotation of one group reading its input straight from global memory (the
// decode kernel's x): pass 1, transpose through T, pass 2; leaves this thread's
// pass-2 pairs in v.  Every thread of the CTA must call it (it contains one
// __syncthreads()).  Inactive threads touch neither global memory nor the tile
// and return zeros.
template <int LOGN, int IN>
__device__ __forceinline__ void rot_group_core(const RotArgs &p, int64_t row, bool active, int g, int t, float2 *T,
                                               float2 (&v)[RotGeom<LOGN>::NP]) {
    using Geo = RotGeom<LOGN>;
    constexpr int N = Geo::N, NP = Geo::NP;
    float2 c[NP];
    const int64_t goff = (int64_t)g * N * N;
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
    hadamard_pass<LOGN, true>(c);
    if (active) pass1_store_tile<LOGN>(c, t, T);
    __syncthreads();
    pass2_from_tile<LOGN>(active, t, T, v);
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
// holds elements 4w..4w+3 of half h.  Returns a bit mask of the words in which
// some t = v*r lies within 1e-4 of a half-integer, where the code might differ
// from rne(fl(v/s)).
template <int NP>
__device__ __forceinline__ uint32_t quant_codes_fast(const float2 (&v)[NP], float r, uint32_t (&words)[2][NP / 4]) {
    const float2 r2 = f2(r, r);
    const float2 magic = f2(12582912.0f, 12582912.0f);  // 1.5 * 2^23: t + magic rounds t to an integer (RNE)
    const float2 nmagic = f2(-12582912.0f, -12582912.0f);
    const float2 mone2 = f2(-1.0f, -1.0f);
    uint32_t bad = 0;
#pragma unroll
    for (int w = 0; w < NP / 4; ++w) {
        uint32_t mx[4], my[4];
        float dmax = 0.0f;
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
        if (dmax > 0.4999f) bad |= 1u << w;
        words[0][w] = __byte_perm(__byte_perm(mx[0], mx[1], 0x0040), __byte_perm(mx[2], mx[3], 0x0040), 0x5410);
        words[1][w] = __byte_perm(__byte_perm(my[0], my[1], 0x0040), __byte_perm(my[2], my[3], 0x0040), 0x5410);
    }
    return bad;
}

// The codes of word w (elements 4w..4w+3 of both halves): clamp(rne(fl(v/s)), +-127) through IEEE division.
template <int NP>
__device__ __forceinline__ void quant_word_exact(const float2 (&v)[NP], int w, float s, uint32_t &wx, uint32_t &wy) {
    wx = 0;
    wy = 0;
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
}

// Quantize a thread's pairs with the row scale s (|v| <= 127 s): the reciprocal
// path, then IEEE division for the words it flagged (or for all of them when
// 1/s is not a safe finite number).
template <int NP>
__device__ __forceinline__ void quant_codes(const float2 (&v)[NP], float s, uint32_t (&words)[2][NP / 4]) {
    uint32_t bad = (NP / 4 >= 32) ? 0xFFFFFFFFu : ((1u << (NP / 4)) - 1u);
    if (s >= 1e-30f) bad = quant_codes_fast<NP>(v, __frcp_rn(s), words);
    if (bad) {
#pragma unroll
        for (int w = 0; w < NP / 4; ++w)
            if (bad & (1u << w)) quant_word_exact<NP>(v, w, s, words[0][w], words[1][w]);
    }
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

// ---------------------------------------------------------------- staged input
// Number of input tensors and bytes per input element of an input kind.
__host__ __device__ constexpr int in_count(int in_kind) { return (in_kind == IN_GLU_BF16 || in_kind == IN_ACC_GLU) ? 2 : 1; }
__host__ __device__ constexpr int in_elem_bytes(int in_kind) {
    return in_kind == IN_S8_ROWSCALE ? 1 : (in_kind == IN_F32 || in_kind == IN_ACC_GLU || in_kind == IN_ACC_ROWSCALE) ? 4 : 2;
}
__host__ __device__ constexpr int out_elem_bytes(int out_kind) { return out_kind == OUT_S8 ? 1 : 2; }

// Elements idx, idx + 1 (idx even, index within the row) of a staged row as an
// fp32 pair, with the same arithmetic as load_in2.  s0 / s1: the row's staged
// input(s); rs: the row's scale (IN_S8_ROWSCALE: s[row]; IN_ACC_GLU: x_scale[row]; IN_ACC_ROWSCALE: t[row]).
template <int IN>
__device__ __forceinline__ float2 staged_pair(const RotArgs &p, const uint8_t *s0, const uint8_t *s1, float rs,
                                              int idx) {
    if constexpr (IN == IN_BF16) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(s0 + 2 * idx);
        return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    } else if constexpr (IN == IN_F32) {
        return *reinterpret_cast<const float2 *>(s0 + 4 * idx);
    } else if constexpr (IN == IN_GLU_BF16) {
        const uint32_t wg = *reinterpret_cast<const uint32_t *>(s0 + 2 * idx);
        const uint32_t wu = *reinterpret_cast<const uint32_t *>(s1 + 2 * idx);
        return f2(silu_mul(__uint_as_float(wg << 16), __uint_as_float(wu << 16)),
                  silu_mul(__uint_as_float(wg & 0xFFFF0000u), __uint_as_float(wu & 0xFFFF0000u)));
    } else if constexpr (IN == IN_S8_ROWSCALE) {
        const char2 q = *reinterpret_cast<const char2 *>(s0 + idx);
        return __fmul2_rn(f2((float)q.x, (float)q.y), f2(rs, rs));
    } else if constexpr (IN == IN_ACC_ROWSCALE) {
        const int2 a = *reinterpret_cast<const int2 *>(s0 + 4 * idx);
        return f2(__fmul_rn(__int2float_rn(a.x), rs), __fmul_rn(__int2float_rn(a.y), rs));
    } else {  // IN_ACC_GLU
        const int2 ag = *reinterpret_cast<const int2 *>(s0 + 4 * idx);
        const int2 au = *reinterpret_cast<const int2 *>(s1 + 4 * idx);
        const float2 sg = __ldg(reinterpret_cast<const float2 *>(p.col_scale0 + idx));
        const float2 su = __ldg(reinterpret_cast<const float2 *>(p.col_scale1 + idx));
        return f2(silu_mul(dequant_bf16_value(ag.x, rs, sg.x), dequant_bf16_value(au.x, rs, su.x)),
                  silu_mul(dequant_bf16_value(ag.y, rs, sg.y), dequant_bf16_value(au.y, rs, su.y)));
    }
}

// One element of a staged row (the same arithmetic as load_in).
template <int IN>
__device__ __forceinline__ float staged_one(const RotArgs &p, const uint8_t *s0, const uint8_t *s1, float rs, int idx) {
    if constexpr (IN == IN_BF16) {
        return bf16_to_float(*reinterpret_cast<const uint16_t *>(s0 + 2 * idx));
    } else if constexpr (IN == IN_F32) {
        return *reinterpret_cast<const float *>(s0 + 4 * idx);
    } else if constexpr (IN == IN_GLU_BF16) {
        return silu_mul(bf16_to_float(*reinterpret_cast<const uint16_t *>(s0 + 2 * idx)),
                        bf16_to_float(*reinterpret_cast<const uint16_t *>(s1 + 2 * idx)));
    } else if constexpr (IN == IN_S8_ROWSCALE) {
        return __fmul_rn((float)*reinterpret_cast<const int8_t *>(s0 + idx), rs);
    } else if constexpr (IN == IN_ACC_ROWSCALE) {
        return __fmul_rn(__int2float_rn(*reinterpret_cast<const int32_t *>(s0 + 4 * idx)), rs);
    } else {
        const int32_t ag = *reinterpret_cast<const int32_t *>(s0 + 4 * idx);
        const int32_t au = *reinterpret_cast<const int32_t *>(s1 + 4 * idx);
        return silu_mul(dequant_bf16_value(ag, rs, __ldg(p.col_scale0 + idx)),
                        dequant_bf16_value(au, rs, __ldg(p.col_scale1 + idx)));
    }
}

// Pass-1 values of thread t of group g from a staged row.
template <int LOGN, int IN>
__device__ __forceinline__ void staged_columns(const RotArgs &p, const uint8_t *s0, const uint8_t *s1, float rs, int g,
                                               int t, float2 (&c)[RotGeom<LOGN>::NP]) {
    using Geo = RotGeom<LOGN>;
    constexpr int N = Geo::N, NP = Geo::NP;
    const int goff = g * N * N;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        if constexpr (Geo::PAIR_TOP)  // column t, rows i and i + N/2
            c[i] = f2(staged_one<IN>(p, s0, s1, rs, goff + i * N + t),
                      staged_one<IN>(p, s0, s1, rs, goff + (i + N / 2) * N + t));
        else  // columns 2t, 2t+1 of row i
            c[i] = staged_pair<IN>(p, s0, s1, rs, goff + i * N + 2 * t);
    }
}

// ---------------------------------------------------------------- the kernel
// Team-wide barrier: one warp, or a named barrier (id 1 + team) over the team.
__device__ __forceinline__ void team_sync(int team, int team_threads) {
    if (team_threads == 32)
        __syncwarp();
    else
        named_bar_sync(1 + team, team_threads);
}
__device__ __forceinline__ bool team_all(int team, int team_threads, bool pred) {
    if (team_threads == 32) return __all_sync(0xffffffffu, pred);
    return named_bar_and(1 + team, team_threads, pred);
}

// Shared memory of one team: [stages][tiles][misc].  misc: full barriers (one
// per stage), an abort flag, and one amax slot per warp of the team.
constexpr uint32_t kRotMiscBytes = 256;

template <int LOGN, int IN, int OUT>
__global__ void __launch_bounds__(RotqMaxThreads<LOGN>::value) rotq_kernel(const __grid_constant__ RotArgs p) {
    using Geo = RotGeom<LOGN>;
    constexpr int NP = Geo::NP, TPG = Geo::TPG;
    constexpr int NIN = in_count(IN);
    constexpr uint32_t OESZ = out_elem_bytes(OUT);
    extern __shared__ __align__(128) uint8_t smem[];

    const int team = threadIdx.x / p.team_threads;
    const int tt = threadIdx.x - team * p.team_threads;  // thread within the team
    const int rt = p.G * TPG;                            // threads of one row
    const int slot = tt / rt;                            // row slot within the team
    const int rem = tt - slot * rt;
    const int g = rem / TPG;
    const int t = rem - g * TPG;
    const bool used = slot < p.rows_per_team;
    const bool leader = tt == 0;
    const int rpt = p.rows_per_team;

    uint8_t *tb = smem + (size_t)team * p.team_bytes;
    uint8_t *stage0 = tb;
    float2 *tiles = reinterpret_cast<float2 *>(tb + (size_t)p.stages * p.stage_bytes);
    uint8_t *misc = tb + (size_t)p.stages * p.stage_bytes + p.tiles_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    volatile int *abort = reinterpret_cast<volatile int *>(misc + 16);
    float *wmax = reinterpret_cast<float *>(misc + 32);  // one per warp of the team (<= 32)

    float2 *T = tiles + (size_t)((used ? slot : 0) * p.G + g) * Geo::TILE;
    uint8_t *ostage = reinterpret_cast<uint8_t *>(tiles + (size_t)(used ? slot : 0) * p.G * Geo::TILE);

    const int64_t nunits = (p.M + rpt - 1) / rpt;
    const int64_t u0 = (int64_t)blockIdx.x * (blockDim.x / p.team_threads) + team;
    const int64_t ustride = (int64_t)gridDim.x * (blockDim.x / p.team_threads);
    const uint32_t in_row_bytes = p.row_in_bytes;

    // Leader: copy the inputs of row unit u into stage st.
    auto issue = [&](int64_t u, int st) {
        const int64_t r0 = u * rpt;
        const int nr = (int)min((int64_t)rpt, p.M - r0);
        uint8_t *dst = stage0 + (size_t)st * p.stage_bytes;
        const int64_t eb = in_elem_bytes(IN);
        if (!GBQ_IN_RANGE(p.status, r0 * p.ld_in * eb, (int64_t)(nr - 1) * p.ld_in * eb + in_row_bytes,
                          p.M * p.ld_in * eb)) {
            mbar_arrive_expect_tx(&full[st], 0);  // debug builds: the copies are skipped, the stage completes empty
            return;
        }
        mbar_arrive_expect_tx(&full[st], (uint32_t)nr * NIN * in_row_bytes);
        for (int r = 0; r < nr; ++r) {
            const int64_t off = (r0 + r) * p.ld_in * in_elem_bytes(IN);
            bulk_g2s(dst + (size_t)(r * NIN) * in_row_bytes, reinterpret_cast<const uint8_t *>(p.in0) + off,
                     in_row_bytes, &full[st]);
            if (NIN == 2)
                bulk_g2s(dst + (size_t)(r * NIN + 1) * in_row_bytes, reinterpret_cast<const uint8_t *>(p.in1) + off,
                         in_row_bytes, &full[st]);
        }
    };

    if (leader) {
        for (int s2 = 0; s2 < p.stages; ++s2) mbar_init(&full[s2], 1);
        *abort = 0;
        fence_mbar_init();
    }
    team_sync(team, p.team_threads);
    // Iteration whose input was last issued into stage 0 / 1 (-1: none); team-uniform.
    int64_t issued0 = -1, issued1 = -1;
    for (int s2 = 0; s2 < p.stages; ++s2)
        if (u0 + s2 * ustride < nunits) {
            if (leader) issue(u0 + s2 * ustride, s2);
            if (s2 == 0) issued0 = 0; else issued1 = 1;
        }

    int64_t it = 0;
    bool failed = false;
    for (int64_t u = u0; u < nunits; u += ustride, ++it) {
        const int st = (int)(it % p.stages);
        uint8_t *sbuf = stage0 + (size_t)st * p.stage_bytes;
        {
            bool ok = mbar_wait(&full[st], (uint32_t)((it / p.stages) & 1), p.status, abort);
            if (!team_all(team, p.team_threads, ok)) {
                failed = true;
                break;
            }
        }
        const int64_t row = u * rpt + slot;
        const bool active = used && row < p.M;

        // ---- pass 1 from the stage ----
        float2 c[NP];
        if (active) {
            const uint8_t *s0 = sbuf + (size_t)(slot * NIN) * in_row_bytes;
            float rs = 0.0f;
            if (IN == IN_S8_ROWSCALE || IN == IN_ACC_GLU || IN == IN_ACC_ROWSCALE) rs = __ldg(p.in_scale + row);
            staged_columns<LOGN, IN>(p, s0, s0 + in_row_bytes, rs, g, t, c);
        } else {
#pragma unroll
            for (int i = 0; i < NP; ++i) c[i] = f2(0.f, 0.f);
        }
        hadamard_pass<LOGN, true>(c);
        // The tile doubles as the previous row's output staging: its bulk store must have read it.
        if (leader && it > 0) tma_store_wait_read<0>();
        team_sync(team, p.team_threads);
        if (active) pass1_store_tile<LOGN>(c, t, T);
        team_sync(team, p.team_threads);
        // Every thread has read the stage: refill it with the unit `stages` iterations ahead.
        if (u + p.stages * ustride < nunits) {
            if (leader) issue(u + p.stages * ustride, st);
            if (st == 0) issued0 = it + p.stages; else issued1 = it + p.stages;
        }

        // ---- pass 2 ----
        float2 v[NP];
        pass2_from_tile<LOGN>(active, t, T, v);

        if constexpr (OUT == OUT_BF16) {
            team_sync(team, p.team_threads);  // every pass-2 read of the tiles is done
            if (active) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint4 *dst = reinterpret_cast<uint4 *>(ostage + out_offset<LOGN>(g, t, h) * 2);
#pragma unroll
                    for (int j8 = 0; j8 < NP / 8; ++j8) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float a0 = h ? v[8 * j8 + 2 * k].y : v[8 * j8 + 2 * k].x;
                            const float a1 = h ? v[8 * j8 + 2 * k + 1].y : v[8 * j8 + 2 * k + 1].x;
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
                            w[k] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        dst[j8] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        } else {
            // ---- row amax -> scale -> codes ----
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < NP; ++j) m = fmaxf(m, pair_max_abs(v[j]));
            float amax;
            if (32 % rt == 0) {  // a row is rt consecutive lanes of one warp
                for (int o = rt / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                amax = m;
                team_sync(team, p.team_threads);  // every pass-2 read of the tiles is done
            } else {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if ((tt & 31) == 0) wmax[tt >> 5] = m;
                team_sync(team, p.team_threads);  // also: every pass-2 read of the tiles is done
                amax = wmax[0];
                for (int w = 1; w < p.team_threads / 32; ++w) amax = fmaxf(amax, wmax[w]);
            }
            const float s = __fdiv_rn(amax, 127.0f);
            if (active && rem == 0) p.out_scale[row] = s;
            if (active) {
                uint32_t words[2][NP / 4];
                quant_codes<NP>(v, s, words);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    store_codes<OUT, NP / 4>(ostage, out_offset<LOGN>(g, t, h), words[h]);
            }
        }
        fence_proxy_async_smem();
        team_sync(team, p.team_threads);
        if (leader) {
            const int64_t r0 = u * rpt;
            const int nr = (int)min((int64_t)rpt, p.M - r0);
            const uint32_t ob = (uint32_t)(p.K * OESZ);
            for (int r = 0; r < nr; ++r)
                if (GBQ_IN_RANGE(p.status, (r0 + r) * (int64_t)ob, ob, p.M * (int64_t)ob))
                bulk_s2g(reinterpret_cast<uint8_t *>(p.out) + (r0 + r) * (int64_t)ob,
                         reinterpret_cast<const uint8_t *>(tiles) + (size_t)r * p.G * Geo::TILE * sizeof(float2), ob);
            tma_store_commit();
        }
        // The amax slots are rewritten next row only after two more team barriers.
    }
    if (leader) {
        tma_store_wait_all<0>();  // stores complete before the team's shared memory goes away
        if (failed) {
            // A wait gave up at iteration `it`: let every copy still in flight land (bounded) before leaving.
            for (int s2 = 0; s2 < p.stages; ++s2) {
                const int64_t is = s2 == 0 ? issued0 : issued1;
                if (is < it) continue;
                const uint32_t par = (uint32_t)((is / p.stages) & 1);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&full[s2], par) && globaltimer() - t0 < kWaitLimitNs) {
                }
            }
        }
    }
}

}  // namespace gbq
