// rotate_g.cu -- the rotation for every descriptor: any powers of two a, b with a*b*groups = K.
//
// What it computes (PyPI page "xpu-kernels 0.2.0", sections "Algorithm: fused ConvRot rotation"
// and "API"): each group of a*b contiguous values of a row, read as X[a][b] (x[i*b + j] = X[i][j]),
// becomes V = H_a X H_b / sqrt(a*b) = ((H_a (x) H_b) / sqrt(a*b)) x in fp32, then (quantizing
// outputs) per row amax = max|v|, s = amax/127, q = clamp(rne(v/s), +-127).
//
// H_n is a Kronecker power of the printed H4, with an unnormalised H2 on the most significant index
// bit when log2 n is odd, so the transform of a group is a list of "levels", each acting on index
// bits of the group: H4/2 on two adjacent bits (a base-4 digit) or H2 on one bit; i's bits sit
// above j's (bit lb + d of the group index is bit d of i).  The H2 levels are unnormalised and
// their factor is removed once after the last level: one exact halving for two of them, one
// multiplication by fl(sqrt(1/2)) for one.
//
// Level order.  For a = b in {16, 32, 64, 128} the list is the square kernels' order
// (rotate_impl.cuh: hadamard_pass), and every level uses the same fp32 operations as they do
// (s = (x0 + x1) + (x2 + x3), out_i = s/2 - x_(3-i); H2 as (a + b, a - b)), so this kernel's
// values equal theirs bit for bit and a descriptor may be served by either.  Every other
// descriptor takes i's levels first (H4 digits from the lowest up, then H2 on i's top bit when
// log2 a is odd), then j's the same way.  All entry points use this one list per descriptor, so
// they produce identical values for it.
//
// GB300 design.  HBM-streaming, persistent CTAs of 256 threads.  A CTA takes a chunk of R whole
// rows (R*K values, about 8 K), loads it with 16-byte coalesced loads (four per thread in flight),
// converts to fp32 and writes it into a shared tile padded by one float per 32 (bank-conflict free
// for the contiguous phases, at most two-way for the strided ones).  The levels then run two at a
// time: a pass holds, per thread, the 2^(w1+w2) values that the two levels mix (register indices
// fixed at compile time, bit positions at run time), applies both and writes the values back.
// The last pass applies the H2 normalisation and folds the per-row maximum into a shared slot
// (the values of one pass item always lie in one row).  A final phase reads 16 contiguous values
// per thread, quantizes them with the per-element rule of the square kernels (quant_codes: the
// reciprocal with an IEEE-division fallback, identical to rne(fl(v/s))) and writes 16-byte stores.
#include "kernels.h"
#include "rotate_launch.cuh"

namespace gbq {
namespace {

constexpr int kGenThreads = 256;
constexpr int kGenMaxLevels = 16;
constexpr int kGenTargetElems = 8192;  // values per chunk (rows are never split)
constexpr int kGenMaxRows = 512;

struct GenArgs {
    const void *in0;
    const void *in1;
    const float *in_scale;
    const float *col_scale0;
    const float *col_scale1;
    int64_t ld_in;
    void *out;
    float *out_scale;
    int64_t M;
    int K;       // row length (a multiple of 16)
    int R;       // rows per chunk
    int nlev;    // levels in application order
    uint8_t pos[kGenMaxLevels];
    uint8_t wid[kGenMaxLevels];  // 2: H4/2 on bits pos, pos+1; 1: H2 on bit pos
    float post;                  // factor after the last level: 1, 1/2 or fl(sqrt(1/2))
    uint32_t rowmax_off;         // byte offsets in dynamic shared memory
    uint32_t rowscale_off;
    unsigned int *status;        // device status word (debug builds: bounds checks)
};

__device__ __forceinline__ int tix(int e) { return e + (e >> 5); }  // padded tile index

// ---- phase 0: eight contiguous input values (col a multiple of 8) as fp32, with the arithmetic
// of the square kernels' loaders (load_in / staged_pair).
template <int IN>
__device__ __forceinline__ void gen_load8(const GenArgs &p, int64_t grow, int col, float (&x)[8]) {
    const int64_t gi = grow * p.ld_in + col;
    if constexpr (IN == IN_BF16) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.in0) + gi));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(ws[k] << 16);
            x[2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
        }
    } else if constexpr (IN == IN_F32) {
        const float4 *src = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.in0) + gi);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else if constexpr (IN == IN_GLU_BF16) {
        const uint4 g = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.in0) + gi));
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.in1) + gi));
        const uint32_t gs[4] = {g.x, g.y, g.z, g.w}, us[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = silu_mul(__uint_as_float(gs[k] << 16), __uint_as_float(us[k] << 16));
            x[2 * k + 1] = silu_mul(__uint_as_float(gs[k] & 0xFFFF0000u), __uint_as_float(us[k] & 0xFFFF0000u));
        }
    } else if constexpr (IN == IN_S8_ROWSCALE) {
        const float rs = __ldg(p.in_scale + grow);
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const int8_t *>(p.in0) + gi));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int8_t q = (int8_t)(((k < 4 ? w.x : w.y) >> (8 * (k & 3))) & 0xFF);
            x[k] = __fmul_rn((float)q, rs);
        }
    } else if constexpr (IN == IN_ACC_ROWSCALE) {
        const float rs = __ldg(p.in_scale + grow);
        const int4 *src = reinterpret_cast<const int4 *>(reinterpret_cast<const int32_t *>(p.in0) + gi);
        const int4 a = __ldg(src), b = __ldg(src + 1);
        const int v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = __fmul_rn(__int2float_rn(v[k]), rs);
    } else {  // IN_ACC_GLU
        const float rs = __ldg(p.in_scale + grow);
        const int4 *sg = reinterpret_cast<const int4 *>(reinterpret_cast<const int32_t *>(p.in0) + gi);
        const int4 *su = reinterpret_cast<const int4 *>(reinterpret_cast<const int32_t *>(p.in1) + gi);
        const int4 g0 = __ldg(sg), g1 = __ldg(sg + 1), u0 = __ldg(su), u1 = __ldg(su + 1);
        const float4 *cg = reinterpret_cast<const float4 *>(p.col_scale0 + col);
        const float4 *cu = reinterpret_cast<const float4 *>(p.col_scale1 + col);
        const float4 cg0 = __ldg(cg), cg1 = __ldg(cg + 1), cu0 = __ldg(cu), cu1 = __ldg(cu + 1);
        const int gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const int uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float gs[8] = {cg0.x, cg0.y, cg0.z, cg0.w, cg1.x, cg1.y, cg1.z, cg1.w};
        const float us[8] = {cu0.x, cu0.y, cu0.z, cu0.w, cu1.x, cu1.y, cu1.z, cu1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k)
            x[k] = silu_mul(dequant_bf16_value(gv[k], rs, gs[k]), dequant_bf16_value(uv[k], rs, us[k]));
    }
}

// ---- one level on register bits [RB, RB + W) of a thread's values; with PB >= 0 the values are taken
// in pairs across register bit PB (outside the level's bits), so each operation runs on the packed
// fp32x2 pipe.  Per value the operations are the scalar ones.
template <int W, int RB, int NV, int PB>
__device__ __forceinline__ void gen_level(float (&v)[NV]) {
    if constexpr (W == 2) {
#pragma unroll
        for (int base = 0; base < NV; ++base) {
            if ((base >> RB) & 3) continue;
            if (PB >= 0 && ((base >> (PB < 0 ? 0 : PB)) & 1)) continue;
            const int b1 = base | (1 << RB), b2 = base | (2 << RB), b3 = base | (3 << RB);
            if constexpr (PB >= 0) {
                constexpr int o = 1 << (PB < 0 ? 0 : PB);
                const float2 x0 = make_float2(v[base], v[base | o]), x1 = make_float2(v[b1], v[b1 | o]);
                const float2 x2 = make_float2(v[b2], v[b2 | o]), x3 = make_float2(v[b3], v[b3 | o]);
                const float2 m1 = make_float2(-1.0f, -1.0f);
                const float2 h = __fmul2_rn(__fadd2_rn(__fadd2_rn(x0, x1), __fadd2_rn(x2, x3)), make_float2(0.5f, 0.5f));
                const float2 y0 = __ffma2_rn(x3, m1, h), y1 = __ffma2_rn(x2, m1, h);
                const float2 y2 = __ffma2_rn(x1, m1, h), y3 = __ffma2_rn(x0, m1, h);
                v[base] = y0.x; v[base | o] = y0.y;
                v[b1] = y1.x; v[b1 | o] = y1.y;
                v[b2] = y2.x; v[b2 | o] = y2.y;
                v[b3] = y3.x; v[b3 | o] = y3.y;
            } else {
                const float x0 = v[base], x1 = v[b1], x2 = v[b2], x3 = v[b3];
                const float h = __fmul_rn(__fadd_rn(__fadd_rn(x0, x1), __fadd_rn(x2, x3)), 0.5f);  // exact halving
                v[base] = __fmaf_rn(x3, -1.0f, h);
                v[b1] = __fmaf_rn(x2, -1.0f, h);
                v[b2] = __fmaf_rn(x1, -1.0f, h);
                v[b3] = __fmaf_rn(x0, -1.0f, h);
            }
        }
    } else if constexpr (W == 1) {
#pragma unroll
        for (int base = 0; base < NV; ++base) {
            if ((base >> RB) & 1) continue;
            if (PB >= 0 && ((base >> (PB < 0 ? 0 : PB)) & 1)) continue;
            const int b1 = base | (1 << RB);
            if constexpr (PB >= 0) {
                constexpr int o = 1 << (PB < 0 ? 0 : PB);
                const float2 a = make_float2(v[base], v[base | o]), b = make_float2(v[b1], v[b1 | o]);
                const float2 sm = __fadd2_rn(a, b), df = __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
                v[base] = sm.x; v[base | o] = sm.y;
                v[b1] = df.x; v[b1 | o] = df.y;
            } else {
                const float a = v[base], b = v[b1];
                v[base] = __fadd_rn(a, b);
                v[b1] = __fmaf_rn(b, -1.0f, a);
            }
        }
    }
}

// ---- one pass: the levels (p1, W1) and, when W2 > 0, (p2, W2), on every item of the chunk.
// An item is the 2^(W1+W2) values whose group indices differ only in those bits; items are
// enumerated by inserting zero bits at the two positions into the item number.  An item's base index
// and its offsets use disjoint bits, so the padded index is tix(base) + tix(offset): the offsets are
// computed once per pass.
template <int W1, int W2, bool LAST, int OUT>
__device__ __forceinline__ void gen_pass(float *T, int E, int p1, int p2, const GenArgs &p, unsigned int *rowmax) {
    constexpr int NV = 1 << (W1 + W2);
    const int items = E >> (W1 + W2);
    int pl = p1, wl = W1, ph = p2, wh = W2;
    if (W2 > 0 && p2 < p1) {
        pl = p2;
        wl = W2;
        ph = p1;
        wh = W1;
    }
    int toff[NV];
#pragma unroll
    for (int r = 0; r < NV; ++r) {
        const int d1 = r & ((1 << W1) - 1), d2 = r >> W1;
        toff[r] = tix(d1 << p1) + (W2 > 0 ? tix(d2 << p2) : 0);
    }
    for (int w = threadIdx.x; w < items; w += kGenThreads) {
        int base = (w & ((1 << pl) - 1)) | ((w >> pl) << (pl + wl));
        if (W2 > 0) base = (base & ((1 << ph) - 1)) | ((base >> ph) << (ph + wh));
        float *tb = T + tix(base);
        float v[NV];
#pragma unroll
        for (int r = 0; r < NV; ++r) v[r] = tb[toff[r]];
        // level 1 pairs across the top register bit (level 2's), level 2 across register bit 0
        gen_level<W1, 0, NV, (W2 > 0 ? W1 + W2 - 1 : -1)>(v);
        gen_level<W2, W1, NV, 0>(v);
        if constexpr (LAST) {
            if (p.post != 1.0f) {
#pragma unroll
                for (int r = 0; r < NV; ++r) v[r] = __fmul_rn(v[r], p.post);
            }
            if constexpr (OUT != OUT_BF16) {
                float m = 0.0f;
#pragma unroll
                for (int r = 0; r < NV; ++r) m = fmaxf(m, fabsf(v[r]));
                // One atomic per warp when the warp's items lie in one row (wide rows), else one per item.
                const int row = base / p.K;
                const unsigned act = __activemask();
                const int row0 = __shfl_sync(act, row, __ffs(act) - 1);
                if (act == 0xffffffffu && __all_sync(act, row == row0)) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if ((threadIdx.x & 31) == 0) atomicMax(&rowmax[row], __float_as_uint(m));
                } else {
                    atomicMax(&rowmax[row], __float_as_uint(m));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < NV; ++r) tb[toff[r]] = v[r];
    }
}

template <bool LAST, int OUT>
__device__ __forceinline__ void gen_pass_dispatch(int w1, int w2, float *T, int E, int p1, int p2, const GenArgs &p,
                                                  unsigned int *rowmax) {
    switch (w1 * 4 + w2) {
        case 1 * 4 + 0: gen_pass<1, 0, LAST, OUT>(T, E, p1, p2, p, rowmax); break;
        case 1 * 4 + 1: gen_pass<1, 1, LAST, OUT>(T, E, p1, p2, p, rowmax); break;
        case 1 * 4 + 2: gen_pass<1, 2, LAST, OUT>(T, E, p1, p2, p, rowmax); break;
        case 2 * 4 + 0: gen_pass<2, 0, LAST, OUT>(T, E, p1, p2, p, rowmax); break;
        case 2 * 4 + 1: gen_pass<2, 1, LAST, OUT>(T, E, p1, p2, p, rowmax); break;
        default: gen_pass<2, 2, LAST, OUT>(T, E, p1, p2, p, rowmax); break;
    }
}

// Bytes of one input element (per input tensor) and whether a second tensor (in1) is read.
template <int IN>
constexpr int gen_in_bytes() {
    return (IN == IN_BF16 || IN == IN_GLU_BF16) ? 2 : (IN == IN_S8_ROWSCALE ? 1 : 4);
}
template <int IN>
constexpr bool gen_two_inputs() {
    return IN == IN_GLU_BF16 || IN == IN_ACC_GLU;
}

// L2 prefetch hint for the input rows [r0, r0 + nr): one bulk prefetch per row and input tensor, issued
// by threads 0..nr-1 (a row is K elements, a multiple of 16 bytes, at a 16-byte aligned address).
template <int IN>
__device__ __forceinline__ void gen_prefetch_rows(const GenArgs &p, int64_t r0, int nr) {
    constexpr int EB = gen_in_bytes<IN>();
    for (int i = threadIdx.x; i < nr; i += kGenThreads) {
        const int64_t off = (r0 + i) * p.ld_in * EB;
        const uint32_t bytes = (uint32_t)p.K * EB;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<const uint8_t *>(p.in0) + off),
                     "r"(bytes)
                     : "memory");
        if constexpr (gen_two_inputs<IN>())
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<const uint8_t *>(p.in1) + off),
                         "r"(bytes)
                         : "memory");
    }
}

template <int IN, int OUT>
__global__ void __launch_bounds__(kGenThreads, 3) rotg_kernel(const __grid_constant__ GenArgs p) {
    extern __shared__ __align__(128) uint8_t smem[];
    float *T = reinterpret_cast<float *>(smem);
    unsigned int *rowmax = reinterpret_cast<unsigned int *>(smem + p.rowmax_off);
    float *rowscale = reinterpret_cast<float *>(smem + p.rowscale_off);
    pdl_allow_dependents();  // a GEMM launched after this kernel may set itself up meanwhile

    const int tid = threadIdx.x;
    const int K = p.K;
    const int64_t nchunks = (p.M + p.R - 1) / p.R;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int64_t r0 = c * p.R;
        const int nr = (int)min((int64_t)p.R, p.M - r0);
        const int E = nr * K;
        if constexpr (OUT != OUT_BF16)
            for (int i = tid; i < nr; i += kGenThreads) rowmax[i] = 0u;
        {  // the CTA's next chunk streams into L2 while this one is transformed
            const int64_t cn = c + gridDim.x;
            if (cn < nchunks) gen_prefetch_rows<IN>(p, cn * p.R, (int)min((int64_t)p.R, p.M - cn * p.R));
        }

        // ---- phase 0: global -> fp32 tile, two 8-value loads per thread in flight
        const int E8 = E >> 3;
        for (int u0 = tid; u0 < E8; u0 += 2 * kGenThreads) {
            float x[2][8];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int u = u0 + j * kGenThreads;
                if (u < E8) {
                    const int e = u * 8, row = e / K;
                    if (GBQ_IN_RANGE(p.status, r0 + row, 1, p.M) && GBQ_IN_RANGE(p.status, e - row * K, 8, K)) {
                        gen_load8<IN>(p, r0 + row, e - row * K, x[j]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) x[j][k] = 0.0f;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int u = u0 + j * kGenThreads;
                if (u < E8) {
                    float *t = T + tix(u * 8);  // eight values inside one 32-value block
#pragma unroll
                    for (int k = 0; k < 8; ++k) t[k] = x[j][k];
                }
            }
        }
        __syncthreads();

        // ---- the levels, two per pass
        for (int l = 0; l < p.nlev; l += 2) {
            const bool pair = l + 1 < p.nlev;
            const int w1 = p.wid[l], w2 = pair ? p.wid[l + 1] : 0;
            const int p1 = p.pos[l], p2 = pair ? p.pos[l + 1] : 0;
            if (l + 2 >= p.nlev)
                gen_pass_dispatch<true, OUT>(w1, w2, T, E, p1, p2, p, rowmax);
            else
                gen_pass_dispatch<false, OUT>(w1, w2, T, E, p1, p2, p, rowmax);
            __syncthreads();
        }

        if constexpr (OUT != OUT_BF16) {
            if (p.nlev == 0) {  // identity: the row maxima from 16-value blocks
                for (int u = tid; u < (E >> 4); u += kGenThreads) {
                    const float *t = T + tix(u * 16);
                    float m = 0.0f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) m = fmaxf(m, fabsf(t[k]));
                    const int row = (u * 16) / K;
                    const unsigned act = __activemask();
                    const int row0 = __shfl_sync(act, row, __ffs(act) - 1);
                    if (act == 0xffffffffu && __all_sync(act, row == row0)) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if ((threadIdx.x & 31) == 0) atomicMax(&rowmax[row], __float_as_uint(m));
                    } else {
                        atomicMax(&rowmax[row], __float_as_uint(m));
                    }
                }
                __syncthreads();
            }
            for (int i = tid; i < nr; i += kGenThreads) {
                const float s = __fdiv_rn(__uint_as_float(rowmax[i]), 127.0f);
                rowscale[i] = s;
                if (GBQ_IN_RANGE(p.status, r0 + i, 1, p.M)) p.out_scale[r0 + i] = s;
            }
            __syncthreads();
        }

        // ---- store phase: 16 contiguous values per thread
        for (int u = tid; u < (E >> 4); u += kGenThreads) {
            const int e = u * 16, row = e / K;
            const float *t = T + tix(e);
            float2 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = make_float2(t[k], t[k + 8]);
            const int64_t off = (r0 + row) * (int64_t)K + (e - row * K);
            if (!(GBQ_IN_RANGE(p.status, r0 + row, 1, p.M) && GBQ_IN_RANGE(p.status, e - row * K, 16, K))) continue;
            if constexpr (OUT == OUT_BF16) {
                uint32_t w[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(v[2 * k].x, v[2 * k + 1].x);
                    __nv_bfloat162 hi = __floats2bfloat162_rn(v[2 * k].y, v[2 * k + 1].y);
                    w[k] = *reinterpret_cast<uint32_t *>(&lo);
                    w[4 + k] = *reinterpret_cast<uint32_t *>(&hi);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) + off);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
                uint32_t words[2][2];
                quant_codes<8>(v, rowscale[row], words);
                if constexpr (OUT == OUT_S8) {
                    *reinterpret_cast<uint4 *>(reinterpret_cast<int8_t *>(p.out) + off) =
                        make_uint4(words[0][0], words[0][1], words[1][0], words[1][1]);
                } else {
                    store_codes<OUT_F16Q, 2>(p.out, off, words[0]);
                    store_codes<OUT_F16Q, 2>(p.out, off + 8, words[1]);
                }
            }
        }
        __syncthreads();  // the tile and the row slots are reused by the next chunk
    }
}

// The level list of a descriptor (see the header comment).
void gen_levels(int la, int lb, GenArgs &g) {
    g.nlev = 0;
    auto add = [&](int pos, int w) {
        g.pos[g.nlev] = (uint8_t)pos;
        g.wid[g.nlev] = (uint8_t)w;
        ++g.nlev;
    };
    const int ib = lb;  // i's bits start above j's
    if (la == lb && la >= 4 && la <= 7) {
        switch (la) {
            case 4: add(ib, 2); add(ib + 2, 2); add(0, 2); add(2, 2); break;
            case 5: add(ib, 2); add(ib + 2, 2); add(ib + 4, 1); add(0, 2); add(2, 2); add(4, 1); break;
            case 6: add(ib, 2); add(ib + 2, 2); add(ib + 4, 2); add(4, 2); add(0, 2); add(2, 2); break;
            default:
                add(ib + 6, 1); add(ib, 2); add(ib + 2, 2); add(ib + 4, 2);
                add(4, 2); add(6, 1); add(0, 2); add(2, 2);
                break;
        }
    } else {
        for (int d = 0; d + 1 < la; d += 2) add(ib + d, 2);
        if (la & 1) add(ib + la - 1, 1);
        for (int d = 0; d + 1 < lb; d += 2) add(d, 2);
        if (lb & 1) add(lb - 1, 1);
    }
    const int c2 = (la & 1) + (lb & 1);
    g.post = c2 == 2 ? 0.5f : (c2 == 1 ? 0.70710678118654752f : 1.0f);
}

template <int IN, int OUT>
cudaError_t launch_rotg_t(GenArgs g, int num_sms, cudaStream_t st) {
    static int regs = -1;  // one per instantiation
    constexpr int kMaxSmem = 227 * 1024;
    const int E = g.R * g.K;
    const uint32_t tile_bytes = (uint32_t)(((int64_t)(E + E / 32) * 4 + 127) / 128 * 128);
    g.rowmax_off = tile_bytes;
    g.rowscale_off = tile_bytes + (uint32_t)g.R * 4;
    const size_t smem = tile_bytes + (size_t)g.R * 8;
    if (smem > (size_t)kMaxSmem) return cudaErrorNotSupported;
    if (regs < 0) {
        cudaError_t e = cudaFuncSetAttribute(rotg_kernel<IN, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, rotg_kernel<IN, OUT>);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
    }
    const int per_sm = resident_ctas(regs, kGenThreads, smem);
    if (per_sm < 1) return cudaErrorNotSupported;
    const int64_t nchunks = (g.M + g.R - 1) / g.R;
    const int64_t resident = (int64_t)per_sm * (num_sms > 0 ? num_sms : 1);
    const int grid = (int)(nchunks < resident ? nchunks : resident);
    prof_begin(0, st);
    rotg_kernel<IN, OUT><<<grid, kGenThreads, smem, st>>>(g);
    prof_end(st);
    return cudaGetLastError();
}

}  // namespace

bool rotg_fits(int64_t K) { return K >= 16 && K % 16 == 0 && K <= kGenMaxK; }

cudaError_t launch_rotg(int in_kind, int out_kind, const RotArgs &a, int la, int lb, cudaStream_t st) {
    if (!rotg_fits(a.K)) return cudaErrorNotSupported;
    if (a.M == 0) return cudaSuccess;
    // 16-byte loads and stores: every row start must be 16-byte aligned.
    const uintptr_t align = (uintptr_t)a.in0 | (uintptr_t)(a.in1 ? a.in1 : a.in0) | (uintptr_t)a.out;
    if ((align & 15) != 0 || (a.ld_in * in_elem_bytes(in_kind)) % 16 != 0) return cudaErrorNotSupported;
    GenArgs g{};
    g.in0 = a.in0;
    g.in1 = a.in1;
    g.in_scale = a.in_scale;
    g.col_scale0 = a.col_scale0;
    g.col_scale1 = a.col_scale1;
    g.ld_in = a.ld_in;
    g.out = a.out;
    g.out_scale = a.out_scale;
    g.status = a.status;
    g.M = a.M;
    g.K = (int)a.K;
    int R = kGenTargetElems / g.K;
    if (R < 1) R = 1;
    if (R > kGenMaxRows) R = kGenMaxRows;
    if ((int64_t)R > a.M) R = (int)a.M;
    g.R = R;
    if (la == 0 && lb == 0) {
        g.nlev = 0;
        g.post = 1.0f;
    } else {
        gen_levels(la, lb, g);
    }
    const int sms = a.num_sms;
    if (out_kind == OUT_S8) {
        switch (in_kind) {
            case IN_BF16: return launch_rotg_t<IN_BF16, OUT_S8>(g, sms, st);
            case IN_GLU_BF16: return launch_rotg_t<IN_GLU_BF16, OUT_S8>(g, sms, st);
            case IN_ACC_GLU: return launch_rotg_t<IN_ACC_GLU, OUT_S8>(g, sms, st);
            default: return cudaErrorNotSupported;
        }
    } else if (out_kind == OUT_F16Q) {
        switch (in_kind) {
            case IN_BF16: return launch_rotg_t<IN_BF16, OUT_F16Q>(g, sms, st);
            case IN_GLU_BF16: return launch_rotg_t<IN_GLU_BF16, OUT_F16Q>(g, sms, st);
            default: return cudaErrorNotSupported;
        }
    } else {
        switch (in_kind) {
            case IN_BF16: return launch_rotg_t<IN_BF16, OUT_BF16>(g, sms, st);
            case IN_F32: return launch_rotg_t<IN_F32, OUT_BF16>(g, sms, st);
            case IN_S8_ROWSCALE: return launch_rotg_t<IN_S8_ROWSCALE, OUT_BF16>(g, sms, st);
            case IN_ACC_ROWSCALE: return launch_rotg_t<IN_ACC_ROWSCALE, OUT_BF16>(g, sms, st);
            default: return cudaErrorNotSupported;
        }
    }
}

}  // namespace gbq
