// rotate_g.cuh -- the generic rotation's building blocks (any powers of two a, b with a*b*groups = K),
// shared by rotg_kernel (rotate_g.cu) and the decode GEMV that rotates its tokens in place (gemv.cu).
//
// The group transform is a list of levels, each acting on index bits of the group: H4/2 on two adjacent
// bits (a base-4 digit) or an unnormalised H2 on one bit; i's bits sit above j's.  For a = b in
// {16, 32, 64, 128} the list is the square kernels' order, with their fp32 operations; every other
// descriptor takes i's levels first (H4 digits from the lowest up, then H2 on i's top bit when log2 a is
// odd), then j's the same way.  The H2 levels' factor is removed once after the last level.  A tile
// holds R whole rows as fp32, padded by one float per 32; a pass applies two levels to every "item"
// (the 2^(w1+w2) values the two levels mix).
#pragma once

#include "kernels.h"
#include "rotate_impl.cuh"

namespace gbq {
namespace gen {

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
    uint32_t kdiv;  // ceil(2^32 / K) (gen_set_k): the row of chunk index e is umulhi(e, kdiv)
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

// Row length and its reciprocal multiplier.  With kdiv = ceil(2^32 / K) = (2^32 + r) / K, 0 <= r < K,
// e * kdiv / 2^32 = e / K + e r / (K 2^32), whose integer part is floor(e / K) whenever e r < 2^32;
// r < K, so every chunk index e < 2^32 / K qualifies (chunks hold at most max(8192, K) values and
// K <= kGenMaxK, so e K < 2^32 always).  One multiply-high replaces an integer division.
inline void gen_set_k(GenArgs &g, int K) {
    g.K = K;
    g.kdiv = (uint32_t)((((uint64_t)1 << 32) + (uint64_t)K - 1) / (uint64_t)K);
}
__device__ __forceinline__ int gen_row(const GenArgs &p, int e) { return (int)__umulhi((unsigned)e, p.kdiv); }

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
                const int row = gen_row(p, base);
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

// The level list of a descriptor (see the order above).
inline void gen_levels(int la, int lb, GenArgs &g) {
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

}  // namespace gen
}  // namespace gbq
