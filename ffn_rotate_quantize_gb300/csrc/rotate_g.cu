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
#include "rotate_g.cuh"
#include "rotate_launch.cuh"

namespace gbq {
namespace {

using namespace gen;

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
                    const int e = u * 8, row = gen_row(p, e);
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
                    const int row = gen_row(p, u * 16);
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
            const int e = u * 16, row = gen_row(p, e);
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
    gen_set_k(g, (int)a.K);
    int R = kGenTargetElems / g.K;
    if (R < 1) R = 1;
    if (R > kGenMaxRows) R = kGenMaxRows;
    if ((int64_t)R > a.M) R = (int)a.M;
    g.R = R;
    if ((uint64_t)R * (uint64_t)g.K * (uint64_t)g.K >= ((uint64_t)1 << 32)) return cudaErrorNotSupported;  // gen_row
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
