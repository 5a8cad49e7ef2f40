// rotate_b.cu -- rotate-only instantiations (bf16 output) and the identity quantizer.
#include "rotate_launch.cuh"

namespace gbq {

cudaError_t launch_rotb(int logn, int in_kind, RotArgs a, cudaStream_t st) {
    switch (in_kind) {
        case IN_BF16: return launch_rotq_logn<IN_BF16, OUT_BF16>(logn, a, st);
        case IN_F32: return launch_rotq_logn<IN_F32, OUT_BF16>(logn, a, st);
        case IN_S8_ROWSCALE: return launch_rotq_logn<IN_S8_ROWSCALE, OUT_BF16>(logn, a, st);
        case IN_ACC_ROWSCALE: return launch_rotq_logn<IN_ACC_ROWSCALE, OUT_BF16>(logn, a, st);
        default: return cudaErrorNotSupported;
    }
}

// ---------------------------------------------------------------------------
// Per-row quantizer with R = I (the dy side of linear_dx_int8, and identity
// rotation descriptors).  One CTA of 256 threads per row; each thread keeps its
// (up to 16) chunks of 8 values in registers across load -> amax -> quantize.
// Long rows (>= 16384 values) take 512 threads, so each thread holds at most 32
// values and four CTAs fit an SM: enough loads in flight to stream from HBM.
// Optional fp32 column scale: v = bf16(dy[m,n]) * s[n] in fp32 (the weight scale
// moved onto the contraction index, "The backward: dL/dx, weight-only").
// ---------------------------------------------------------------------------
constexpr int kIdChunkCap = 8;  // K <= 512 * 8 * 8 = 32768

template <int OUT, int kIdMaxChunks, int kIdThreads>
__global__ void __launch_bounds__(kIdThreads) quant_identity_kernel(IdArgs p) {
    __shared__ float s_warp[kIdThreads / 32];
    __shared__ int s_l1[32];  // per 1024-long block: sum of |code| (K <= 32768)
    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_allow_dependents();  // a GEMM launched after this kernel may set itself up meanwhile
    const int nchunks = (int)(p.K / 8);
    const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.in) + row * p.ld_in);
    float v[kIdMaxChunks][8];
    float m = 0.0f;
#pragma unroll
    for (int c = 0; c < kIdMaxChunks; ++c) {
        const int ch = tid + c * kIdThreads;
        if (ch < nchunks) {
            const uint4 w = __ldg(src + ch);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[c][2 * h] = __uint_as_float(ws[h] << 16);
                v[c][2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
            }
            if (p.col_scale) {
                const float4 c0 = __ldg(reinterpret_cast<const float4 *>(p.col_scale + 8 * ch));
                const float4 c1 = __ldg(reinterpret_cast<const float4 *>(p.col_scale + 8 * ch + 4));
                const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) v[c][e] = __fmul_rn(v[c][e], cs[e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[c][e]));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[c][e] = 0.0f;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) s_warp[tid >> 5] = m;
    __syncthreads();
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kIdThreads / 32; ++w) amax = fmaxf(amax, s_warp[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) p.out_scale[row] = s;
    // Codes rne(fl(v/s)): the reciprocal path (see rotate_impl.cuh), then IEEE division for
    // the chunks whose products lie within 1e-4 of a half-integer (or all, for a tiny scale).
    uint32_t words[kIdMaxChunks][2];
    uint32_t bad = 0xFFFFFFFFu;
    if (s >= 1e-30f) {
        bad = 0;
        const float r = __frcp_rn(s);
#pragma unroll
        for (int c = 0; c < kIdMaxChunks; ++c) {
            uint32_t mb[8];
            float dmax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float t = __fmul_rn(v[c][e], r);
                const float m = __fadd_rn(t, 12582912.0f);
                dmax = fmaxf(dmax, fabsf(__fsub_rn(t, __fsub_rn(m, 12582912.0f))));
                mb[e] = __float_as_uint(m);
            }
            if (dmax > 0.4999f) bad |= 1u << c;
            words[c][0] = __byte_perm(__byte_perm(mb[0], mb[1], 0x0040), __byte_perm(mb[2], mb[3], 0x0040), 0x5410);
            words[c][1] = __byte_perm(__byte_perm(mb[4], mb[5], 0x0040), __byte_perm(mb[6], mb[7], 0x0040), 0x5410);
        }
    }
    if (bad) {
#pragma unroll
        for (int c = 0; c < kIdMaxChunks; ++c) {
            if (!(bad & (1u << c))) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int qq = 0;
                    if (s != 0.0f) qq = max(-127, min(127, __float2int_rn(__fdiv_rn(v[c][4 * h + e], s))));
                    w |= (uint32_t)(qq & 0xFF) << (8 * e);
                }
                words[c][h] = w;
            }
        }
    }
    if (p.out_l1) {  // uniform over the CTA
        // Chunk ch lies in block ch / 128; a warp's 32 chunks of one c share a block (threads come in
        // groups of 128), so one warp sum per c goes into the block's shared counter.
        const int nb = (int)((p.K + 1023) / 1024);
        if (tid < 32) s_l1[tid] = 0;
        __syncthreads();
#pragma unroll
        for (int c = 0; c < kIdMaxChunks; ++c) {
            int l = __dp4a((int)__vabsss4(words[c][0]), 0x01010101, __dp4a((int)__vabsss4(words[c][1]), 0x01010101, 0));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            const int b = (tid + c * kIdThreads) >> 7;
            if ((tid & 31) == 0 && b < nb && l) atomicAdd(&s_l1[b], l);
        }
        __syncthreads();
        if (tid < nb) p.out_l1[row * nb + tid] = s_l1[tid];
    }
#pragma unroll
    for (int c = 0; c < kIdMaxChunks; ++c) {
        const int ch = tid + c * kIdThreads;
        if (ch >= nchunks) continue;
        if constexpr (OUT == OUT_S8) {
            reinterpret_cast<uint2 *>(reinterpret_cast<int8_t *>(p.out) + row * p.K)[ch] =
                make_uint2(words[c][0], words[c][1]);
        } else {
            const uint32_t a = words[c][0], b = words[c][1];
            reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(p.out) + row * p.K)[ch] =
                make_uint4(s8pair_to_f16x2(__byte_perm(a, 0, 0x4140)), s8pair_to_f16x2(__byte_perm(a, 0, 0x4342)),
                           s8pair_to_f16x2(__byte_perm(b, 0, 0x4140)), s8pair_to_f16x2(__byte_perm(b, 0, 0x4342)));
        }
    }
}

cudaError_t launch_quant_identity(int out_kind, IdArgs a, cudaStream_t st) {
    const int threads = (a.K / 8 >= 2048) ? 512 : 256;
    if (a.K % 8 != 0 || a.K / 8 > (int64_t)threads * kIdChunkCap) return cudaErrorNotSupported;
    if (a.M > 0x7fffffff) return cudaErrorInvalidValue;
    if (out_kind != OUT_S8 && out_kind != OUT_F16Q) return cudaErrorNotSupported;
    const int64_t chunks = (a.K / 8 + threads - 1) / threads;  // per thread
    const unsigned grid = (unsigned)a.M;
    prof_begin(0, st);
#define GBQ_ID_LAUNCH(CH, TH)                                                                          \
    do {                                                                                               \
        if (out_kind == OUT_S8)                                                                        \
            quant_identity_kernel<OUT_S8, CH, TH><<<grid, TH, 0, st>>>(a);                             \
        else                                                                                           \
            quant_identity_kernel<OUT_F16Q, CH, TH><<<grid, TH, 0, st>>>(a);                           \
    } while (0)
    if (threads == 512) {
        if (chunks <= 4)
            GBQ_ID_LAUNCH(4, 512);
        else
            GBQ_ID_LAUNCH(8, 512);
    } else {
        if (chunks <= 4)
            GBQ_ID_LAUNCH(4, 256);
        else
            GBQ_ID_LAUNCH(8, 256);
    }
#undef GBQ_ID_LAUNCH
    prof_end(st);
    return cudaGetLastError();
}

}  // namespace gbq
