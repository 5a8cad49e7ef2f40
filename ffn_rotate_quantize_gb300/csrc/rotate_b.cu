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

// ---------------------------------------------------------------------------
// Streaming variant for long rows of fp16-coded output (8192 <= K <= 16384, the
// dy rows of linear_dx_int8).  One persistent CTA of 1024 threads per SM walks the rows
// blockIdx.x, blockIdx.x + gridDim.x, ...; every row reaches shared memory in one
// bulk copy issued up to kIdsStageCap rows ahead, so HBM keeps streaming while
// the CTA reduces, quantizes and stores the rows already landed (the register
// kernel above stops loading during each row's reduction).  Each thread owns two
// chunks of 8 columns and keeps their column scales in registers for all rows.
// Arithmetic, codes, scales and block sums are those of quant_identity_kernel.
// ---------------------------------------------------------------------------
constexpr int kIdsThreads = 1024;
constexpr int kIdsChunks = 2;  // chunks of 8 values per thread: K <= 16384
constexpr int kIdsStageCap = 6;
constexpr size_t kIdsSmemCap = 200 * 1024;

template <int OUT>
__global__ void __launch_bounds__(kIdsThreads, 1) quant_identity_stream_kernel(IdArgs p, int stages) {
    extern __shared__ __align__(128) unsigned char ids_smem[];
    __shared__ uint64_t full[kIdsStageCap];
    __shared__ int abort_flag;
    __shared__ float s_red[kIdsThreads / 32];
    __shared__ int s_part[kIdsThreads / 32][kIdsChunks];  // per warp and chunk slot: sum of |code|
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t G = gridDim.x;
    const int64_t n_local = (p.M - (int64_t)blockIdx.x + G - 1) / G;  // rows of this CTA
    const uint32_t row_bytes = (uint32_t)(p.K * 2);
    const int nchunks = (int)(p.K / 8);
    const int nb = (int)((p.K + 1023) / 1024);
    const uint16_t *in = reinterpret_cast<const uint16_t *>(p.in);
    auto row_of = [&](int64_t i) { return (int64_t)blockIdx.x + i * G; };
    pdl_allow_dependents();  // a GEMM launched after this kernel may set itself up meanwhile
    int64_t issued = 0;      // rows whose copy was issued (thread 0's count)
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_mbar_init();
        for (; issued < n_local && issued < stages; ++issued) {
            mbar_arrive_expect_tx(&full[issued], row_bytes);
            bulk_g2s(ids_smem + (size_t)issued * row_bytes, in + row_of(issued) * p.ld_in, row_bytes, &full[issued]);
        }
    }
    const bool has_cs = p.col_scale != nullptr;
    float cs[kIdsChunks][8];
#pragma unroll
    for (int c = 0; c < kIdsChunks; ++c) {
        const int ch = tid + c * kIdsThreads;
        if (has_cs && ch < nchunks) {
            const float4 c0 = __ldg(reinterpret_cast<const float4 *>(p.col_scale + 8 * ch));
            const float4 c1 = __ldg(reinterpret_cast<const float4 *>(p.col_scale + 8 * ch + 4));
            cs[c][0] = c0.x, cs[c][1] = c0.y, cs[c][2] = c0.z, cs[c][3] = c0.w;
            cs[c][4] = c1.x, cs[c][5] = c1.y, cs[c][6] = c1.z, cs[c][7] = c1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) cs[c][e] = 1.0f;
        }
    }
    __syncthreads();  // barriers initialised

    for (int64_t i = 0; i < n_local; ++i) {
        const int stage = (int)(i % stages);
        const bool ok = mbar_wait(&full[stage], (uint32_t)((i / stages) & 1), p.status, &abort_flag);
        const uint4 *src = reinterpret_cast<const uint4 *>(ids_smem + (size_t)stage * row_bytes);
        float v[kIdsChunks][8];
        float m = 0.0f;
#pragma unroll
        for (int c = 0; c < kIdsChunks; ++c) {
            const int ch = tid + c * kIdsThreads;
            if (ok && ch < nchunks) {
                const uint4 w = src[ch];
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    v[c][2 * h] = __uint_as_float(ws[h] << 16);
                    v[c][2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
                }
                if (has_cs) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[c][e] = __fmul_rn(v[c][e], cs[c][e]);
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
        if (lane == 0) s_red[warp] = m;
        // The row is in registers (every value fed the maximum above): its stage is free.
        if (__syncthreads_or(!ok)) {
            // A wait gave up: the copies still in flight land (bounded) before the CTA leaves.
            if (tid == 0) {
                for (int64_t j = i; j < issued; ++j) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(&full[j % stages], (uint32_t)((j / stages) & 1)) &&
                           globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
            return;
        }
        if (tid == 0 && issued < n_local) {  // row i + stages into the stage just read
            mbar_arrive_expect_tx(&full[stage], row_bytes);
            bulk_g2s(ids_smem + (size_t)stage * row_bytes, in + row_of(issued) * p.ld_in, row_bytes, &full[stage]);
            ++issued;
        }
        float amax = 0.0f;
#pragma unroll
        for (int w = 0; w < kIdsThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
        const float s = __fdiv_rn(amax, 127.0f);
        const int64_t row = row_of(i);
        if (tid == 0) p.out_scale[row] = s;
        // Codes rne(fl(v/s)) as in quant_identity_kernel: the reciprocal path, then IEEE division for
        // the chunks whose products lie within 1e-4 of a half-integer (or all, for a tiny scale).
        uint32_t words[kIdsChunks][2];
        uint32_t bad = 0xFFFFFFFFu;
        if (s >= 1e-30f) {
            bad = 0;
            const float r = __frcp_rn(s);
#pragma unroll
            for (int c = 0; c < kIdsChunks; ++c) {
                uint32_t mb[8];
                float dmax = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float t = __fmul_rn(v[c][e], r);
                    const float mm = __fadd_rn(t, 12582912.0f);
                    dmax = fmaxf(dmax, fabsf(__fsub_rn(t, __fsub_rn(mm, 12582912.0f))));
                    mb[e] = __float_as_uint(mm);
                }
                if (dmax > 0.4999f) bad |= 1u << c;
                words[c][0] = __byte_perm(__byte_perm(mb[0], mb[1], 0x0040), __byte_perm(mb[2], mb[3], 0x0040), 0x5410);
                words[c][1] = __byte_perm(__byte_perm(mb[4], mb[5], 0x0040), __byte_perm(mb[6], mb[7], 0x0040), 0x5410);
            }
        }
        if (bad) {
#pragma unroll
            for (int c = 0; c < kIdsChunks; ++c) {
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
        if (p.out_l1) {  // uniform over the CTA; a warp's 32 chunks of one slot lie in one 1024-long block
#pragma unroll
            for (int c = 0; c < kIdsChunks; ++c) {
                int l = __dp4a((int)__vabsss4(words[c][0]), 0x01010101, __dp4a((int)__vabsss4(words[c][1]), 0x01010101, 0));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                if (lane == 0) s_part[warp][c] = l;
            }
        }
#pragma unroll
        for (int c = 0; c < kIdsChunks; ++c) {
            const int ch = tid + c * kIdsThreads;
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
        __syncthreads();  // block partials complete; s_red and s_part free for the next row after this
        if (p.out_l1 && tid < nb) {
            // block b holds chunks [128 b, 128 b + 128): slot c = b / 8 of warps 4 (b % 8) .. 4 (b % 8) + 3
            constexpr int kGroups = kIdsThreads / 128;
            const int c = tid / kGroups, w0 = 4 * (tid % kGroups);
            p.out_l1[row * nb + tid] = s_part[w0][c] + s_part[w0 + 1][c] + s_part[w0 + 2][c] + s_part[w0 + 3][c];
        }
    }
}

template <int OUT>
static cudaError_t launch_quant_identity_stream(const IdArgs &a, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(quant_identity_stream_kernel<OUT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIdsSmemCap);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const size_t row_bytes = (size_t)a.K * 2;
    int stages = (int)(kIdsSmemCap / row_bytes);
    if (stages > kIdsStageCap) stages = kIdsStageCap;
    const unsigned grid = (unsigned)(a.M < a.num_sms ? a.M : a.num_sms);
    prof_begin(0, st);
    quant_identity_stream_kernel<OUT><<<grid, kIdsThreads, (size_t)stages * row_bytes, st>>>(a, stages);
    prof_end(st);
    return cudaGetLastError();
}

cudaError_t launch_quant_identity(int out_kind, IdArgs a, cudaStream_t st) {
    const int threads = (a.K / 8 >= 2048) ? 512 : 256;
    if (a.K % 8 != 0 || a.K / 8 > (int64_t)threads * kIdChunkCap) return cudaErrorNotSupported;
    if (a.M > 0x7fffffff) return cudaErrorInvalidValue;
    if (out_kind != OUT_S8 && out_kind != OUT_F16Q) return cudaErrorNotSupported;
    if (a.M == 0) return cudaSuccess;
    // Long rows of fp16-coded output stream through shared memory (bulk copies need a 16-byte aligned
    // row start).  For int8 output the register kernel below is faster (about 71 us against 85 us
    // at 4096 x 16384): its two CTAs per SM alternate their reductions, where the streaming CTA waits.
    if (out_kind == OUT_F16Q && a.status != nullptr && a.num_sms > 0 && a.K >= 8192 &&
        a.K <= (int64_t)kIdsThreads * kIdsChunks * 8 && a.ld_in % 8 == 0 && (reinterpret_cast<uintptr_t>(a.in) & 15) == 0)
        return launch_quant_identity_stream<OUT_F16Q>(a, st);
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
