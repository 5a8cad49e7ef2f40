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
        if (ch < nchunks && GBQ_IN_RANGE(p.status, row * p.ld_in + 8 * ch, 8, p.M * p.ld_in)) {
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
        if (!GBQ_IN_RANGE(p.status, row * p.K + 8 * ch, 8, p.M * p.K)) continue;
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
// dy rows of linear_dx_int8).  Persistent CTAs of 512 threads, two per SM, walk
// the rows blockIdx.x, blockIdx.x + gridDim.x, ...; every row reaches shared
// memory in one bulk copy issued up to six rows ahead, so HBM keeps streaming
// while the CTAs work, and the two CTAs of an SM overlap one row's reduction
// with the other's arithmetic.  Two passes over the staged row: the maximum,
// then the codes (the row is re-read from shared memory, not held in
// registers).  Each thread owns four chunks of 8 columns and keeps their column
// scales in registers for all rows; pairs of values go through the packed
// fp32x2 instructions, each lane rounded as the scalar one.  Arithmetic, codes,
// scales and block sums are those of quant_identity_kernel.
// ---------------------------------------------------------------------------
constexpr int kIdsThreads = 512;
constexpr int kIdsChunks = 4;  // chunks of 8 values per thread: K <= 16384
constexpr int kIdsStageCap = 6;
constexpr size_t kIdsSmemCap = 96 * 1024;  // per CTA: two CTAs per SM

// Eight staged bf16 values of one chunk as fp32 pairs, times their column scales.
__device__ __forceinline__ void ids_values(const uint4 w, const float2 (&cs)[4], bool has_cs, float2 (&v)[4]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        v[h] = make_float2(__uint_as_float(ws[h] << 16), __uint_as_float(ws[h] & 0xFFFF0000u));
        if (has_cs) v[h] = __fmul2_rn(v[h], cs[h]);
    }
}

template <int OUT>
__global__ void __launch_bounds__(kIdsThreads, 2) quant_identity_stream_kernel(IdArgs p, int stages) {
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
            if (!GBQ_IN_RANGE(p.status, row_of(issued) * p.ld_in, row_bytes / 2, p.M * p.ld_in)) {
                mbar_arrive_expect_tx(&full[issued], 0);  // debug builds: skipped, the stage completes empty
                continue;
            }
            mbar_arrive_expect_tx(&full[issued], row_bytes);
            bulk_g2s(ids_smem + (size_t)issued * row_bytes, in + row_of(issued) * p.ld_in, row_bytes, &full[issued]);
        }
    }
    const bool has_cs = p.col_scale != nullptr;
    float2 cs[kIdsChunks][4];
#pragma unroll
    for (int c = 0; c < kIdsChunks; ++c) {
        const int ch = tid + c * kIdsThreads;
        if (has_cs && ch < nchunks) {
            const float4 c0 = __ldg(reinterpret_cast<const float4 *>(p.col_scale + 8 * ch));
            const float4 c1 = __ldg(reinterpret_cast<const float4 *>(p.col_scale + 8 * ch + 4));
            cs[c][0] = make_float2(c0.x, c0.y), cs[c][1] = make_float2(c0.z, c0.w);
            cs[c][2] = make_float2(c1.x, c1.y), cs[c][3] = make_float2(c1.z, c1.w);
        } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) cs[c][h] = make_float2(1.0f, 1.0f);
        }
    }
    __syncthreads();  // barriers initialised

    for (int64_t i = 0; i < n_local; ++i) {
        const int stage = (int)(i % stages);
        const bool ok = mbar_wait(&full[stage], (uint32_t)((i / stages) & 1), p.status, &abort_flag);
        const uint4 *src = reinterpret_cast<const uint4 *>(ids_smem + (size_t)stage * row_bytes);
        // pass 1: the row's maximum
        float m = 0.0f;
#pragma unroll
        for (int c = 0; c < kIdsChunks; ++c) {
            const int ch = tid + c * kIdsThreads;
            if (ok && ch < nchunks) {
                float2 v[4];
                ids_values(src[ch], cs[c], has_cs, v);
#pragma unroll
                for (int h = 0; h < 4; ++h) m = fmaxf(m, fmaxf(fabsf(v[h].x), fabsf(v[h].y)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_red[warp] = m;
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
        float amax = s_red[lane & (kIdsThreads / 32 - 1)];
#pragma unroll
        for (int o = kIdsThreads / 64; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(amax, 127.0f);
        const int64_t row = row_of(i);
        if (tid == 0) p.out_scale[row] = s;
        // pass 2: codes rne(fl(v/s)) as in quant_identity_kernel -- the reciprocal path, then IEEE division
        // for a chunk with a product within 1e-4 of a half-integer (or every chunk, for a tiny scale)
        const bool recip = s >= 1e-30f;
        const float r = recip ? __frcp_rn(s) : 0.0f;
        const float2 r2 = make_float2(r, r), magic = make_float2(12582912.0f, 12582912.0f);
        const float2 nmagic = make_float2(-12582912.0f, -12582912.0f), neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
        for (int c = 0; c < kIdsChunks; ++c) {
            const int ch = tid + c * kIdsThreads;
            uint32_t w0 = 0, w1 = 0;
            if (ch < nchunks) {
                float2 v[4];
                ids_values(src[ch], cs[c], has_cs, v);
                bool bad = !recip;
                if (recip) {
                    uint32_t mb[8];
                    float dmax = 0.0f;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 t = __fmul2_rn(v[h], r2);
                        const float2 mm = __fadd2_rn(t, magic);
                        const float2 d = __ffma2_rn(__fadd2_rn(mm, nmagic), neg1, t);  // t - (mm - magic)
                        dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
                        mb[2 * h] = __float_as_uint(mm.x);
                        mb[2 * h + 1] = __float_as_uint(mm.y);
                    }
                    bad = dmax > 0.4999f;
                    w0 = __byte_perm(__byte_perm(mb[0], mb[1], 0x0040), __byte_perm(mb[2], mb[3], 0x0040), 0x5410);
                    w1 = __byte_perm(__byte_perm(mb[4], mb[5], 0x0040), __byte_perm(mb[6], mb[7], 0x0040), 0x5410);
                }
                if (bad) {
                    w0 = w1 = 0;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        int q0 = 0, q1 = 0;
                        if (s != 0.0f) {
                            q0 = max(-127, min(127, __float2int_rn(__fdiv_rn(v[h].x, s))));
                            q1 = max(-127, min(127, __float2int_rn(__fdiv_rn(v[h].y, s))));
                        }
                        const uint32_t pair = (uint32_t)(q0 & 0xFF) | (uint32_t)(q1 & 0xFF) << 8;
                        if (h < 2)
                            w0 |= pair << (16 * h);
                        else
                            w1 |= pair << (16 * (h - 2));
                    }
                }
                if (!GBQ_IN_RANGE(p.status, row * p.K + 8 * ch, 8, p.M * p.K)) {
                } else if constexpr (OUT == OUT_S8) {
                    reinterpret_cast<uint2 *>(reinterpret_cast<int8_t *>(p.out) + row * p.K)[ch] = make_uint2(w0, w1);
                } else {
                    reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(p.out) + row * p.K)[ch] =
                        make_uint4(s8pair_to_f16x2(__byte_perm(w0, 0, 0x4140)), s8pair_to_f16x2(__byte_perm(w0, 0, 0x4342)),
                                   s8pair_to_f16x2(__byte_perm(w1, 0, 0x4140)), s8pair_to_f16x2(__byte_perm(w1, 0, 0x4342)));
                }
            }
            if (p.out_l1) {  // uniform over the CTA; a warp's 32 chunks of one slot lie in one 1024-long block
                int l = __dp4a((int)__vabsss4(w0), 0x01010101, __dp4a((int)__vabsss4(w1), 0x01010101, 0));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                if (lane == 0) s_part[warp][c] = l;
            }
        }
        __syncthreads();  // the stage is read, the block partials are complete
        if (tid == 0 && issued < n_local) {  // row i + stages into the stage just read
            if (GBQ_IN_RANGE(p.status, row_of(issued) * p.ld_in, row_bytes / 2, p.M * p.ld_in)) {
                mbar_arrive_expect_tx(&full[stage], row_bytes);
                bulk_g2s(ids_smem + (size_t)stage * row_bytes, in + row_of(issued) * p.ld_in, row_bytes, &full[stage]);
            } else {
                mbar_arrive_expect_tx(&full[stage], 0);  // debug builds: skipped, the stage completes empty
            }
            ++issued;
        }
        if (p.out_l1 && tid < nb) {
            // block b holds chunks [128 b, 128 b + 128): slot c = b / 4 of warps 4 (b % 4) .. 4 (b % 4) + 3
            constexpr int kGroups = kIdsThreads / 128;
            const int c = tid / kGroups, w = 4 * (tid % kGroups);
            p.out_l1[row * nb + tid] = s_part[w][c] + s_part[w + 1][c] + s_part[w + 2][c] + s_part[w + 3][c];
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
    const int64_t ctas = 2 * (int64_t)a.num_sms;
    const unsigned grid = (unsigned)(a.M < ctas ? a.M : ctas);
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
