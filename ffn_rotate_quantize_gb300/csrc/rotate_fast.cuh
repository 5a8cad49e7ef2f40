// rotate_fast.cuh -- three-pass rotate(+quantize) kernels for the wide factors
// n = 64 (K = 4096) and n = 128 (K = 16384), one group per row.
//
// What they compute is the same as rotq_kernel (PyPI page "xpu-kernels 0.2.0",
// "Algorithm: fused ConvRot rotation"): V = (H_n X H_n) / n per row, in the
// library's fixed level order (hadamard_pass), then the optional per-row INT8
// quantization -- bit for bit the values of rotq_kernel.
//
// Why three passes: holding a whole length-n line per thread (the two-pass
// layout) needs 128 fp32 values per thread, ~255 registers and so only a few
// warps per SM, which leaves these HBM-streaming kernels latency-bound.  Here a
// thread holds 32 values (16 float2 pairs): four index bits in registers (two
// base-4 digits, so two H4 levels run on registers), one bit across the pair,
// the rest across threads.  Three passes cover the levels, with two exchanges
// through a shared-memory tile:
//   n = 64  (bits i0..i5 j0..j5; 128 threads per row)
//     A: regs {i0..i3}, pair j0   : i(0,1) i(2,3)
//     B: regs {i4,i5,j4,j5}, pair j0 : i(4,5) j(4,5)      (in place in the tile)
//     C: regs {j0..j3}, pair i0   : j(0,1) j(2,3)
//   n = 128 (bits i0..i6 j0..j6; 512 threads per row)
//     A: regs {i0..i3}, pair i6   : H2(i6) i(0,1) i(2,3)
//     B: regs {i4,i5,j4,j5}, pair i6 : i(4,5) j(4,5)
//     C: regs {j0..j3}, pair j6   : H2(j6) j(0,1) j(2,3), then the exact halving
// Pass C leaves each thread 16 contiguous outputs of one or two rows of X, so
// results (codes or bf16) go to global memory with 16-byte stores.  Inputs come
// from a shared-memory stage filled by bulk copies (cp.async.bulk); for n = 64
// the stage is double-buffered (the next row streams in while this one is
// rotated), for n = 128 the tile reuses the stage's memory and two CTAs per SM
// alternate.
#pragma once

#include "rotate_impl.cuh"

namespace gbq {

struct FastArgs {
    RotArgs a;
    uint32_t stage_bytes;  // one stage (inputs of one row), multiple of 128
    uint32_t tile_off;     // byte offset of the tile
    uint32_t misc_off;     // byte offset of barriers / amax slots
    int stages;
};

// n = 64 tile: row pitch 35 float2, and one pad float2 after the first 16 of a row (column jh is stored
// at jh + jh / 16), which makes every 8-byte access of the three passes free of bank conflicts.
constexpr int kP64 = 35;
__device__ __forceinline__ int t64(int i, int jh) { return i * kP64 + jh + (jh >> 4); }
constexpr int kP128A = 129;  // n = 128 tile pitch for passes A/B (float2, pairs over i6)
constexpr int kP128C = 66;   // n = 128 tile pitch for pass C (float2, pairs over j6)
constexpr uint32_t kFastMisc = 256;

__host__ __device__ constexpr uint32_t fast_tile_bytes(int logn) {
    return logn == 6 ? (uint32_t)(64 * kP64 * 8)
                     : (uint32_t)((64 * kP128A * 8) > (128 * kP128C * 8) ? (64 * kP128A * 8) : (128 * kP128C * 8));
}

// Quantized output of one 16-value chunk (words: 4 codes per word) or bf16 output.
template <int OUT>
__device__ __forceinline__ void store_chunk_codes(void *out, int64_t off, const uint32_t (&w)[4]) {
    store_codes<OUT, 4>(out, off, w);
}
__device__ __forceinline__ void store_chunk_bf16(void *out, int64_t off, const float (&x)[16]) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t *>(&b2);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(out) + off);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Sum of |code| over a thread's 32 int8 codes (8 words of four).
__device__ __forceinline__ int codes_l1(const uint32_t (&w)[2][4]) {
    unsigned acc = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc = __dp4a(__vabsss4(w[h][k]), 0x01010101u, acc);
    return (int)acc;
}

// Per-warp totals of a per-thread value, stored by lane 0 of each warp at dst[warp].  In pass C
// of both three-pass kernels warp w holds exactly elements [1024 w, 1024 w + 1024) of the row,
// so these are the row's per-1024-block sums.
__device__ __forceinline__ void warp_sums_store(int v, int32_t *dst) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) dst[threadIdx.x >> 5] = v;
}

// Row scale from the per-warp maxima (NW warps) after a CTA barrier.
__device__ __forceinline__ float block_amax(float m, float *wmax, int nwarps) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    float a = wmax[0];
    for (int w = 1; w < nwarps; ++w) a = fmaxf(a, wmax[w]);
    return a;
}

__device__ __forceinline__ float pairs_amax(const float2 (&v)[16]) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, pair_max_abs(v[j]));
    return m;
}

// Bulk-copy the NIN inputs of one row into a stage.
template <int IN>
__device__ __forceinline__ void fast_issue(const RotArgs &p, int64_t row, uint8_t *dst, uint64_t *bar) {
    constexpr int NIN = in_count(IN);
    const uint32_t rb = p.row_in_bytes;
    const int64_t off = row * p.ld_in * in_elem_bytes(IN);
    if (!GBQ_IN_RANGE(p.status, off, rb, p.M * p.ld_in * in_elem_bytes(IN))) {
        mbar_arrive_expect_tx(bar, 0);  // debug builds: the copy is skipped, the stage completes empty
        return;
    }
    mbar_arrive_expect_tx(bar, NIN * rb);
    bulk_g2s(dst, reinterpret_cast<const uint8_t *>(p.in0) + off, rb, bar);
    if (NIN == 2) bulk_g2s(dst + rb, reinterpret_cast<const uint8_t *>(p.in1) + off, rb, bar);
}

// ============================================================== n = 64
// One row through the three passes: s0 / s1 the row's staged input(s), rs its
// row scale, T the 64 x kP64 tile.  Threads tau = 0..127 take part and meet at
// bar() (a CTA barrier or a named barrier over those 128 threads); after_a() runs
// (on every thread) right after the barrier that ends the reads of the stage.
// Leaves this thread's pass-C pairs: v[c] = (X[2r][16 jq + c], X[2r + 1][16 jq + c])
// with r = tau / 4, jq = tau % 4.
template <int IN, class Bar, class Hook>
__device__ __forceinline__ void rot64_row(const RotArgs &p, const uint8_t *s0, const uint8_t *s1, float rs,
                                          float2 *T, int tau, Bar bar, Hook after_a, float2 (&v)[16]) {
    // ---- pass A: regs i0..i3, pair j0; thread = (j1..j5, i4 i5) ----
    {
        const int jh = tau & 31, ih = tau >> 5;
#pragma unroll
        for (int a = 0; a < 16; ++a) v[a] = staged_pair<IN>(p, s0, s1, rs, 64 * (a + 16 * ih) + 2 * jh);
        h4_level<16, 0>(v);
        h4_level<16, 2>(v);
#pragma unroll
        for (int a = 0; a < 16; ++a) T[t64(a + 16 * ih, jh)] = v[a];
    }
    bar();
    after_a();
    // ---- pass B: regs (i4 i5 | j4 j5), pair j0; thread = (i0..i3, j1 j2 j3); in place ----
    {
        const int il = tau & 15, jm = tau >> 4;
#pragma unroll
        for (int b = 0; b < 16; ++b) v[b] = T[t64(il + 16 * (b & 3), jm + 8 * (b >> 2))];
        h4_level<16, 0>(v);
        h4_level<16, 2>(v);
#pragma unroll
        for (int b = 0; b < 16; ++b) T[t64(il + 16 * (b & 3), jm + 8 * (b >> 2))] = v[b];
    }
    bar();
    // ---- pass C: regs j0..j3, pair i0 (rows 2r, 2r+1); thread = (j4 j5, i1..i5) ----
    const int r = tau >> 2, jq = tau & 3;
    // Slots 8 jq .. 8 jq + 7 of rows 2r and 2r + 1 (all on one side of the pad: 8 jq / 16 = jq / 2).
    const float2 *t0 = T + t64(2 * r, 8 * jq);
    const float2 *t1 = T + t64(2 * r + 1, 8 * jq);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float2 a0 = t0[m], b0 = t1[m];
        v[2 * m] = f2(a0.x, b0.x);
        v[2 * m + 1] = f2(a0.y, b0.y);
    }
    h4_level<16, 0>(v);
    h4_level<16, 2>(v);
}

template <int IN, int OUT>
__global__ void __launch_bounds__(128) rot64_kernel(const __grid_constant__ FastArgs f) {
    const RotArgs &p = f.a;
    extern __shared__ __align__(128) uint8_t smem[];
    float2 *T = reinterpret_cast<float2 *>(smem + f.tile_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + f.misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + f.misc_off + 16);
    float *wmax = reinterpret_cast<float *>(smem + f.misc_off + 32);
    const int tau = threadIdx.x;
    const uint32_t rb = p.row_in_bytes;
    pdl_allow_dependents();  // a GEMM launched after this kernel may set itself up meanwhile

    if (tau == 0) {
        for (int s = 0; s < f.stages; ++s) mbar_init(&full[s], 1);
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tau == 0)
        for (int s = 0; s < f.stages; ++s) {
            const int64_t r = blockIdx.x + (int64_t)s * gridDim.x;
            if (r < p.M) fast_issue<IN>(p, r, smem + (size_t)s * f.stage_bytes, &full[s]);
        }

    int64_t it = 0;
    int64_t pending = -1;  // last iteration whose stage was issued but not yet consumed
    {
        const int64_t r_last = blockIdx.x + (int64_t)(f.stages - 1) * gridDim.x;
        pending = r_last < p.M ? f.stages - 1 : (blockIdx.x < p.M ? 0 : -1);
    }
    bool failed = false;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++it) {
        const int st = (int)(it % f.stages);
        const uint8_t *s0 = smem + (size_t)st * f.stage_bytes;
        const bool ok = mbar_wait(&full[st], (uint32_t)((it / f.stages) & 1), p.status, abort);
        if (!__syncthreads_and(ok)) {  // also: the previous row's pass-C reads of the tile are done
            failed = true;
            break;
        }
        float rs = 0.0f;
        if (IN == IN_S8_ROWSCALE || IN == IN_ACC_GLU || IN == IN_ACC_ROWSCALE) rs = __ldg(p.in_scale + row);

        float2 v[16];
        rot64_row<IN>(
            p, s0, s0 + rb, rs, T, tau, [] { __syncthreads(); },
            [&] {
                if (tau == 0) {  // every thread has read the stage: stream the row `stages` iterations ahead into it
                    const int64_t r2 = row + (int64_t)f.stages * gridDim.x;
                    if (r2 < p.M) {
                        fast_issue<IN>(p, r2, smem + (size_t)st * f.stage_bytes, &full[st]);
                        pending = it + f.stages;
                    }
                }
            },
            v);
        const int r = tau >> 2, jq = tau & 3;
        const int64_t o0 = row * 4096 + (2 * r) * 64 + 16 * jq;  // element offset of row 2r's chunk
        const bool out_ok = GBQ_IN_RANGE(p.status, o0, 64 + 16, p.M * p.K);
        if constexpr (OUT == OUT_BF16) {
            float x0[16], x1[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                x0[c] = v[c].x;
                x1[c] = v[c].y;
            }
            if (out_ok) {
                store_chunk_bf16(p.out, o0, x0);
                store_chunk_bf16(p.out, o0 + 64, x1);
            }
        } else {
            const float amax = block_amax(pairs_amax(v), wmax, 4);
            const float s = __fdiv_rn(amax, 127.0f);
            if (tau == 0) p.out_scale[row] = s;
            uint32_t words[2][4];
            quant_codes<16>(v, s, words);
            if (out_ok) {
                store_chunk_codes<OUT>(p.out, o0, words[0]);
                store_chunk_codes<OUT>(p.out, o0 + 64, words[1]);
            }
            if (p.out_l1) warp_sums_store(codes_l1(words), p.out_l1 + row * 4);  // K = 4096: 4 blocks
        }
    }
    if (tau == 0 && failed) {
        // A wait gave up: let every copy still in flight land (bounded) before the CTA leaves.
        for (int64_t k = it; k <= pending; ++k) {
            const int st = (int)(k % f.stages);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&full[st], (uint32_t)((k / f.stages) & 1)) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ============================================================== n = 128
template <int IN, int OUT>
__global__ void __launch_bounds__(512, 2) rot128_kernel(const __grid_constant__ FastArgs f) {
    const RotArgs &p = f.a;
    extern __shared__ __align__(128) uint8_t smem[];
    float2 *T = reinterpret_cast<float2 *>(smem);  // the tile reuses the stage's memory
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + f.misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + f.misc_off + 16);
    float *wmax = reinterpret_cast<float *>(smem + f.misc_off + 32);
    const int tau = threadIdx.x;
    const uint32_t rb = p.row_in_bytes;
    pdl_allow_dependents();  // a GEMM launched after this kernel may set itself up meanwhile

    if (tau == 0) {
        mbar_init(&full[0], 1);
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (tau == 0 && blockIdx.x < p.M) fast_issue<IN>(p, blockIdx.x, smem, &full[0]);

    int64_t it = 0;
    bool failed = false;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++it) {
        const bool ok = mbar_wait(&full[0], (uint32_t)(it & 1), p.status, abort);
        if (!__syncthreads_and(ok)) {
            failed = true;
            break;
        }
        float rs = 0.0f;
        if (IN == IN_S8_ROWSCALE || IN == IN_ACC_GLU || IN == IN_ACC_ROWSCALE) rs = __ldg(p.in_scale + row);
        float2 v[16];
        // ---- pass A: regs i0..i3, pair i6; thread = (j0..j6, i4 i5) ----
        {
            const int j = tau & 127, ih = tau >> 7;
#pragma unroll
            for (int a = 0; a < 16; ++a) {
                const int e = 128 * (a + 16 * ih) + j;
                v[a] = f2(staged_one<IN>(p, smem, smem + rb, rs, e), staged_one<IN>(p, smem, smem + rb, rs, e + 8192));
            }
            h2_pairs<16>(v);
            h4_level<16, 0>(v);
            h4_level<16, 2>(v);
            __syncthreads();  // every stage read is done: the tile overwrites it
#pragma unroll
            for (int a = 0; a < 16; ++a) T[(a + 16 * ih) * kP128A + j] = v[a];
        }
        __syncthreads();
        // ---- pass B: regs (i4 i5 | j4 j5), pair i6; thread = (i0..i3, j0..j3, j6) ----
        {
            const int il = tau & 15, jl = (tau >> 4) & 15, j6 = tau >> 8;
#pragma unroll
            for (int b = 0; b < 16; ++b) v[b] = T[(il + 16 * (b & 3)) * kP128A + jl + 16 * (b >> 2) + 64 * j6];
            h4_level<16, 0>(v);
            h4_level<16, 2>(v);
            __syncthreads();  // every pass-B read is done: re-lay the tile out as pairs over j6
            // element (i, j) -> pair slot (i, j mod 64), half j6; within a row's 16-column block
            // q = (j mod 64) / 16, the float4 m = (j mod 16) / 2 sits at m ^ 2q (conflict-free reads in C).
            float *Tf = reinterpret_cast<float *>(smem);
#pragma unroll
            for (int b = 0; b < 16; ++b) {
                const int i = il + 16 * (b & 3);
                const int jlo = jl + 16 * (b >> 2);
                const int q = jlo >> 4, c = jlo & 15;
                const int col = 16 * q + 2 * ((c >> 1) ^ (2 * q)) + (c & 1);
                Tf[(i * kP128C + col) * 2 + j6] = v[b].x;
                Tf[((i + 64) * kP128C + col) * 2 + j6] = v[b].y;
            }
        }
        __syncthreads();
        // ---- pass C: regs j0..j3, pair j6; thread = (j4 j5, i0..i6) ----
        const int jq = tau & 3, i = tau >> 2;
        {
            const float4 *t = reinterpret_cast<const float4 *>(T + i * kP128C + 16 * jq);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 a = t[m ^ (2 * jq)];
                v[2 * m] = f2(a.x, a.y);
                v[2 * m + 1] = f2(a.z, a.w);
            }
            h2_pairs<16>(v);
            h4_level<16, 0>(v);
            h4_level<16, 2>(v);
            const float2 half2 = f2(0.5f, 0.5f);
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = __fmul2_rn(v[c], half2);  // the two H2 levels: (1/sqrt2)^2
        }
        const int64_t o0 = row * 16384 + i * 128 + 16 * jq;  // element offset of the j6 = 0 chunk
        const bool out_ok = GBQ_IN_RANGE(p.status, o0, 64 + 16, p.M * p.K);
        if constexpr (OUT == OUT_BF16) {
            float x0[16], x1[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                x0[c] = v[c].x;
                x1[c] = v[c].y;
            }
            __syncthreads();  // pass-C reads done before the next row's copy lands in the tile
            if (tau == 0 && row + gridDim.x < p.M) fast_issue<IN>(p, row + gridDim.x, smem, &full[0]);
            if (out_ok) {
                store_chunk_bf16(p.out, o0, x0);
                store_chunk_bf16(p.out, o0 + 64, x1);
            }
        } else {
            const float amax = block_amax(pairs_amax(v), wmax, 16);  // its barrier also ends the pass-C reads
            if (tau == 0 && row + gridDim.x < p.M) fast_issue<IN>(p, row + gridDim.x, smem, &full[0]);
            const float s = __fdiv_rn(amax, 127.0f);
            if (tau == 0) p.out_scale[row] = s;
            uint32_t words[2][4];
            quant_codes<16>(v, s, words);
            if (out_ok) {
                store_chunk_codes<OUT>(p.out, o0, words[0]);
                store_chunk_codes<OUT>(p.out, o0 + 64, words[1]);
            }
            if (p.out_l1) warp_sums_store(codes_l1(words), p.out_l1 + row * 16);  // K = 16384: 16 blocks
        }
    }
    if (tau == 0 && failed) {
        const uint64_t t0 = globaltimer();  // the copy of the failed iteration may still land
        while (!mbar_try_wait(&full[0], (uint32_t)(it & 1)) && globaltimer() - t0 < kWaitLimitNs) {
        }
    }
}

}  // namespace gbq
