// gemm_i8.cu -- exact int8 x int8 -> int32 GEMM on the sm_103a tensor cores.
//
// What it computes: acc[m, n] = sum_k q[m, k] * W8[n, k] exactly (the int8 GEMM
// of the rotated-INT8 linear layer, PyPI page "xpu-kernels 0.2.0", "Use from C"),
// followed by one of the epilogues of gemm.h (the page's dequant epilogue:
// out = acc * x_scale[m] * w_scale[n] + bias[n]).
//
// sm_103a has no int8 tcgen05 MMA kind, so the contraction runs on kind::f16:
//   * int8 values are exact in fp16, products (|p| <= 127^2) are exact, and an
//     fp32 accumulator is exact while every partial sum stays below 2^24 in
//     magnitude; 1024 products of magnitude <= 127^2 sum to < 2^24.
//   * K is cut into chunks of 1024.  Chunks alternate between two fp32 TMEM
//     accumulators; the epilogue warps drain a finished chunk (fp32 -> int32,
//     exact) into an int32 running total kept in TMEM, while the MMA works on
//     the next chunk in the other accumulator.
//
// Tile: 128 weight rows (TMEM lanes, MMA M) x 128 tokens (MMA N) x 64 K per
// pipeline stage.  The weight is the A operand and lives in TMEM: converter
// warps read the TMA-staged int8 tile from shared memory, widen it to fp16
// (byte-permute + one half2 subtract per pair) and tcgen05.st it into a 4-stage
// TMEM ring, so the widened weight never costs shared-memory bandwidth.  The
// activations are the B operand: fp16-coded integers staged by TMA with the
// 128-byte swizzle.  One persistent CTA per SM walks the tile list.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 4-7 converters, warps 8-11 epilogue (each converter/epilogue
// warp owns the TMEM lane quadrant warp%4).  Every mbarrier wait is bounded.
//
// TMEM columns: [0,128) A ring (4 x 32), [128,256) acc0, [256,384) acc1,
// [384,512) int32 totals.
#include "common.cuh"
#include "gemm.h"

namespace gbq {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kAStages = 4;
constexpr int kChunkStages = 16;  // 16 * 64 = 1024 K per fp32 accumulator
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0, kColAcc0 = 128, kColAcc1 = 256, kColTot = 384;
constexpr int kThreads = 384;
constexpr uint32_t kBStageBytes = kBN * kBK * 2;  // 16 KB fp16 tokens
constexpr uint32_t kWStageBytes = kBM * kBK;      // 8 KB int8 weights
constexpr size_t kSmemBytes = (size_t)kStages * (kBStageBytes + kWStageBytes) + 1024 /*barriers*/ + 1024 /*align*/;

struct alignas(64) Params {
    CUtensorMap tm_b;
    CUtensorMap tm_w0;
    CUtensorMap tm_w1;
    int64_t M, N, K;
    int64_t n_split;
    int64_t ld_out;
    void *out;
    const float *x_scale;
    const float *w_scale0;
    const float *w_scale1;
    const __nv_bfloat16 *bias;
    unsigned int *status;
    int w_layout;
    int epi;
};

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t afull[kAStages];
    uint64_t aempty[kAStages];
    uint64_t accfull[2];
    uint64_t accempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void tile_coords(int64_t t, int64_t m_tiles, int64_t *n0, int64_t *m0) {
    *n0 = (t / m_tiles) * kBM;
    *m0 = (t % m_tiles) * kBN;
}

// 4 int8 (one 32-bit word, k ascending) -> 2 words of fp16x2 pairs (k, k+1).
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t f = w ^ 0x80808080u;  // b + 128 as unsigned bytes
    const uint32_t p0 = __byte_perm(f, 0x64646464u, 0x4140);  // [b0+128, 0x64, b1+128, 0x64]
    const uint32_t p1 = __byte_perm(f, 0x64646464u, 0x4342);
    const __half2 off = __floats2half2_rn(1152.0f, 1152.0f);
    __half2 h0 = __hsub2(*reinterpret_cast<const __half2 *>(&p0), off);
    __half2 h1 = __hsub2(*reinterpret_cast<const __half2 *>(&p1), off);
    lo = *reinterpret_cast<uint32_t *>(&h0);
    hi = *reinterpret_cast<uint32_t *>(&h1);
}

__global__ void __launch_bounds__(kThreads, 1) i8gemm_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *bbuf = smem;
    uint8_t *wbuf = smem + kStages * kBStageBytes;
    Bars *bars = reinterpret_cast<Bars *>(wbuf + kStages * kWStageBytes);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t m_tiles = (p.M + kBN - 1) / kBN;
    const int64_t n_tiles = (p.N + kBM - 1) / kBM;
    const int64_t num_tiles = m_tiles * n_tiles;
    const int KT = (int)(p.K / kBK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1 + 4);
        }
        for (int a = 0; a < kAStages; ++a) {
            mbar_init(&bars->afull[a], 4);
            mbar_init(&bars->aempty[a], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->accfull[b], 1);
            mbar_init(&bars->accempty[b], 4);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_b);
        tma_prefetch_desc(&p.tm_w0);
        tma_prefetch_desc(&p.tm_w1);
    }
    if (warp == 1) tmem_alloc(&bars->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
                int64_t n0, m0;
                tile_coords(t, m_tiles, &n0, &m0);
                const bool src1 = n0 >= p.n_split;
                const CUtensorMap *tw = src1 ? &p.tm_w1 : &p.tm_w0;
                const int wrow = (int)(src1 ? n0 - p.n_split : n0);
                for (int kt = 0; kt < KT; ++kt) {
                    if (!mbar_wait(&bars->empty[stage], phase ^ 1, p.status, abort)) break;
                    mbar_arrive_expect_tx(&bars->full[stage], kBStageBytes + kWStageBytes);
                    if (p.w_layout == W_KMAJOR)
                        tma_load_2d(wbuf + stage * kWStageBytes, tw, &bars->full[stage], kt * kBK, wrow);
                    else
                        tma_load_2d(wbuf + stage * kWStageBytes, tw, &bars->full[stage], wrow, kt * kBK);
                    tma_load_2d(bbuf + stage * kBStageBytes, &p.tm_b, &bars->full[stage], kt * kBK, (int)m0);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBM, kBN, 0, 0, 0);
            int stage = 0, astage = 0;
            uint32_t phase = 0, aphase = 0;
            uint32_t chunk = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                uint32_t acc_col = kColAcc0;
                for (int kt = 0; kt < KT && ok; ++kt) {
                    const int cpos = kt % kChunkStages;
                    if (cpos == 0) {
                        const uint32_t ab = chunk & 1u;
                        ok = mbar_wait(&bars->accempty[ab], ((chunk >> 1) & 1u) ^ 1u, p.status, abort);
                        if (!ok) break;
                        acc_col = ab ? kColAcc1 : kColAcc0;
                    }
                    ok = mbar_wait(&bars->full[stage], phase, p.status, abort) &&
                         mbar_wait(&bars->afull[astage], aphase, p.status, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t b_base = smem_u32(bbuf + stage * kBStageBytes);
#pragma unroll
                    for (int k16 = 0; k16 < kBK / 16; ++k16) {
                        const uint64_t bdesc = smem_desc(b_base + k16 * 32, 16, 1024, kLayoutSw128);
                        mma_ts_f16(tmem + acc_col, tmem + kColA + astage * 32 + k16 * 8, bdesc, idesc,
                                   (cpos > 0 || k16 > 0) ? 1u : 0u);
                    }
                    tc_commit(&bars->empty[stage]);
                    tc_commit(&bars->aempty[astage]);
                    if (cpos == kChunkStages - 1 || kt == KT - 1) {
                        tc_commit(&bars->accfull[chunk & 1u]);
                        ++chunk;
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++astage == kAStages) {
                        astage = 0;
                        aphase ^= 1;
                    }
                }
            }
            // Let every issued MMA finish before the CTA can release TMEM.
            tc_commit(&bars->drain);
            mbar_wait(&bars->drain, 0, p.status, abort);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ int8 -> fp16 converters (A operand into TMEM)
        const int q = warp & 3;
        const int r = q * 32 + lane;  // TMEM lane = A row of the tile
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        int stage = 0, astage = 0;
        uint32_t phase = 0, aphase = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            for (int kt = 0; kt < KT; ++kt) {
                ok = mbar_wait(&bars->full[stage], phase, p.status, abort);
                if (!ok) break;
                uint32_t a[32];
                const uint8_t *ws = wbuf + stage * kWStageBytes;
                if (p.w_layout == W_KMAJOR) {
                    // Row r: 64 bytes, 64-byte swizzle (16-byte chunk c stored at c ^ ((r >> 1) & 3)).
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int pc = c ^ ((r >> 1) & 3);
                        const uint4 v = *reinterpret_cast<const uint4 *>(ws + r * 64 + pc * 16);
                        s8x4_to_f16x4(v.x, a[8 * c + 0], a[8 * c + 1]);
                        s8x4_to_f16x4(v.y, a[8 * c + 2], a[8 * c + 3]);
                        s8x4_to_f16x4(v.z, a[8 * c + 4], a[8 * c + 5]);
                        s8x4_to_f16x4(v.w, a[8 * c + 6], a[8 * c + 7]);
                    }
                } else {
                    // Tile [64 contraction rows][128 output columns], 128-byte swizzle:
                    // byte (n, r) at n*128 + 16*((r >> 4) ^ (n & 7)) + (r & 15).
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int n = 2 * j;
                        const uint32_t b0 = ws[n * 128 + 16 * ((r >> 4) ^ (n & 7)) + (r & 15)];
                        const uint32_t b1 = ws[(n + 1) * 128 + 16 * ((r >> 4) ^ ((n + 1) & 7)) + (r & 15)];
                        a[j] = s8pair_to_f16x2(b0 | (b1 << 16));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->empty[stage]);
                ok = mbar_wait(&bars->aempty[astage], aphase ^ 1, p.status, abort);
                if (!ok) break;
                tc_fence_after();
                tmem_st32(lane_addr + kColA + astage * 32, a);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->afull[astage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++astage == kAStages) {
                    astage = 0;
                    aphase ^= 1;
                }
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ epilogue: drain chunks, write outputs
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const int nchunks = (KT + kChunkStages - 1) / kChunkStages;
        uint32_t chunk = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int64_t n0, m0;
            tile_coords(t, m_tiles, &n0, &m0);
            const int64_t n = n0 + q * 32 + lane;  // output column owned by this thread
            const bool n_ok = n < p.N;
            float ws = 0.0f, bias = 0.0f;
            if (n_ok && p.epi == EPI_DEQUANT_BF16) {
                ws = n < p.n_split ? __ldg(p.w_scale0 + n) : __ldg(p.w_scale1 + (n - p.n_split));
                if (p.bias) bias = __bfloat162float(p.bias[n]);
            }
            for (int c = 0; c < nchunks; ++c) {
                const uint32_t ab = chunk & 1u;
                ok = mbar_wait(&bars->accfull[ab], (chunk >> 1) & 1u, p.status, abort);
                if (!ok) break;
                tc_fence_after();
                const bool last = (c == nchunks - 1);
                const uint32_t acc_col = ab ? kColAcc1 : kColAcc0;
#pragma unroll 1
                for (int j = 0; j < kBN / 32; ++j) {
                    uint32_t r[32], tot[32];
                    tmem_ld32(lane_addr + acc_col + 32 * j, r);
                    if (c > 0) tmem_ld32(lane_addr + kColTot + 32 * j, tot);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int32_t part = __float2int_rn(__uint_as_float(r[i]));
                        tot[i] = (uint32_t)((c > 0 ? (int32_t)tot[i] : 0) + part);
                    }
                    if (!last) {
                        tmem_st32(lane_addr + kColTot + 32 * j, tot);
                        continue;
                    }
                    // Final chunk: write the 32 token rows m0 + 32j + i of column n.
                    const int64_t mb = m0 + 32 * j;
                    float xs_l = 0.0f;
                    if (p.epi != EPI_ACC_I32 && mb + lane < p.M) xs_l = __ldg(p.x_scale + mb + lane);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float xs = __shfl_sync(0xffffffffu, xs_l, i);
                        const int64_t m = mb + i;
                        if (!n_ok || m >= p.M) continue;
                        const int32_t acc = (int32_t)tot[i];
                        if (p.epi == EPI_ACC_I32) {
                            reinterpret_cast<int32_t *>(p.out)[m * p.ld_out + n] = acc;
                        } else if (p.epi == EPI_DEQUANT_BF16) {
                            const float tv = __fmul_rn(__int2float_rn(acc), xs);
                            const float y = __fmaf_rn(tv, ws, bias);
                            reinterpret_cast<__nv_bfloat16 *>(p.out)[m * p.ld_out + n] = __float2bfloat16_rn(y);
                        } else {
                            reinterpret_cast<float *>(p.out)[m * p.ld_out + n] = __fmul_rn(__int2float_rn(acc), xs);
                        }
                    }
                }
                if (!last) tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->accempty[ab]);
                ++chunk;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int launch_i8gemm(const I8GemmProblem &q, cudaStream_t st) {
    Params p;  // host staging; copied into the launch's parameter buffer
    memset(&p, 0, sizeof(p));
    int rc;
    // Activations: fp16 [M][K], box 64 x 128, 128-byte swizzle.
    rc = encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.b_f16, (uint64_t)q.K, (uint64_t)q.M,
                        (uint64_t)q.K * 2, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    for (int s = 0; s < 2; ++s) {
        const int8_t *w = s ? q.w1 : q.w0;
        const int64_t rows = s ? q.w_rows_total1 : q.w_rows_total0;
        CUtensorMap *tm = s ? &p.tm_w1 : &p.tm_w0;
        if (q.w_layout == W_KMAJOR)  // [rows][K], box 64 B x 128 rows, 64-byte swizzle
            rc = encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)q.K, (uint64_t)rows,
                                (uint64_t)q.ld_w, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_64B);
        else  // [K rows][ld_w]: box 128 B (output columns) x 64 rows, 128-byte swizzle
            rc = encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)q.N, (uint64_t)rows,
                                (uint64_t)q.ld_w, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
    }
    p.M = q.M;
    p.N = q.N;
    p.K = q.K;
    p.n_split = q.n_split;
    p.ld_out = q.ld_out;
    p.out = q.out;
    p.x_scale = q.x_scale;
    p.w_scale0 = q.w_scale0;
    p.w_scale1 = q.w_scale1;
    p.bias = reinterpret_cast<const __nv_bfloat16 *>(q.bias);
    p.status = q.status;
    p.w_layout = q.w_layout;
    p.epi = q.epi;

    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(i8gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
        attr = true;
    }
    const int64_t tiles = ((q.M + kBN - 1) / kBN) * ((q.N + kBM - 1) / kBM);
    const int grid = (int)(tiles < q.num_sms ? tiles : q.num_sms);
    prof_begin(1, st);
    i8gemm_kernel<<<grid, kThreads, kSmemBytes, st>>>(p);
    prof_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
    return GBQ_OK;
}

}  // namespace gbq
