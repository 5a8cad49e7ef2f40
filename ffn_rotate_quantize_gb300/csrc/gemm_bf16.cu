// gemm_bf16.cu -- bf16 tensor-core GEMMs with fp32 accumulation:
//
//   linear_dx   ("The backward: dL/dx, weight-only" on the PyPI page "xpu-kernels 0.2.0"):
//               dx[M][K] = dy[M][N] @ W[N][K]  (B operand MN-major: the contraction runs along W's rows)
//   linear_bf16 (the rotate-only BF16 path of "Use from C" on the same page):
//               y[M][N] = x[M][K] @ W[N][K]^T + bias[N]  (B operand K-major)
//
// Both are one kernel template; below, "red" is the contraction length and "cols" the number of
// output columns (linear_dx: red = N, cols = K; linear_bf16: red = K, cols = N).
//
// Design: tcgen05 kind::f16 with both operands in shared memory.  A = the left operand's tile
// (128 rows, K-major, 128-byte swizzle).  B = 256 output columns: MN-major as four TMA boxes of
// 64 columns x 64 rows (LBO = 8 KB between 64-column blocks, SBO = 1 KB between 8-row groups), or
// K-major as one box of 64 x 256 rows laid out like A.  Tile 128 x 256 x 64 per stage, 4 stages,
// accumulators double-buffered in TMEM (2 x 256 columns) so the epilogue of one tile overlaps the
// main loop of the next.  One persistent CTA per SM.  Warps: 0, 2, 3, 8 TMA producers (one per
// stage: TMA loads issued by one thread are processed one stage at a time), 1 TMEM owner + MMA
// issuer, 4-7 epilogue (fp32 -> + bias -> bf16).
#include "common.cuh"
#include "gemm.h"

namespace gbq {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 288;
constexpr int kProducers = 4;  // warps 0, 2, 3, 8
static_assert(kStages % kProducers == 0, "each producer owns whole stages");

__device__ __forceinline__ int producer_id(int warp) {
    if (warp == 0) return 0;
    if (warp == 2 || warp == 3) return warp - 1;
    if (warp == 8) return 3;
    return -1;
}
constexpr uint32_t kAStage = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBStage = kBN * kBK * 2;  // 32 KB
constexpr size_t kSmem = (size_t)kStages * (kAStage + kBStage) + 1024 + 1024;

struct Params {
    CUtensorMap tm_a;  // left operand [M][red] bf16, box {64, 128}
    CUtensorMap tm_b;  // MN-major: W [red][cols], box {64 (cols), 64 (red)}; K-major: W [cols][red], box {64, 256}
    int64_t M, red, cols;
    __nv_bfloat16 *out;                // [M][cols]
    const __nv_bfloat16 *bias;         // [cols] or nullptr
    unsigned int *status;
};

struct Bars {
    uint64_t full[kStages], empty[kStages], accfull[2], accempty[2], drain;
    uint32_t tmem_base;
    int abort;
};

template <bool B_KMAJOR>
__global__ void __launch_bounds__(kThreads, 1) bf16_gemm_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *abuf = smem;
    uint8_t *bbuf = smem + kStages * kAStage;
    Bars *bars = reinterpret_cast<Bars *>(bbuf + kStages * kBStage);
    volatile int *abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m_tiles = (p.M + kBM - 1) / kBM;
    const int64_t n_tiles = (p.cols + kBN - 1) / kBN;
    const int64_t num_tiles = m_tiles * n_tiles;
    const int KT = (int)(p.red / kBK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->accfull[b], 1);
            mbar_init(&bars->accempty[b], 4);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_a);
        tma_prefetch_desc(&p.tm_b);
    }
    if (warp == 1) tmem_alloc(&bars->tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (producer_id(warp) >= 0) {
        const uint32_t pid = (uint32_t)producer_id(warp);
        if (lane == 0) {
            uint32_t gs = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int m0 = (int)((t % m_tiles) * kBM);
                const int k0 = (int)((t / m_tiles) * kBN);
                for (int kt = 0; kt < KT; ++kt) {
                    const uint32_t my = gs++;
                    if (my % kProducers != pid) continue;
                    const int stage = (int)(my % kStages);
                    ok = mbar_wait(&bars->empty[stage], ((my / kStages) & 1u) ^ 1u, p.status, abort);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bars->full[stage], kAStage + kBStage);
                    tma_load_2d(abuf + stage * kAStage, &p.tm_a, &bars->full[stage], kt * kBK, m0);
                    if (B_KMAJOR) {
                        tma_load_2d(bbuf + stage * kBStage, &p.tm_b, &bars->full[stage], kt * kBK, k0);
                    } else {
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j)
                            tma_load_2d(bbuf + stage * kBStage + j * 8192, &p.tm_b, &bars->full[stage], k0 + 64 * j,
                                        kt * kBK);
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBM, kBN, 1, 0, B_KMAJOR ? 0 : 1);
            int stage = 0;
            uint32_t phase = 0, tcount = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tcount) {
                const uint32_t ab = tcount & 1u;
                ok = mbar_wait(&bars->accempty[ab], ((tcount >> 1) & 1u) ^ 1u, p.status, abort);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + ab * 256;
                for (int kt = 0; kt < KT; ++kt) {
                    ok = mbar_wait(&bars->full[stage], phase, p.status, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(abuf + stage * kAStage);
                    const uint32_t b0 = smem_u32(bbuf + stage * kBStage);
#pragma unroll
                    for (int k16 = 0; k16 < kBK / 16; ++k16) {
                        const uint64_t ad = smem_desc(a0 + k16 * 32, 16, 1024, kLayoutSw128);
                        const uint64_t bd = B_KMAJOR ? smem_desc(b0 + k16 * 32, 16, 1024, kLayoutSw128)
                                                     : smem_desc(b0 + k16 * 2048, 8192, 1024, kLayoutSw128);
                        mma_ss_f16(d, ad, bd, idesc, (kt > 0 || k16 > 0) ? 1u : 0u);
                    }
                    tc_commit(&bars->empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) tc_commit(&bars->accfull[ab]);
            }
            tc_commit(&bars->drain);
            mbar_wait(&bars->drain, 0, p.status, abort);
        }
    } else if (warp >= 4 && warp < 8) {
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t tcount = 0;
        for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tcount) {
            const int64_t m0 = (t % m_tiles) * kBM;
            const int64_t k0 = (t / m_tiles) * kBN;
            const uint32_t ab = tcount & 1u;
            if (!mbar_wait(&bars->accfull[ab], (tcount >> 1) & 1u, p.status, abort)) break;
            tc_fence_after();
            const int64_t m = m0 + q * 32 + lane;
#pragma unroll 1
            for (int j = 0; j < kBN / 32; ++j) {
                uint32_t r[32];
                tmem_ld32(lane_addr + ab * 256 + 32 * j, r);
                tc_wait_ld();
                const int64_t kb = k0 + 32 * j;
                if (m < p.M && kb < p.cols &&
                    GBQ_IN_RANGE(p.status, m * p.cols + kb, min((int64_t)32, p.cols - kb), p.M * p.cols)) {
                    if (p.bias) {  // the same 32 values for every lane: broadcast loads
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (kb + i < p.cols)
                                r[i] = __float_as_uint(__fadd_rn(__uint_as_float(r[i]), __bfloat162float(p.bias[kb + i])));
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                        w[i] = *reinterpret_cast<uint32_t *>(&h);
                    }
                    __nv_bfloat16 *row = p.out + m * p.cols + kb;
                    if (kb + 32 <= p.cols && p.cols % 8 == 0) {  // 16-byte aligned row segments
                        uint4 *dst = reinterpret_cast<uint4 *>(row);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    } else {
                        const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(w);
                        for (int i = 0; i < 32 && kb + i < p.cols; ++i) row[i] = h[i];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->accempty[ab]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool B_KMAJOR>
int launch_bf16_gemm(Params &p, cudaStream_t st, int num_sms) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(bf16_gemm_kernel<B_KMAJOR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmem);
        if (e != cudaSuccess) return gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
        attr = true;
    }
    const int64_t tiles = ((p.M + kBM - 1) / kBM) * ((p.cols + kBN - 1) / kBN);
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    prof_begin(2, st);
    bf16_gemm_kernel<B_KMAJOR><<<grid, kThreads, kSmem, st>>>(p);
    prof_end(st);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GBQ_OK : gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
}

}  // namespace

int launch_bf16_gemm_nn(const void *dy, const void *w, void *dx, int64_t M, int64_t N, int64_t K,
                        unsigned int *status, int num_sms, cudaStream_t st) {
    Params p;
    memset(&p, 0, sizeof(p));
    int rc = encode_tmap_2d(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2,
                            kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64,
                        kBK, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    p.M = M;
    p.red = N;
    p.cols = K;
    p.out = reinterpret_cast<__nv_bfloat16 *>(dx);
    p.bias = nullptr;
    p.status = status;
    return launch_bf16_gemm<false>(p, st, num_sms);
}

int launch_bf16_gemm_tn(const void *x, const void *w, const void *bias, void *y, int64_t M, int64_t N, int64_t K,
                        unsigned int *status, int num_sms, cudaStream_t st) {
    Params p;
    memset(&p, 0, sizeof(p));
    int rc = encode_tmap_2d(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2,
                            kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, kBK,
                        kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    p.M = M;
    p.red = K;
    p.cols = N;
    p.out = reinterpret_cast<__nv_bfloat16 *>(y);
    p.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
    p.status = status;
    return launch_bf16_gemm<true>(p, st, num_sms);
}

}  // namespace gbq
