// gemv.cu -- decode and small-batch path (M <= 16): y = dequant(quantize(R x) @ W8^T), weight streaming.
//
// What it computes: the rotated-INT8 linear layer of the PyPI page
// "xpu-kernels 0.2.0" ("Use from Python": linear), for a handful of tokens,
// where the cost is reading the int8 weight once from HBM.
//
// Design: one CTA per SM, each owning a contiguous slice of weight rows.  At
// entry one thread issues bulk copies (cp.async.bulk, mbarrier-tracked) of the
// slice into a shared-memory ring, so the HBM stream starts before any
// arithmetic.  Four kernels share that structure:
//   gemv_direct_kernel  n = 64, K = 4096, one or two tokens: the register-streaming
//                       variant, consecutive calls overlapping (described below);
//   gemv_kernel         other square shapes, one or two tokens: while the bytes
//                       are in flight the CTA rotates and quantizes x with the
//                       same core (and fp32 operation order) as the standalone
//                       rotate+quantize kernel, so its codes are bit-identical to
//                       gbq_quantize_act;
//   gemv_gen_kernel     one or two tokens, any descriptor: as gemv_kernel, with
//                       the generic rotation's passes (rotate_g.cuh) inside;
//   gemv_codes_kernel   up to 16 tokens, any descriptor: the codes and scales
//                       come from the rotation kernels (launched before it).
// The ring kernels' dot phase: each warp takes its share of the K columns of
// every staged weight row, does 16-byte shared loads and int8 dp4a dot products
// against the quantized x, the partial sums are reduced across lanes and warps,
// and the dequant epilogue runs (fp32(acc) * x_scale, fmaf with the row scale
// and bias, bf16).
#include <algorithm>

#include "gemm.h"
#include "rotate_fast.cuh"
#include "rotate_g.cuh"

namespace gbq {
namespace {

constexpr int kGvThreads = 256;
constexpr int kGvStages = 4;
constexpr int kGvMaxM = 4;
constexpr size_t kGvSmem = 220 * 1024;

struct GemvArgs {
    const void *x;
    const int8_t *w8;
    const float *ws;
    // Ring kernels: rows [n_split, N) of the weight come from w8b / wsb (row n - n_split); n_split = N
    // for one weight tensor.
    const int8_t *w8b;
    const float *wsb;
    int64_t n_split;
    const __nv_bfloat16 *bias;
    __nv_bfloat16 *y;
    int64_t M, N, K;
    int64_t ld_y;           // elements between token rows of y (ring kernels)
    int G;
    int rows_per_cta;
    int rows_per_stage;
    int nstages;            // ring kernels: stages in use (3 or kGvStages)
    uint32_t stage_bytes;   // rows_per_stage * K, multiple of 128
    uint32_t x_off, t_off, misc_off;
    uint32_t xb_off;        // bf16 staging of the M token rows (three-pass n = 64 path), else 0
    uint32_t wrow_off;      // register-streaming kernel: staging of slice rows 16.. (0: rows 16.. via registers)
    uint32_t ep_off;        // ring kernels: epilogue operands of the slice (gv_ep_bytes)
    unsigned int *status;
};

constexpr int kGvWarps = kGvThreads / 32;
constexpr int kGcMaxM = 16;  // tokens of the codes GEMV (the kernels that rotate in-kernel take kGvMaxM)
constexpr int kGvGenMaxM = 2;  // tokens of the GEMV with the generic rotation inside

// Tokens padded to a power of two; the dot phase keeps up to NV / MP rows of a stage in flight per lane
// (NV partial sums per lane: kGvNV for the kernels that rotate in-kernel, kGcNV for the codes GEMV).
__host__ __device__ constexpr int gv_pad_m(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }
constexpr int kGvNV = 32;
constexpr int kGcNV = 64;
// The ring kernels' misc block (token scales, amax slots, stage barriers, abort flag, token barrier)
// fits in the 128 bytes before the epilogue operands.
static_assert(2 * kGvMaxM * 4 + (kGvStages + 2) * 8 + 16 <= 128, "misc block exceeds 128 bytes");

// Shared memory of the ring kernels' epilogue operands: w_scale and bias (as fp32) of the CTA's rows,
// then the warps' partial sums of two consecutive stages (nv per warp and stage).
__host__ __device__ constexpr size_t gv_ep_bytes(int64_t rows_per_cta, int nv) {
    return ((size_t)rows_per_cta * 8 + 2 * kGvWarps * (size_t)nv * 4 + 127) & ~(size_t)127;
}

// The slice's w_scale and bias into shared memory (read before the dot products need them; the first
// stage's barrier, at the latest, publishes them).
__device__ __forceinline__ void gv_load_epilogue(const GemvArgs &p, float *ep, int64_t r0, int nrows) {
    for (int t = threadIdx.x; t < nrows; t += kGvThreads) {
        const int64_t n = r0 + t;
        ep[t] = n < p.n_split ? __ldg(p.ws + n) : __ldg(p.wsb + (n - p.n_split));
        ep[p.rows_per_cta + t] = p.bias ? __bfloat162float(p.bias[n]) : 0.0f;
    }
}

// Bulk copy of weight rows [r, r + rows) into dst (contiguous, K bytes a row), completing on bar; the
// rows may straddle the split between the two weight tensors.
__device__ __forceinline__ void gv_copy_rows(const GemvArgs &p, uint8_t *dst, int64_t r, int rows, uint64_t *bar) {
    const int64_t lo = r < p.n_split ? min((int64_t)rows, p.n_split - r) : 0;  // rows from w8
    if (lo > 0) bulk_g2s(dst, p.w8 + r * p.K, (uint32_t)(lo * p.K), bar);
    if (lo < rows)
        bulk_g2s(dst + lo * p.K, p.w8b + (r + lo - p.n_split) * p.K, (uint32_t)((rows - lo) * p.K), bar);
}

// 16-byte load from shared memory at a shared-window address (a .shared access, whatever the
// compiler can prove about the generic pointer it came from).  The memory clobber keeps it after the
// barriers and plain stores that publish what it reads.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Dot products of the staged weight slice against the quantized tokens xq (row
// stride K) and the dequant epilogue; every thread of the CTA takes part.  Warp w
// owns the same 1/8 of the K columns (16-byte groups) in every stage: per group it
// reads the tokens' codes once and the group of each of the stage's rows (at most
// PS / MP rows, MP = the token count padded to a power of two), so each weight
// byte is read from shared memory once, with independent dp4a chains per row and
// token.  A transposing shuffle reduction leaves every lane of every warp with
// NV / 32 of the warp's sums (NV >= 32) or every NV-th lane group with one; the
// eight warps' partial sums are added after the stage's barrier (exact integers:
// the order does not matter) by NV threads, which run the epilogue while the other
// warps go on with the next stage.  One CTA barrier per stage: it also carries the
// vote on the stage wait, and the partial sums alternate between two buffers, so a
// stage's sums are never overwritten before its epilogue has read them.  w_scale
// and bias come from shared memory (gv_load_epilogue).
template <int MP, int RB, int PS>  // tokens and rows per stage padded to powers of two; PS >= MP * RB slots
__device__ __forceinline__ void gemv_dot_phase_t(const GemvArgs &p, uint8_t *stages, const int8_t *xq,
                                                 const float *xs_s, uint64_t *full, int *abort_flag, int64_t r0,
                                                 int nrows, int nchunks, float *ep) {
    constexpr int NV = MP * RB;  // partial sums per lane before the reduction
    static_assert(NV >= 2 && NV <= PS && PS <= 64, "2..64 partial sums per lane");
    constexpr int VPL = NV > 32 ? NV / 32 : 1;            // sums a lane holds after the transposing levels
    constexpr int LANES_PER_V = NV < 32 ? 32 / NV : 1;     // lanes that end up holding one value's total
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const float *ep_ws = ep;
    const float *ep_b = ep + p.rows_per_cta;
    int *part_base = reinterpret_cast<int *>(ep + 2 * p.rows_per_cta);  // [2][kGvWarps][PS]
    auto issue = [&](int c) {
        const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
        const uint32_t bytes = (uint32_t)rows * (uint32_t)p.K;
        uint64_t *bar = &full[c % p.nstages];
        mbar_arrive_expect_tx(bar, bytes);
        gv_copy_rows(p, stages + (size_t)(c % p.nstages) * p.stage_bytes, r0 + (int64_t)c * p.rows_per_stage, rows,
                     bar);
    };
    const int kq = (int)(p.K / 16);
    const int cpw = (kq + kGvWarps - 1) / kGvWarps;  // 16-byte groups per warp
    const int i0 = warp * cpw + lane, i1 = min(kq, (warp + 1) * cpw);
    const uint32_t xq_s = smem_u32(xq), kb = (uint32_t)p.K;
    for (int c = 0; c < nchunks; ++c) {
        const bool ok = mbar_wait(&full[c % p.nstages], (uint32_t)((c / p.nstages) & 1), p.status, abort_flag);
        const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
        const uint32_t st_s = smem_u32(stages + (size_t)(c % p.nstages) * p.stage_bytes);
        int acc[NV];  // [row j][token m] at j * MP + m
#pragma unroll
        for (int q = 0; q < NV; ++q) acc[q] = 0;
        for (int i = ok ? i0 : i1; i < i1; i += 32) {  // a stage whose wait gave up is not read
            uint4 xv[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m)
                xv[m] = m < p.M ? lds128(xq_s + (uint32_t)m * kb + 16u * (uint32_t)i) : make_uint4(0, 0, 0, 0);
            // Rows in groups of up to eight: the group's loads first (independent, in flight together),
            // then its dot products; rows past the stage's end read as zero and add nothing.
            constexpr int GR = RB < 8 ? RB : 8;
#pragma unroll
            for (int jg = 0; jg < RB; jg += GR) {
                uint4 w[GR];
#pragma unroll
                for (int jj = 0; jj < GR; ++jj)
                    w[jj] = jg + jj < rows ? lds128(st_s + (uint32_t)(jg + jj) * kb + 16u * (uint32_t)i)
                                           : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int jj = 0; jj < GR; ++jj) {
#pragma unroll
                    for (int m = 0; m < MP; ++m) {
                        int a = acc[(jg + jj) * MP + m];
                        a = __dp4a((int)w[jj].x, (int)xv[m].x, a);
                        a = __dp4a((int)w[jj].y, (int)xv[m].y, a);
                        a = __dp4a((int)w[jj].z, (int)xv[m].z, a);
                        a = __dp4a((int)w[jj].w, (int)xv[m].w, a);
                        acc[(jg + jj) * MP + m] = a;
                    }
                }
            }
        }
        // Transposing reduction over the lanes: at each level (lane bits 4, 3, ...) a lane keeps the half
        // of its values selected by its lane bit and adds the partner's copy of that half, until VPL values
        // are left (lane l then holds values VPL l .. VPL l + VPL - 1); below 32 values, plain butterflies
        // over the remaining lane bits, after which lane l holds the total of value l / LANES_PER_V.
#pragma unroll
        for (int o = 16, n = NV; n > VPL; o >>= 1, n >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int q = 0; q < n / 2; ++q) {
                const int send = up ? acc[q] : acc[q + n / 2];
                const int keep = up ? acc[q + n / 2] : acc[q];
                acc[q] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
#pragma unroll
        for (int o = LANES_PER_V / 2; o >= 1; o >>= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
        int *part = part_base + (c & 1) * (kGvWarps * PS);
        if constexpr (VPL > 1) {
#pragma unroll
            for (int t = 0; t < VPL; ++t) part[warp * PS + VPL * lane + t] = acc[t];
        } else {
            if (lane % LANES_PER_V == 0) part[warp * PS + lane / LANES_PER_V] = acc[0];
        }
        if (!__syncthreads_and(ok)) break;  // every thread leaves together; the stage and its sums are complete
        if (tid < NV) {
            const int j = tid / MP, m = tid % MP;
            if (j < rows && m < p.M) {
                int a = 0;
#pragma unroll
                for (int w = 0; w < kGvWarps; ++w) a += part[w * PS + tid];
                const int jr = c * p.rows_per_stage + j;  // row within the slice
                const int64_t n = r0 + jr;
                const float tv = __fmul_rn(__int2float_rn(a), xs_s[m]);
                if (GBQ_IN_RANGE(p.status, (int64_t)m * p.ld_y + n, 1, (p.M - 1) * p.ld_y + p.N))
                    p.y[(int64_t)m * p.ld_y + n] = __float2bfloat16_rn(__fmaf_rn(tv, ep_ws[jr], ep_b[jr]));
            }
        }
        if (tid == 0 && c + p.nstages < nchunks) issue(c + p.nstages);  // every warp has read stage c
    }
}

// Rows per stage padded to a power of two, capped at PS / MP (with at least two partial sums per lane).
template <int MP, int PS, int WANT>
constexpr int gv_rb() {
    return WANT * MP <= PS ? WANT : (PS / MP >= 1 ? PS / MP : 1);
}

// The dot phase for the launch's token count and rows per stage (PS: partial-sum slots per warp).
template <int MP, int PS>
__device__ __forceinline__ void gemv_dot_phase_m(const GemvArgs &p, uint8_t *stages, const int8_t *xq,
                                                 const float *xs_s, uint64_t *full, int *abort_flag, int64_t r0,
                                                 int nrows, int nchunks, float *ep) {
    const int rb = p.rows_per_stage;  // <= PS / MP (gv_plan_ring)
    if (rb <= 2 || MP * 4 > PS)
        gemv_dot_phase_t<MP, gv_rb<MP, PS, 2>(), PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    else if (rb <= 4 || MP * 8 > PS)
        gemv_dot_phase_t<MP, gv_rb<MP, PS, 4>(), PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    else if (rb <= 8 || MP * 16 > PS)
        gemv_dot_phase_t<MP, gv_rb<MP, PS, 8>(), PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    else if (rb <= 16 || MP * 32 > PS)
        gemv_dot_phase_t<MP, gv_rb<MP, PS, 16>(), PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    else if (rb <= 32 || MP * 64 > PS)
        gemv_dot_phase_t<MP, gv_rb<MP, PS, 32>(), PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    else
        gemv_dot_phase_t<MP, gv_rb<MP, PS, 64>(), PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
}

template <int MAXM, int PS>
__device__ __forceinline__ void gemv_dot_phase(const GemvArgs &p, uint8_t *stages, const int8_t *xq,
                                               const float *xs_s, uint64_t *full, int *abort_flag, int64_t r0,
                                               int nrows, int nchunks, float *ep) {
    switch (gv_pad_m(p.M)) {
        case 1: gemv_dot_phase_m<1, PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep); break;
        case 2: gemv_dot_phase_m<2, PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep); break;
        case 4:
            if constexpr (MAXM >= 4) gemv_dot_phase_m<4, PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
            break;
        default:
            if constexpr (MAXM > 4) {
                if (gv_pad_m(p.M) == 8)
                    gemv_dot_phase_m<8, PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
                else
                    gemv_dot_phase_m<16, PS>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
            }
            break;
    }
}

template <int LOGN>
__global__ void __launch_bounds__(kGvThreads, 1) gemv_kernel(GemvArgs p) {
    using Geo = RotGeom<LOGN>;
    constexpr int NP = Geo::NP, TPG = Geo::TPG;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    int8_t *xq = reinterpret_cast<int8_t *>(smem + p.x_off);
    float2 *T = reinterpret_cast<float2 *>(smem + p.t_off);
    float *xs_s = reinterpret_cast<float *>(smem + p.misc_off);
    unsigned *amax_s = reinterpret_cast<unsigned *>(xs_s + kGvMaxM);
    uint64_t *full = reinterpret_cast<uint64_t *>(amax_s + kGvMaxM);
    int *abort_flag = reinterpret_cast<int *>(full + kGvStages);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t r0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int64_t r1 = min(p.N, r0 + p.rows_per_cta);
    const int nrows = (int)(r1 - r0);
    // Debug builds: the CTA's weight slice (every weight copy below) lies inside W8.
    if (!GBQ_IN_RANGE(p.status, r0 * p.K, (int64_t)nrows * p.K, p.N * p.K)) return;
    const int nchunks = (nrows + p.rows_per_stage - 1) / p.rows_per_stage;

    if (tid == 0) {
        for (int s = 0; s < kGvStages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (tid < kGvMaxM) amax_s[tid] = 0u;
    __syncthreads();
    auto issue = [&](int c) {
        const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
        const uint32_t bytes = (uint32_t)rows * (uint32_t)p.K;
        uint64_t *bar = &full[c % p.nstages];
        mbar_arrive_expect_tx(bar, bytes);
        gv_copy_rows(p, stages + (size_t)(c % p.nstages) * p.stage_bytes, r0 + (int64_t)c * p.rows_per_stage, rows,
                     bar);
    };
    const bool fast_x = (LOGN == 6 && p.G == 1);
    uint64_t *xfull = full + kGvStages + 1;  // after the abort flag's slot
    if (fast_x) {
        // The tokens first (the rotation waits on them), then the weight slice, its copies spread
        // over the eight warps (one row each, round robin) so that many are in flight at once.
        if (tid == 0) {
            mbar_init(xfull, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(xfull, (uint32_t)(p.M * p.K * 2));
            bulk_g2s(smem + p.xb_off, p.x, (uint32_t)(p.M * p.K * 2), xfull);
            for (int c = 0; c < nchunks && c < p.nstages; ++c) {
                const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
                mbar_arrive_expect_tx(&full[c], (uint32_t)rows * (uint32_t)p.K);
            }
        }
        __syncthreads();
        if (lane == 0)
            for (int c = 0; c < nchunks && c < p.nstages; ++c) {
                const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
                for (int j = warp; j < rows; j += kGvThreads / 32)
                    gv_copy_rows(p, stages + (size_t)c * p.stage_bytes + (size_t)j * p.K,
                                 r0 + (int64_t)c * p.rows_per_stage + j, 1, &full[c]);
            }
    } else if (tid == 0) {
        for (int c = 0; c < nchunks && c < p.nstages; ++c) issue(c);
    }
    float *ep = reinterpret_cast<float *>(smem + p.ep_off);
    gv_load_epilogue(p, ep, r0, nrows);

    if constexpr (LOGN == 6) {
        if (p.G == 1) {
            // ---- rotate + quantize x: the three-pass n = 64 row transform on threads 0..127
            // (the same operations as the standalone kernel), one token row at a time ----
            if (tid < 128) {
                float *wmax = reinterpret_cast<float *>(amax_s);  // 4 slots (one per warp of the 128)
                auto bar = [] { named_bar_sync(1, 128); };
                RotArgs ra{};
                const bool ok = named_bar_and(1, 128, mbar_wait(xfull, 0, p.status, abort_flag));
                for (int m = 0; m < p.M && ok; ++m) {
                    const uint8_t *xb = smem + p.xb_off + (size_t)m * p.K * 2;
                    float2 v[16];
                    rot64_row<IN_BF16>(ra, xb, xb, 0.0f, T, tid, bar, [] {}, v);
                    float mx = pairs_amax(v);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0) wmax[warp] = mx;
                    bar();
                    const float amax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
                    const float s = __fdiv_rn(amax, 127.0f);
                    if (tid == 0) xs_s[m] = s;
                    uint32_t words[2][4];
                    quant_codes<16>(v, s, words);
                    const int r = tid >> 2, jq = tid & 3;
                    store_codes<OUT_S8, 4>(xq, (int64_t)m * p.K + 128 * r + 16 * jq, words[0]);
                    store_codes<OUT_S8, 4>(xq, (int64_t)m * p.K + 128 * r + 64 + 16 * jq, words[1]);
                    bar();  // the tile, the staging row and the amax slots are free for the next token
                }
            }
            __syncthreads();
            gemv_dot_phase<kGvMaxM, kGvNV>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
            if (tid == 0 && *(volatile int *)abort_flag) {
                // A wait gave up: let the copies issued at entry land (bounded) before the CTA leaves.
                for (int c = 0; c <= min(nchunks, p.nstages); ++c) {
                    uint64_t *b = c < min(nchunks, p.nstages) ? &full[c] : xfull;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(b, 0) && globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
            return;
        }
    }
    // ---- rotate + quantize x (the same core and operation order as rotq_kernel) ----
    const int row_threads = p.G * TPG;
    const bool in_row = tid < row_threads;
    const int g = in_row ? tid / TPG : 0;
    const int t = in_row ? tid - g * TPG : 0;
    RotArgs ra{};
    ra.in0 = p.x;
    ra.ld_in = p.K;
    for (int m = 0; m < p.M; ++m) {
        float2 v[NP];
        rot_group_core<LOGN, IN_BF16>(ra, m, in_row, g, t, T + (size_t)g * Geo::TILE, v);
        float mx = 0.0f;
#pragma unroll
        for (int j = 0; j < NP; ++j) mx = fmaxf(mx, pair_max_abs(v[j]));
        constexpr int W = TPG < 32 ? TPG : 32;
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (in_row && (t & (W - 1)) == 0) atomicMax(&amax_s[m], __float_as_uint(mx));
        __syncthreads();
        const float s = __fdiv_rn(__uint_as_float(amax_s[m]), 127.0f);
        if (tid == 0) xs_s[m] = s;
        if (in_row) {
            uint32_t words[2][NP / 4];
            quant_codes<NP>(v, s, words);
#pragma unroll
            for (int h = 0; h < 2; ++h) store_codes<OUT_S8, NP / 4>(xq, (int64_t)m * p.K + out_offset<LOGN>(g, t, h),
                                                                   words[h]);
        }
        __syncthreads();
    }

    gemv_dot_phase<kGvMaxM, kGvNV>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
}

// ---------------------------------------------------------------------------
// Decode GEMV over tokens already rotated and quantized (the codes and row scales the rotation kernels
// wrote into the workspace): for every descriptor the in-kernel rotations above do not cover.  Launched
// with programmatic stream serialization right after the quantizer: the first weight stages are
// bulk-copied at entry, while the quantizer may still run (it writes only the codes and scales); the
// codes and scales are read after griddepcontrol.wait; then the dot phase of gemv_kernel.
__global__ void __launch_bounds__(kGvThreads, 1) gemv_codes_kernel(GemvArgs p, const int8_t *codes,
                                                                   const float *scales) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    int8_t *xq = reinterpret_cast<int8_t *>(smem + p.x_off);
    // misc block: token scales [kGcMaxM], stage barriers, codes barrier, abort flag (108 bytes)
    static_assert(kGcMaxM * 4 + (kGvStages + 1) * 8 + 4 <= 128, "misc block exceeds 128 bytes");
    float *xs_s = reinterpret_cast<float *>(smem + p.misc_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(xs_s + kGcMaxM);
    uint64_t *xfull = full + kGvStages;
    int *abort_flag = reinterpret_cast<int *>(xfull + 1);

    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int nrows = (int)(min(p.N, r0 + p.rows_per_cta) - r0);
    // Debug builds: the CTA's weight slice (every weight copy below) lies inside W8.
    if (!GBQ_IN_RANGE(p.status, r0 * p.K, (int64_t)nrows * p.K, p.N * p.K)) return;
    const int nchunks = (nrows + p.rows_per_stage - 1) / p.rows_per_stage;
    if (tid == 0) {
        for (int s2 = 0; s2 < kGvStages; ++s2) mbar_init(&full[s2], 1);
        mbar_init(xfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int c = 0; c < nchunks && c < p.nstages; ++c) {
            const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
            const uint32_t bytes = (uint32_t)rows * (uint32_t)p.K;
            mbar_arrive_expect_tx(&full[c], bytes);
            gv_copy_rows(p, stages + (size_t)c * p.stage_bytes, r0 + (int64_t)c * p.rows_per_stage, rows, &full[c]);
        }
    }
    float *ep = reinterpret_cast<float *>(smem + p.ep_off);
    gv_load_epilogue(p, ep, r0, nrows);  // w_scale and bias: not written by the quantizer
    pdl_wait();  // the codes and scales come from the kernel before
    if (tid == 0) {
        mbar_arrive_expect_tx(xfull, (uint32_t)(p.M * p.K));
        bulk_g2s(xq, codes, (uint32_t)(p.M * p.K), xfull);
    }
    if (tid < p.M) xs_s[tid] = scales[tid];
    __syncthreads();  // barriers initialised, scales in place
    const bool xok = mbar_wait(xfull, 0, p.status, abort_flag);
    if (__syncthreads_and(xok)) gemv_dot_phase<kGcMaxM, kGcNV>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    if (tid == 0 && *(volatile int *)abort_flag) {
        // A wait gave up: let the copies issued at entry land (bounded) before the CTA leaves.
        for (int c = 0; c <= min(nchunks, p.nstages); ++c) {
            uint64_t *b = c < min(nchunks, p.nstages) ? &full[c] : xfull;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(b, 0) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Register-streaming variant for K = 4096, n = 64, one group, and at most 32
// weight rows per CTA (4 per warp), launched with programmatic stream
// serialization so that consecutive decode calls overlap:
//   entry: every thread asks L2 for its share of the CTA's weight slice
//     (prefetch.global.L2: a hint that moves no data into the thread, so it is
//     safe on memory the kernel before may still write), then lets the next
//     launch start and waits (griddepcontrol.wait) for the kernel before it;
//     every read of an input comes after that wait.
//   The kernel holds at most 128 registers per thread, so the next call's CTA
//   fits beside this one on the SM: its L2 prefetch streams the next layer's
//   weight from HBM while this layer computes.
//   body: the x rows are bulk-copied and rotated + quantized by threads 0..127
//     (the three-pass n = 64 transform, bit-identical codes to
//     gbq_quantize_act) while every warp loads its first two weight rows into
//     registers and one bulk copy brings the slice's rows 16.. (each warp's
//     third and fourth rows) into shared memory, so the whole slice is in
//     flight before the rotation starts.  When that staging does not fit two
//     CTAs per SM (more than two tokens), the third and fourth rows are loaded
//     into registers after the first two rows' dot products.
// Without a preceding launch of this kind (or after a kernel that never
// signals), the wait returns at once and the launch behaves like a plain one.
constexpr int kDxK = 4096;
constexpr int kDxChunks = kDxK / 16 / 32;  // 16-byte chunks per lane per row

// Dot products of one weight row (held as this lane's 8 chunks) against the quantized tokens, the
// warp reduction and the dequant epilogue (wsn, bn: the row's scale and bias, already loaded).
__device__ __forceinline__ void gemv_row_dot(const GemvArgs &p, const uint4 (&w)[kDxChunks], const int8_t *xq,
                                             const float *xs_s, int64_t n, int lane, float wsn, float bn) {
    int acc[kGvMaxM] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < kDxChunks; ++k) {
#pragma unroll
        for (int m = 0; m < kGvMaxM; ++m) {
            if (m < p.M) {
                const uint4 xv = reinterpret_cast<const uint4 *>(xq + (int64_t)m * kDxK)[lane + 32 * k];
                acc[m] = __dp4a((int)w[k].x, (int)xv.x, acc[m]);
                acc[m] = __dp4a((int)w[k].y, (int)xv.y, acc[m]);
                acc[m] = __dp4a((int)w[k].z, (int)xv.z, acc[m]);
                acc[m] = __dp4a((int)w[k].w, (int)xv.w, acc[m]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kGvMaxM; ++m) {
        if (m < p.M) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
        }
    }
    if (lane < p.M) {
        int a = acc[0];
#pragma unroll
        for (int m = 1; m < kGvMaxM; ++m)
            if (lane == m) a = acc[m];
        const float tv = __fmul_rn(__int2float_rn(a), xs_s[lane]);
        if (GBQ_IN_RANGE(p.status, (int64_t)lane * p.N + n, 1, p.M * p.N))
            p.y[(int64_t)lane * p.N + n] = __float2bfloat16_rn(__fmaf_rn(tv, wsn, bn));
    }
}

// One token (M = 1): the dot product of a weight row with the lane's eight code chunks xr, in four
// independent dp4a chains; the lane's partial sum (the warp reduction follows).
__device__ __forceinline__ int gemv_dot_m1(const uint4 (&w)[kDxChunks], const uint4 (&xr)[kDxChunks]) {
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int k = 0; k < kDxChunks; ++k) {
        a0 = __dp4a((int)w[k].x, (int)xr[k].x, a0);
        a1 = __dp4a((int)w[k].y, (int)xr[k].y, a1);
        a2 = __dp4a((int)w[k].z, (int)xr[k].z, a2);
        a3 = __dp4a((int)w[k].w, (int)xr[k].w, a3);
    }
    return (a0 + a1) + (a2 + a3);
}

// Warp sums of four per-lane values v[0..3] in six shuffles: afterwards lanes 8 q .. 8 q + 7 hold
// the total of v[q] (a transposing reduction: halve the values held, then sum within 8 lanes).
__device__ __forceinline__ int warp_sum4(const int (&v)[4], int lane) {
    const bool hi = (lane >> 4) & 1;
    const int s0 = __shfl_xor_sync(0xffffffffu, hi ? v[0] : v[2], 16);
    const int s1 = __shfl_xor_sync(0xffffffffu, hi ? v[1] : v[3], 16);
    const int k0 = (hi ? v[2] : v[0]) + s0;  // row 2 hi
    const int k1 = (hi ? v[3] : v[1]) + s1;  // row 2 hi + 1
    const bool b = (lane >> 3) & 1;
    int t = (b ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b ? k0 : k1, 8);
    t += __shfl_xor_sync(0xffffffffu, t, 4);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    return t;
}

__device__ __forceinline__ void gemv_load_row(uint4 (&w)[kDxChunks], const int8_t *w8, int64_t n, int lane) {
    const uint4 *src = reinterpret_cast<const uint4 *>(w8 + n * kDxK);
#pragma unroll
    for (int k = 0; k < kDxChunks; ++k) w[k] = __ldcs(src + lane + 32 * k);
}

// One H4/2 level on register digit D (register bits 2D, 2D + 1) of 16 values: the operations of
// h4_level, so the values equal the square kernels' bit for bit.
template <int D>
__device__ __forceinline__ void h4_regs16(float (&v)[16]) {
#pragma unroll
    for (int base = 0; base < 16; ++base) {
        if ((base >> (2 * D)) & 3) continue;
        const int b1 = base | (1 << (2 * D)), b2 = base | (2 << (2 * D)), b3 = base | (3 << (2 * D));
        const float x0 = v[base], x1 = v[b1], x2 = v[b2], x3 = v[b3];
        const float h = __fmul_rn(__fadd_rn(__fadd_rn(x0, x1), __fadd_rn(x2, x3)), 0.5f);
        v[base] = __fmaf_rn(x3, -1.0f, h);
        v[b1] = __fmaf_rn(x2, -1.0f, h);
        v[b2] = __fmaf_rn(x1, -1.0f, h);
        v[b3] = __fmaf_rn(x0, -1.0f, h);
    }
}

constexpr int kDxPitch = 80;                         // floats per row of the 64-row exchange tile
constexpr uint32_t kDxTileBytes = 64 * kDxPitch * 4;  // 20 KB

// Rotate + quantize one 4096-long token row (bf16, staged at xb) with all 256 threads of the CTA:
// X[i][j] (element 64 i + j) becomes V = H64 X H64 / 64 in the level order of the n = 64 kernels
// (i01, i23, i45, j45, j01, j23) with their operations, so the codes are gbq_quantize_act's bit for
// bit.  Each thread holds 16 values in three layouts (register bits / lane bits / warp bits):
//   1: (i0..i3) / (j0..j4) / (j5, i4, i5)   levels i01, i23     from the staged x
//   2: (i4, i5, j4, j5) / (j0..j3, i0) / (i1, i2, i3)   levels i45, j45   via the tile T
//   3: (j0..j3) / (i4, i5, j4, j5, i0) / (i1, i2, i3)   levels j01, j23   via warp shuffles
// Layout 3 leaves 16 consecutive values per thread: one 16-byte store of codes.  T is 64 rows of
// kDxPitch floats (both tile patterns are free of bank conflicts).  Two CTA barriers.
__device__ __forceinline__ void gemv_rot64_all(const uint8_t *xb, float *T, float *wmax, int8_t *xq_row,
                                               float *xs_out, int tid) {
    const int w = tid >> 5, l = tid & 31;
    float v[16];
    {
        const uint16_t *x16 = reinterpret_cast<const uint16_t *>(xb);
        const int j = l + 32 * (w & 1), i0 = 16 * (w >> 1);
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = bf16_to_float(x16[64 * (i0 + r) + j]);
        h4_regs16<0>(v);
        h4_regs16<1>(v);
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(i0 + r) * kDxPitch + j] = v[r];
    }
    __syncthreads();
    {
        const int jl = l & 15, ib = (l >> 4) + 2 * w;
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = T[(ib + 16 * (r & 3)) * kDxPitch + jl + 16 * (r >> 2)];
        h4_regs16<0>(v);
        h4_regs16<1>(v);
    }
    // register bit k <-> lane bit k, k = 0..3
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool up = (l >> k) & 1;
#pragma unroll
        for (int r0 = 0; r0 < 16; ++r0) {
            if ((r0 >> k) & 1) continue;
            const int r1 = r0 | (1 << k);
            const float got = __shfl_xor_sync(0xffffffffu, up ? v[r0] : v[r1], 1 << k);
            if (up)
                v[r0] = got;
            else
                v[r1] = got;
        }
    }
    h4_regs16<0>(v);
    h4_regs16<1>(v);
    float m = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) m = fmaxf(m, fabsf(v[r]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (l == 0) wmax[w] = m;
    __syncthreads();  // also: every layout-2 read of T is done
    float amax = wmax[0];
#pragma unroll
    for (int k = 1; k < kGvThreads / 32; ++k) amax = fmaxf(amax, wmax[k]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (tid == 0) *xs_out = s;
    float2 pv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pv[k] = make_float2(v[k], v[k + 8]);
    uint32_t words[2][2];
    quant_codes<8>(pv, s, words);
    const int e0 = 16 * ((l >> 2) & 3) + 64 * ((l >> 4) + 2 * w + 16 * (l & 3));
    *reinterpret_cast<uint4 *>(xq_row + e0) = make_uint4(words[0][0], words[0][1], words[1][0], words[1][1]);
}

template <int RPW>
__global__ void __launch_bounds__(kGvThreads, 2) gemv_direct_kernel(GemvArgs p) {
    extern __shared__ __align__(128) uint8_t smem[];
    int8_t *xq = reinterpret_cast<int8_t *>(smem + p.x_off);
    float2 *T = reinterpret_cast<float2 *>(smem + p.t_off);
    float *xs_s = reinterpret_cast<float *>(smem + p.misc_off);
    float *wmax = xs_s + kGvMaxM;                                             // one slot per warp
    uint64_t *xfull = reinterpret_cast<uint64_t *>(wmax + kGvThreads / 32);  // byte 48 of misc
    int *abort_flag = reinterpret_cast<int *>(xfull + 1);
    uint64_t *wfull = xfull + 2;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t r0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int nrows = (int)(min(p.N, r0 + p.rows_per_cta) - r0);
    // Debug builds: the CTA's weight slice (every weight copy and load below) lies inside W8.
    if (!GBQ_IN_RANGE(p.status, r0 * kDxK, (int64_t)nrows * kDxK, p.N * kDxK)) return;
    const int wrows = p.wrow_off ? max(0, nrows - 16) : 0;  // slice rows 16.. staged in shared memory

    // L2 prefetch of the slice (nrows * 4096 bytes, 128-byte lines), spread over the threads.
    {
        const char *base = reinterpret_cast<const char *>(p.w8 + r0 * kDxK);
        for (int l = tid; l < nrows * (kDxK / 128); l += kGvThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (size_t)l * 128));
        if (tid < nrows) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.ws + r0 + tid));
    }
    pdl_allow_dependents();  // the next call may start and prefetch its weight
    pdl_wait();              // every input may come from the kernel before
    if (tid == 0) {
        mbar_init(xfull, 1);
        mbar_init(wfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(xfull, (uint32_t)(p.M * kDxK * 2));
        bulk_g2s(smem + p.xb_off, p.x, (uint32_t)(p.M * kDxK * 2), xfull);
    }
    // Lane q < RPW holds the scale and bias of row warp + 8 q (loaded now, off the epilogue's path).
    float ws_l = 0.0f, b_l = 0.0f;
    if (lane < RPW && warp + 8 * lane < nrows) {
        ws_l = __ldg(p.ws + r0 + warp + 8 * lane);
        if (p.bias) b_l = __bfloat162float(p.bias[r0 + warp + 8 * lane]);
    }
    __syncthreads();  // the barriers are initialised
    // The x copy goes first (the rotation waits on it); the weight requests follow once it has landed
    // and arrive while x is rotated: this warp's rows j = warp + 8 q, the first two into registers,
    // the slice's rows 16.. into shared memory.
    const bool xok = mbar_wait(xfull, 0, p.status, abort_flag);
    if (tid == 0 && wrows > 0 && xok) {
        mbar_arrive_expect_tx(wfull, (uint32_t)wrows * kDxK);
        bulk_g2s(smem + p.wrow_off, p.w8 + (r0 + 16) * kDxK, (uint32_t)wrows * kDxK, wfull);
    }
    uint4 wa[kDxChunks], wb[kDxChunks];
    const bool has0 = warp < nrows, has1 = RPW > 1 && warp + 8 < nrows;
    if (has0) gemv_load_row(wa, p.w8, r0 + warp, lane);
    if (has1) gemv_load_row(wb, p.w8, r0 + warp + 8, lane);

    // ---- rotate + quantize x: every thread, one token at a time ----
    if (__syncthreads_and(xok)) {
        float *Tf = reinterpret_cast<float *>(T);
        for (int m = 0; m < p.M; ++m)
            gemv_rot64_all(smem + p.xb_off + (size_t)m * kDxK * 2, Tf, wmax, xq + (int64_t)m * kDxK, xs_s + m, tid);
    }
    __syncthreads();
    // Copies in flight when a wait gave up land (bounded) before the CTA leaves: x (if its wait gave
    // up) and the staged weight rows (issued only after x landed).
    auto drain = [&] {
        if (tid == 0 && !xok) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(xfull, 0) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
        if (tid == 0 && wrows > 0 && xok) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(wfull, 0) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    };
    if (*(volatile int *)abort_flag) {
        drain();
        return;
    }

    // ---- dot products: rows 0, 1 from registers; rows 2, 3 from shared memory or, after the first
    // two, from L2 into the same registers ----
    auto wsq = [&](int q) { return __shfl_sync(0xffffffffu, ws_l, q); };
    auto bq = [&](int q) { return __shfl_sync(0xffffffffu, b_l, q); };
    const bool has2 = RPW > 2 && warp + 16 < nrows, has3 = RPW > 3 && warp + 24 < nrows;
    auto smem_row = [&](uint4 (&w)[kDxChunks], int j) {
        const uint4 *src = reinterpret_cast<const uint4 *>(smem + p.wrow_off + (size_t)(j - 16) * kDxK);
#pragma unroll
        for (int k = 0; k < kDxChunks; ++k) w[k] = src[lane + 32 * k];
    };
    if (p.M == 1) {
        // One token: the lane's codes stay in registers for all rows; one reduction for the four rows.
        uint4 xr[kDxChunks];
#pragma unroll
        for (int k = 0; k < kDxChunks; ++k) xr[k] = reinterpret_cast<const uint4 *>(xq)[lane + 32 * k];
        int part[4] = {0, 0, 0, 0};
        if (has0) part[0] = gemv_dot_m1(wa, xr);
        if (has1) part[1] = gemv_dot_m1(wb, xr);
        if (has2 || has3) {
            if (wrows > 0) {
                if (!mbar_wait(wfull, 0, p.status, abort_flag)) {
                    drain();
                    return;
                }
                if (has2) smem_row(wa, warp + 16);
                if (has3) smem_row(wb, warp + 24);
            } else {
                if (has2) gemv_load_row(wa, p.w8, r0 + warp + 16, lane);
                if (has3) gemv_load_row(wb, p.w8, r0 + warp + 24, lane);
            }
            if (has2) part[2] = gemv_dot_m1(wa, xr);
            if (has3) part[3] = gemv_dot_m1(wb, xr);
        }
        const int tot = warp_sum4(part, lane);
        const int q = lane >> 3;
        const float wsv = __shfl_sync(0xffffffffu, ws_l, q), bv = __shfl_sync(0xffffffffu, b_l, q);
        if ((lane & 7) == 0 && q < RPW && warp + 8 * q < nrows) {
            const float tv = __fmul_rn(__int2float_rn(tot), xs_s[0]);
            if (GBQ_IN_RANGE(p.status, r0 + warp + 8 * q, 1, p.N))
                p.y[r0 + warp + 8 * q] = __float2bfloat16_rn(__fmaf_rn(tv, wsv, bv));
        }
        if (wrows > 0 && !(has2 || has3)) {  // this warp had no staged rows: the copy still lands before exit
            if (!mbar_wait(wfull, 0, p.status, abort_flag)) drain();
        }
        return;
    }
    if (has0) gemv_row_dot(p, wa, xq, xs_s, r0 + warp, lane, wsq(0), bq(0));
    if (wrows > 0) {
        if (has1) gemv_row_dot(p, wb, xq, xs_s, r0 + warp + 8, lane, wsq(1), bq(1));
        if (!mbar_wait(wfull, 0, p.status, abort_flag)) {
            drain();
            return;
        }
        if (has2) {
            smem_row(wa, warp + 16);
            gemv_row_dot(p, wa, xq, xs_s, r0 + warp + 16, lane, wsq(2), bq(2));
        }
        if (has3) {
            smem_row(wb, warp + 24);
            gemv_row_dot(p, wb, xq, xs_s, r0 + warp + 24, lane, wsq(3), bq(3));
        }
        return;
    }
    if (has2) gemv_load_row(wa, p.w8, r0 + warp + 16, lane);
    if (has1) gemv_row_dot(p, wb, xq, xs_s, r0 + warp + 8, lane, wsq(1), bq(1));
    if (has3) gemv_load_row(wb, p.w8, r0 + warp + 24, lane);
    if (has2) gemv_row_dot(p, wa, xq, xs_s, r0 + warp + 16, lane, wsq(2), bq(2));
    if (has3) gemv_row_dot(p, wb, xq, xs_s, r0 + warp + 24, lane, wsq(3), bq(3));
}

// Launch the register-streaming kernel when the shape fits it; GBQ_ENOTSUP otherwise.
int launch_gemv_direct(const GemvArgs &base, int num_sms, cudaStream_t st) {
    GemvArgs a = base;
    if (a.K != kDxK || a.G != 1) return GBQ_ENOTSUP;
    const int64_t rpc = (a.N + num_sms - 1) / num_sms;
    if (rpc > 32) return GBQ_ENOTSUP;
    const int rpw = (int)((rpc + 7) / 8);
    a.rows_per_cta = (int)rpc;
    const int64_t grid = (a.N + rpc - 1) / rpc;
    a.x_off = 0;
    a.t_off = (uint32_t)(((size_t)a.M * kDxK + 127) & ~(size_t)127);
    a.misc_off = a.t_off + ((kDxTileBytes + 127) & ~127u);
    a.xb_off = a.misc_off + 128;
    size_t smem = a.xb_off + (size_t)a.M * kDxK * 2;
    // Stage the slice's rows 16.. in shared memory when two CTAs still fit per SM.
    a.wrow_off = 0;
    if (rpc > 16) {
        const size_t off = (smem + 127) & ~(size_t)127;
        const size_t with = off + (size_t)(rpc - 16) * kDxK;
        if (2 * (with + 1024) <= 228 * 1024) {
            a.wrow_off = (uint32_t)off;
            smem = with;
        }
    }
    static bool attr[5] = {false, false, false, false, false};
    auto kern = rpw == 1 ? gemv_direct_kernel<1> : rpw == 2 ? gemv_direct_kernel<2>
              : rpw == 3 ? gemv_direct_kernel<3> : gemv_direct_kernel<4>;
    if (!attr[rpw]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGvSmem) != cudaSuccess)
            return gbq_fail(GBQ_ECUDA, "gemv: cannot set shared memory size");
        attr[rpw] = true;
    }
    cudaLaunchAttribute lattr[1];
    lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    lattr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = lattr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    prof_begin(3, st);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    prof_end(st);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? GBQ_OK : gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
}

// Ring of a slice of rpc weight rows of K bytes beside `fixed` bytes of other shared memory: the number of
// stages (kGvStages or 3) and rows per stage (at most nv / MP for MP padded tokens, and at most a 1/S share of
// the slice so every stage is used).  A chunk costs ~1.5-1.8 K cycles of wait, reduction and epilogue (per-
// stage timestamps) plus its dot products, which run over the rows padded to a power of two (the dot phase's
// instantiations): ~16 MP K / 4096 cycles a padded row.  The plan with the least modelled time wins, so few
// large stages beat many small ones, but not at the price of a half-empty power of two.  Sets nstages,
// rows_per_cta, rows_per_stage and stage_bytes; false when not one row fits per stage.
bool gv_plan_ring(GemvArgs &a, int64_t rpc, int64_t K, size_t fixed, int mp, int nv) {
    if (fixed >= kGvSmem) return false;
    const double chunk_cycles = 1500.0, row_cycles = 16.0 * mp * (double)K / 4096.0;
    double best = -1.0;
    for (int S = kGvStages; S >= 3; --S) {
        const int64_t per = (int64_t)((kGvSmem - fixed) / S) - 127;  // a stage is rounded up to 128 bytes
        const int64_t cap = per > 0 ? per / K : 0;
        const int64_t hi = std::min<int64_t>(std::min<int64_t>((rpc + S - 1) / S, cap), nv / mp);
        for (int64_t rps = 1; rps <= hi; ++rps) {
            int64_t rb = 2;
            while (rb < rps) rb *= 2;
            const int64_t chunks = (rpc + rps - 1) / rps;
            const double cost = (double)chunks * (chunk_cycles + (double)rb * row_cycles);
            if (best < 0.0 || cost < best) {
                best = cost;
                a.nstages = S;
                a.rows_per_stage = (int)rps;
                a.stage_bytes = (uint32_t)(((size_t)rps * K + 127) & ~(size_t)127);
            }
        }
    }
    a.rows_per_cta = (int)rpc;
    return best >= 0.0;
}

template <int LOGN>
int launch_gemv_t(const GemvArgs &base, int num_sms, cudaStream_t st) {
    constexpr int TPG = RotGeom<LOGN>::TPG;
    GemvArgs a = base;
    if (a.G * TPG > kGvThreads) return GBQ_ENOTSUP;
    const size_t x_bytes = (size_t)a.M * a.K;
    size_t t_bytes = (size_t)a.G * RotGeom<LOGN>::TILE * sizeof(float2);
    if (LOGN == 6 && a.G == 1 && t_bytes < fast_tile_bytes(6)) t_bytes = fast_tile_bytes(6);  // three-pass tile
    const size_t xb_bytes = (LOGN == 6 && a.G == 1) ? (size_t)a.M * a.K * 2 + 128 : 0;  // bf16 token staging
    int64_t rpc = (a.N + num_sms - 1) / num_sms;
    const int64_t grid = (a.N + rpc - 1) / rpc;
    const size_t fixed = ((x_bytes + 127) & ~(size_t)127) + ((t_bytes + 127) & ~(size_t)127) + 128 + xb_bytes +
                         gv_ep_bytes(rpc, kGvNV);
    if (fixed + (size_t)kGvStages * a.K > kGvSmem) return GBQ_ENOTSUP;
    if (!gv_plan_ring(a, rpc, a.K, fixed, gv_pad_m(a.M), kGvNV)) return GBQ_ENOTSUP;
    a.x_off = (uint32_t)((size_t)a.nstages * a.stage_bytes);
    a.t_off = a.x_off + (uint32_t)((x_bytes + 127) & ~(size_t)127);
    a.misc_off = a.t_off + (uint32_t)((t_bytes + 127) & ~(size_t)127);
    a.xb_off = 0;
    a.ep_off = a.misc_off + 128;  // misc <= 128 bytes
    size_t smem = a.ep_off + gv_ep_bytes(rpc, kGvNV);
    if (LOGN == 6 && a.G == 1) {
        a.xb_off = (uint32_t)((smem + 127) & ~(size_t)127);
        smem = a.xb_off + (size_t)a.M * a.K * 2;
    }
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemv_kernel<LOGN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGvSmem) !=
            cudaSuccess)
            return gbq_fail(GBQ_ECUDA, "gemv: cannot set shared memory size");
        attr = true;
    }
    prof_begin(3, st);
    gemv_kernel<LOGN><<<(unsigned)grid, kGvThreads, smem, st>>>(a);
    prof_end(st);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GBQ_OK : gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// Decode GEMV for the descriptors the square in-kernel rotations do not take (a != b, odd total log2,
// small factors, many groups, K above 4096), one or two tokens: every CTA rotates and quantizes the
// tokens itself with the generic rotation's passes (rotate_g.cuh: rotg_kernel's level list and fp32
// operations, so the same codes and scales) while its first weight stages stream in.  Launched with
// programmatic stream serialization: the weight copies and the epilogue operands are issued before
// griddepcontrol.wait, x is read after it, and the next launch may start at entry.
__global__ void __launch_bounds__(kGvThreads, 2) gemv_gen_kernel(GemvArgs p, gen::GenArgs g) {
    static_assert(kGvThreads == gen::kGenThreads, "the generic passes stride over the CTA's threads");
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    int8_t *xq = reinterpret_cast<int8_t *>(smem + p.x_off);
    float *xs_s = reinterpret_cast<float *>(smem + p.misc_off);      // [kGvMaxM] token scales
    unsigned *rowmax = reinterpret_cast<unsigned *>(xs_s + kGvMaxM);  // [kGvMaxM]
    uint64_t *full = reinterpret_cast<uint64_t *>(rowmax + kGvMaxM);
    int *abort_flag = reinterpret_cast<int *>(full + kGvStages);
    float *T = reinterpret_cast<float *>(smem + p.t_off);
    float *ep = reinterpret_cast<float *>(smem + p.ep_off);

    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int nrows = (int)(min(p.N, r0 + p.rows_per_cta) - r0);
    // Debug builds: the CTA's weight slice (every weight copy below) lies inside W8.
    if (!GBQ_IN_RANGE(p.status, r0 * p.K, (int64_t)nrows * p.K, p.N * p.K)) return;
    const int nchunks = (nrows + p.rows_per_stage - 1) / p.rows_per_stage;
    if (tid == 0) {
        for (int s2 = 0; s2 < kGvStages; ++s2) mbar_init(&full[s2], 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int c = 0; c < nchunks && c < p.nstages; ++c) {
            const int rows = min(p.rows_per_stage, nrows - c * p.rows_per_stage);
            mbar_arrive_expect_tx(&full[c], (uint32_t)rows * (uint32_t)p.K);
            gv_copy_rows(p, stages + (size_t)c * p.stage_bytes, r0 + (int64_t)c * p.rows_per_stage, rows, &full[c]);
        }
    }
    if (tid < kGvMaxM) rowmax[tid] = 0u;
    gv_load_epilogue(p, ep, r0, nrows);  // w_scale and bias: not written by the kernel before
    pdl_allow_dependents();              // the next call may start and issue its weight copies
    pdl_wait();                          // x may come from the kernel before

    // ---- rotate + quantize the tokens (rotg_kernel's phases on one chunk of M rows) ----
    const int K = g.K;
    const int E = (int)p.M * K;
    for (int u = tid; u < (E >> 3); u += kGvThreads) {
        const int e = u * 8, row = gen::gen_row(g, e);
        float x[8];
        if (GBQ_IN_RANGE(p.status, row, 1, p.M) && GBQ_IN_RANGE(p.status, e - row * K, 8, K)) {
            gen::gen_load8<IN_BF16>(g, row, e - row * K, x);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = 0.0f;
        }
        float *t = T + gen::tix(e);  // eight values inside one 32-value block
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = x[k];
    }
    __syncthreads();  // the tile is complete; rowmax and the barriers are initialised
    for (int l = 0; l < g.nlev; l += 2) {
        const bool pair = l + 1 < g.nlev;
        const int w1 = g.wid[l], w2 = pair ? g.wid[l + 1] : 0;
        const int p1 = g.pos[l], p2 = pair ? g.pos[l + 1] : 0;
        if (l + 2 >= g.nlev)
            gen::gen_pass_dispatch<true, OUT_S8>(w1, w2, T, E, p1, p2, g, rowmax);
        else
            gen::gen_pass_dispatch<false, OUT_S8>(w1, w2, T, E, p1, p2, g, rowmax);
        __syncthreads();
    }
    if (tid < p.M) xs_s[tid] = __fdiv_rn(__uint_as_float(rowmax[tid]), 127.0f);
    __syncthreads();
    for (int u = tid; u < (E >> 4); u += kGvThreads) {  // 16 contiguous codes per thread
        const int e = u * 16, row = gen::gen_row(g, e);
        const float *t = T + gen::tix(e);
        float2 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = make_float2(t[k], t[k + 8]);
        uint32_t words[2][2];
        quant_codes<8>(v, xs_s[row], words);
        *reinterpret_cast<uint4 *>(xq + e) = make_uint4(words[0][0], words[0][1], words[1][0], words[1][1]);
    }
    __syncthreads();  // the codes are complete

    gemv_dot_phase<kGvGenMaxM, kGvNV>(p, stages, xq, xs_s, full, abort_flag, r0, nrows, nchunks, ep);
    if (tid == 0 && *(volatile int *)abort_flag) {
        // A wait gave up: let the copies issued at entry land (bounded) before the CTA leaves.
        for (int c = 0; c < min(nchunks, p.nstages); ++c) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&full[c], 0) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    }
}

}  // namespace

// Shared memory of gemv_codes_kernel besides the weight ring: the codes, the scales and barriers, the
// epilogue operands.
size_t gemv_codes_fixed(int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t rpc = (N + num_sms - 1) / num_sms;
    return (((size_t)M * K + 127) & ~(size_t)127) + 128 + gv_ep_bytes(rpc, kGcNV);
}

bool gemv_codes_fits(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (M < 1 || M > kGcMaxM || K < 16 || K % 16 != 0 || N < 1 || num_sms < 1) return false;
    const size_t fixed = gemv_codes_fixed(M, N, K, num_sms);
    return fixed < kGvSmem && (kGvSmem - fixed) / kGvStages >= (size_t)K + 127;  // one row per stage at least
}

int launch_gemv_codes2(const int8_t *codes, const float *scales, const int8_t *w8, const float *w_scale,
                       const int8_t *w8b, const float *w_scale_b, int64_t n_split, const void *bias, void *y,
                       int64_t ld_y, int64_t M, int64_t N, int64_t K, int num_sms, cudaStream_t st,
                       unsigned int *status) {
    if (!gemv_codes_fits(M, N, K, num_sms) || ld_y < N || n_split < 0 || n_split > N) return GBQ_ENOTSUP;
    if (((uintptr_t)codes | (uintptr_t)w8 | (uintptr_t)w8b) & 15) return GBQ_ENOTSUP;
    GemvArgs a{};
    a.w8 = w8;
    a.ws = w_scale;
    a.w8b = w8b;
    a.wsb = w_scale_b;
    a.n_split = n_split;
    a.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
    a.y = reinterpret_cast<__nv_bfloat16 *>(y);
    a.M = M;
    a.N = N;
    a.K = K;
    a.ld_y = ld_y;
    a.G = 1;
    a.status = status;
    const size_t x_bytes = (size_t)M * K;
    const size_t fixed = gemv_codes_fixed(M, N, K, num_sms);
    const int64_t rpc = (N + num_sms - 1) / num_sms;
    const int64_t grid = (N + rpc - 1) / rpc;
    if (!gv_plan_ring(a, rpc, K, fixed, gv_pad_m(M), kGcNV)) return GBQ_ENOTSUP;
    a.x_off = (uint32_t)((size_t)a.nstages * a.stage_bytes);
    a.misc_off = a.x_off + (uint32_t)((x_bytes + 127) & ~(size_t)127);
    a.ep_off = a.misc_off + 128;  // scales, barriers, abort flag, codes barrier: < 128 bytes
    const size_t smem = a.ep_off + gv_ep_bytes(rpc, kGcNV);
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemv_codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGvSmem) !=
            cudaSuccess)
            return gbq_fail(GBQ_ECUDA, "gemv: cannot set shared memory size");
        attr = true;
    }
    cudaLaunchAttribute lattr[1];
    lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    lattr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = lattr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    prof_begin(3, st);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_codes_kernel, a, codes, scales);
    prof_end(st);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? GBQ_OK : gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
}

int launch_gemv_codes(const int8_t *codes, const float *scales, const int8_t *w8, const float *w_scale,
                      const void *bias, void *y, int64_t ld_y, int64_t M, int64_t N, int64_t K, int num_sms,
                      cudaStream_t st, unsigned int *status) {
    return launch_gemv_codes2(codes, scales, w8, w_scale, w8, w_scale, N, bias, y, ld_y, M, N, K, num_sms, st,
                              status);
}

// Shared memory of gemv_gen_kernel besides the weight ring: the codes, the misc block, the epilogue
// operands, the fp32 rotation tile of the M token rows (one pad float per 32).
size_t gemv_gen_fixed(int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t rpc = (N + num_sms - 1) / num_sms;
    const size_t E = (size_t)M * K;
    return ((E + 127) & ~(size_t)127) + 128 + gv_ep_bytes(rpc, kGvNV) + (((E + E / 32) * 4 + 127) & ~(size_t)127);
}

bool gemv_gen_fits(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (M < 1 || M > kGvGenMaxM || K < 16 || K % 16 != 0 || K > kGenMaxK || N < 1 || num_sms < 1) return false;
    if ((uint64_t)M * (uint64_t)K * (uint64_t)K >= ((uint64_t)1 << 32)) return false;  // gen::gen_row's range
    const size_t fixed = gemv_gen_fixed(M, N, K, num_sms);
    return fixed < kGvSmem && (kGvSmem - fixed) / kGvStages >= (size_t)K + 127;  // one row per stage at least
}

int launch_gemv_gen(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y, int64_t M,
                    int64_t N, int64_t K, int la, int lb, int num_sms, cudaStream_t st, unsigned int *status) {
    if (!gemv_gen_fits(M, N, K, num_sms) || la + lb < 1) return GBQ_ENOTSUP;
    if (((uintptr_t)x | (uintptr_t)w8) & 15) return GBQ_ENOTSUP;
    GemvArgs a{};
    a.x = x;
    a.w8 = w8;
    a.ws = w_scale;
    a.w8b = w8;
    a.wsb = w_scale;
    a.n_split = N;
    a.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
    a.y = reinterpret_cast<__nv_bfloat16 *>(y);
    a.M = M;
    a.N = N;
    a.K = K;
    a.ld_y = N;
    a.G = 1;
    a.status = status;
    gen::GenArgs g{};
    g.in0 = x;
    g.ld_in = K;
    g.M = M;
    gen::gen_set_k(g, (int)K);
    g.R = (int)M;
    g.status = status;
    gen::gen_levels(la, lb, g);
    const size_t fixed = gemv_gen_fixed(M, N, K, num_sms);
    const int64_t rpc = (N + num_sms - 1) / num_sms;
    const int64_t grid = (N + rpc - 1) / rpc;
    if (!gv_plan_ring(a, rpc, K, fixed, gv_pad_m(M), kGvNV)) return GBQ_ENOTSUP;
    a.x_off = (uint32_t)((size_t)a.nstages * a.stage_bytes);
    a.misc_off = a.x_off + (uint32_t)(((size_t)M * K + 127) & ~(size_t)127);
    a.ep_off = a.misc_off + 128;  // token scales, row maxima, stage barriers, abort flag: < 128 bytes
    a.t_off = a.ep_off + (uint32_t)gv_ep_bytes(rpc, kGvNV);
    const size_t E = (size_t)M * K;
    const size_t smem = a.t_off + (((E + E / 32) * 4 + 127) & ~(size_t)127);
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemv_gen_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGvSmem) !=
            cudaSuccess)
            return gbq_fail(GBQ_ECUDA, "gemv: cannot set shared memory size");
        attr = true;
    }
    cudaLaunchAttribute lattr[1];
    lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    lattr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = lattr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    prof_begin(3, st);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_gen_kernel, a, g);
    prof_end(st);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? GBQ_OK : gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
}

int launch_gemv(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y, int64_t M, int64_t N,
                int64_t K, int logn, int groups, int num_sms, cudaStream_t st, unsigned int *status) {
    if (M < 1 || M > kGvMaxM || K % 128 != 0) return GBQ_ENOTSUP;
    GemvArgs a{};
    a.x = x;
    a.w8 = w8;
    a.ws = w_scale;
    a.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
    a.y = reinterpret_cast<__nv_bfloat16 *>(y);
    a.M = M;
    a.N = N;
    a.K = K;
    a.ld_y = N;
    a.w8b = w8;
    a.wsb = w_scale;
    a.n_split = N;
    a.G = groups;
    a.status = status;
    // Both kernels rotate every token in each CTA, one token after the other: past two tokens or K = 4096
    // the rotation kernels plus gemv_codes_kernel are faster (measured: K = 8192 as 64x64x2, one token, 27
    // vs 24 us; K = 4096 as 32x32x4, four tokens, 17.8 vs 15.1 us; K = 4096 as 64x64, three / four tokens,
    // 11.4 / 13.6 vs 9.8 / 9.9 us), so those return GBQ_ENOTSUP.
    if (M > 2 || K > 4096) return GBQ_ENOTSUP;
    switch (logn) {
        case 4: return launch_gemv_t<4>(a, num_sms, st);
        case 5: return launch_gemv_t<5>(a, num_sms, st);
        case 6: {
            const int rc = launch_gemv_direct(a, num_sms, st);
            return rc == GBQ_ENOTSUP ? launch_gemv_t<6>(a, num_sms, st) : rc;
        }
        default: return GBQ_ENOTSUP;
    }
}

}  // namespace gbq
