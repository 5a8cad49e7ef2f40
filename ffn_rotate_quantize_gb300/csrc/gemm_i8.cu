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
//   * K is cut into exact chunks: 1024 long for any int8 data, or 2^j x 1024
//     for a token tile whose rows' sums of |q| over those blocks allow it (the
//     chunk plan below).  After each chunk the eight epilogue warps drain the
//     fp32 accumulator (fp32 -> int32, exact) into int32 running totals held in
//     their registers; the MMA of the next chunk starts once all of them have
//     read it.  There is one N = 256 accumulator: with the weight's A ring it
//     fills the 512 TMEM columns, so drains cannot be double-buffered.
//
// CTA pairs.  Two CTAs of a cluster share one 256 x 256 tile: the pair MMA
// (tcgen05 cta_group::2, M = 256, N = 256) takes weight rows 128r..128r+127 from
// CTA r's tensor memory and tokens 128r..128r+127 from CTA r's shared memory,
// and writes D rows 128r.. into CTA r's tensor memory.  Each SM so stages only
// half the token tile: 384 bytes of operands per unit of K for 128 x 256
// products, against 640 for a one-CTA 128 x 256 tile.  The fp16-coded tokens
// are what fills shared memory and the L2 -> SM path; halving them is what lets
// four 48 KB stages stay in flight.
//
// The weight is the A operand and lives in TMEM: a converter warpgroup in each
// CTA widens the TMA-staged int8 tile to fp16 in 64-deep sub-steps
// (byte-permute + one half2 subtract per pair) and tcgen05.st's it into an
// 8-slot ring.  CTA 0's warp 1 issues every MMA of the pair once both CTAs'
// converters have published the sub-step (remote mbarrier arrivals); its
// commits arrive on the barriers of both CTAs (multicast).
//
// Warp roles per CTA (512 threads): warps 0 and 2 TMA producers (alternate
// stages), warp 1 TMEM owner (+ the MMA issuer in CTA 0), warps 4-7
// converters, warps 8-15 epilogue (warp w owns TMEM lane quadrant w%4 and
// token half (w/4)%2).  Register budgets per warpgroup (setmaxnreg; launch
// total 512 x 128 = 65,536): 48 + 88 + 184 + 184 = 504 per lane -> 64,512.
// Every mbarrier wait is bounded; a timeout in one CTA aborts its peer too.
//
// TMEM columns: [0,256) A ring (8 x 32), [256,512) accumulator.
#include "common.cuh"
#include "gemm.h"

namespace gbq {
namespace {

constexpr int kPairM = 256;              // weight rows per CTA pair (pair MMA M)
constexpr int kBM = 128;                 // weight rows per CTA
constexpr int kBN = 256;                 // tokens per tile (MMA N)
constexpr int kBNHalf = kBN / 2;         // tokens staged by each CTA
constexpr int kBK = 128;                 // K per shared-memory stage
constexpr int kSub = 64;                 // K per converter / A-ring sub-step
constexpr int kSubs = kBK / kSub;        // sub-steps per stage
constexpr int kStages = 4;
constexpr int kAStages = 8;
constexpr int kChunkSubs = 1024 / kSub;  // sub-steps per exact fp32 chunk
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0, kColAcc = 256;
constexpr int kProducers = 2;  // warps 0 and 2
constexpr int kThreads = 512;
constexpr int kEpiWarps = 8;
constexpr int kPlanTiles = 64;      // token tiles with a chunk plan (M <= 16384); beyond, 1024-long chunks
constexpr int kPlanMaxBlocks = 16;  // 1024-long K blocks per row the plan looks at (K <= 16384)
constexpr int kRegsWG0 = 48, kRegsConv = 88, kRegsEpi = 184;
static_assert(128 * (kRegsWG0 + kRegsConv + 2 * kRegsEpi) <= 65536, "register split exceeds the launch total");
static_assert(kStages % kProducers == 0, "each producer owns whole stages");
static_assert(kChunkSubs % kSubs == 0, "chunks end on stage boundaries");

// Producer index of a warp, or -1.
__device__ __forceinline__ int producer_id(int warp) {
    if (warp == 0) return 0;
    if (warp == 2) return 1;
    return -1;
}

constexpr uint32_t kTokBox = kBNHalf * 128;         // one 128-row x 128-byte token box (64 K)
constexpr uint32_t kBStageBytes = kSubs * kTokBox;  // 32 KB fp16 tokens
constexpr uint32_t kWStageBytes = kBM * kBK;        // 16 KB int8 weights (one 128 x 128-byte box)
constexpr uint32_t kOutBlock = 2048;                   // 32 columns x (32 bf16 | 16 four-byte) token rows
constexpr uint32_t kOutStaging = kEpiWarps * 2 * kOutBlock;  // per epilogue warp, double-buffered
constexpr size_t kSmemBytes =
    (size_t)kStages * (kBStageBytes + kWStageBytes) + kOutStaging + 1024 /*barriers*/ + 1024 /*align*/;
static_assert(kSmemBytes <= 232448, "shared memory exceeds the per-CTA limit");

struct Params {
    CUtensorMap tm_b;
    CUtensorMap tm_w0;
    CUtensorMap tm_w1;
    CUtensorMap tm_out;  // output [M][ld_out], box 32 columns x (kOutBlock / 32 / esz) rows
    int64_t M, N, K;
    int64_t n_split;
    int64_t ld_out;
    void *out;
    const float *x_scale;
    const float *w_scale0;
    const float *w_scale1;
    const __nv_bfloat16 *bias;
    const int32_t *row_l1;  // optional [M][l1_ld]: sum of |q| over each 1024-long block of a token row
    int64_t l1_ld;
    unsigned int *status;
    int w_layout;
    int epi;
    int use_tma_out;
    int reduce_out;  // EPI_ACC_I32: add into out instead of storing
    int wfast;       // tile order: weight blocks fastest (see tile_coords)
};

struct Bars {
    uint64_t full[kStages];     // local: TMA bytes landed
    uint64_t empty[kStages];    // local: pair MMA done reading (multicast commit) + local converters
    uint64_t afull[kAStages];   // CTA 0 only: converter warps of both CTAs published the sub-step
    uint64_t aempty[kAStages];  // both: pair MMA done reading the A slot (multicast commit)
    uint64_t accfull;           // both: chunk accumulated (multicast commit)
    uint64_t accempty;          // CTA 0 only: epilogue warps of both CTAs drained the accumulator
    uint64_t drain;             // CTA 0 only: every MMA finished
    uint64_t plan_ready;        // CTA 0 only: the epilogue warps published the chunk plan
    uint32_t plan[kPlanTiles];  // per token tile: bit j set = chunks of 2^j K blocks are exact for every token
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(Bars) <= 1024, "barriers exceed their shared-memory slot");

// Pair tile t: weight rows [n0, n0 + 256), tokens [m0, m0 + 256).  Consecutive tiles (run side by side
// by consecutive CTA pairs) share their weight block and walk the token tiles, so each wave reads its
// few weight blocks once and re-reads the token operand from L2 -- unless the token operand is the
// larger one per unit of K (wfast: more token bytes than weight bytes, e.g. the dx contraction over
// 4096 tokens), which then walks the weight blocks instead, reading each wave's token tiles once.
__device__ __forceinline__ void tile_coords(int64_t t, int64_t m_tiles, int64_t n_tiles, int wfast, int64_t *n0,
                                            int64_t *m0) {
    if (wfast) {
        *n0 = (t % n_tiles) * kPairM;
        *m0 = (t / n_tiles) * kBN;
    } else {
        *n0 = (t / m_tiles) * kPairM;
        *m0 = (t % m_tiles) * kBN;
    }
}
__device__ __forceinline__ int64_t tile_token_index(int64_t t, int64_t m_tiles, int64_t n_tiles, int wfast) {
    return wfast ? t / n_tiles : t % m_tiles;
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

// Sub-steps per exact chunk of token tile mt from its plan bits (longest level j whose bit is set;
// bits are only ever set for a prefix of levels).  Without a plan: 1024-long chunks.
__device__ __forceinline__ int tile_chunk_subs(const uint32_t *plan, const Params &p, int64_t mt, int tile_subs) {
    if (!p.row_l1 || p.K % 1024 != 0 || p.K / 1024 > kPlanMaxBlocks || mt >= kPlanTiles) return kChunkSubs;
    const uint32_t bits = plan[mt];
    const int j = 31 - __clz(bits);  // bit 0 is always set
    const int c = kChunkSubs << j;
    return c < tile_subs ? c : tile_subs;
}

// Add 32 exact integer-valued fp32 partial sums to int32 totals.  When every
// value of the warp is below 2^22 in magnitude, v + 1.5*2^23 lands in
// [2^23, 2^24) where the fp32 spacing is 1, so its bit pattern minus that of
// 1.5*2^23 is v exactly: one FADD + one integer add instead of a (quarter-rate)
// float -> int conversion.  Otherwise convert each value with round-to-nearest.
__device__ __forceinline__ void add_exact_totals(int32_t *tot, const uint32_t (&rr)[32]) {
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(rr[i])));
    if (__all_sync(0xffffffffu, mx < 4194304.0f)) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            tot[i] += (int32_t)(__float_as_uint(__fadd_rn(__uint_as_float(rr[i]), 12582912.0f)) - 0x4B400000u);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) tot[i] += __float2int_rn(__uint_as_float(rr[i]));
    }
}

// Write this thread's 128 token values of output column n: each epilogue warp
// stages blocks of ROWS tokens x its 32 columns in its own double-buffered
// shared-memory slots and lane 0 stores each block with one TMA tensor store
// (which clips rows and columns past the edge).  No warp waits on another.
// xs4[g] holds x_scale of token row m0 + 128h + 32g + lane (loaded when the tile starts).
template <int ROWS, int EPI>
__device__ __forceinline__ void store_tile_tma(const Params &p, const int32_t (&tot)[128], const float (&xs4)[4],
                                               uint8_t *wbuf_out, int h, int q, int lane, int64_t n0, int64_t m0,
                                               float ws, float bias) {
    constexpr uint32_t esz = EPI == EPI_DEQUANT_BF16 ? 2u : 4u;
    static_assert(ROWS * 32 * esz == kOutBlock, "block geometry");
#pragma unroll
    for (int j = 0; j < 128 / ROWS; ++j) {
        uint8_t *buf = wbuf_out + (uint32_t)(j & 1) * kOutBlock;
        const int64_t mb = m0 + 128 * h + ROWS * j;
        const float xs_l = xs4[(ROWS * j) / 32];
        const int xs_lane0 = (ROWS * j) % 32;
        if (lane == 0) tma_store_wait_read<1>();  // the store that last read `buf` is done
        __syncwarp();
        uint8_t *col = buf + (uint32_t)lane * esz;
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            const int32_t acc = tot[ROWS * j + i];
            if (EPI == EPI_ACC_I32) {
                *reinterpret_cast<int32_t *>(col + i * 32 * esz) = acc;
            } else if (EPI == EPI_DEQUANT_BF16) {
                const float xs = __shfl_sync(0xffffffffu, xs_l, xs_lane0 + i);
                const float tv = __fmul_rn(__int2float_rn(acc), xs);
                *reinterpret_cast<__nv_bfloat16 *>(col + i * 32 * esz) = __float2bfloat16_rn(__fmaf_rn(tv, ws, bias));
            } else {
                const float xs = __shfl_sync(0xffffffffu, xs_l, xs_lane0 + i);
                *reinterpret_cast<float *>(col + i * 32 * esz) = __fmul_rn(__int2float_rn(acc), xs);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (EPI == EPI_ACC_I32 && p.reduce_out)
                tma_reduce_add_2d(&p.tm_out, buf, (int)(n0 + 32 * q), (int)mb);
            else
                tma_store_2d(&p.tm_out, buf, (int)(n0 + 32 * q), (int)mb);
            tma_store_commit();
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) i8gemm_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // same offset in both CTAs
    uint8_t *bbuf = smem;
    uint8_t *wbuf = smem + kStages * kBStageBytes;
    uint8_t *obuf = wbuf + kStages * kWStageBytes;  // output staging
    Bars *bars = reinterpret_cast<Bars *>(obuf + kOutStaging);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();  // 0 leads the pair
    const uint32_t peer_abort = cluster_map(smem_u32(&bars->abort), rank ^ 1u);
    const int64_t pair = blockIdx.x >> 1;
    const int64_t npairs = gridDim.x >> 1;
    const int64_t m_tiles = (p.M + kBN - 1) / kBN;
    const int64_t n_tiles = (p.N + kPairM - 1) / kPairM;
    const int64_t num_tiles = m_tiles * n_tiles;
    const int KT = (int)((p.K + kBK - 1) / kBK);  // stages per tile (the K tail reads zeros)
    const int tile_subs = KT * kSubs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1 + 4 * kSubs);  // pair-MMA commit + every local converter warp per sub-step
        }
        for (int a = 0; a < kAStages; ++a) {
            mbar_init(&bars->afull[a], 8);  // four converter warps in each CTA
            mbar_init(&bars->aempty[a], 1);
        }
        mbar_init(&bars->accfull, 1);
        mbar_init(&bars->accempty, 2 * kEpiWarps);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->plan_ready, 1);
        for (int i = 0; i < kPlanTiles; ++i) bars->plan[i] = ~0u;
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_b);
        tma_prefetch_desc(&p.tm_w0);
        tma_prefetch_desc(&p.tm_w1);
        if (p.use_tma_out) tma_prefetch_desc(&p.tm_out);
    }
    if (warp == 1) tmem_alloc_pair(&bars->tmem_base, kTmemCols);
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const int wg = warp >> 2;
    const uint32_t lead_accempty = cluster_map(smem_u32(&bars->accempty), 0);

    if (wg == 0) {
        setmaxnreg_dec<kRegsWG0>();
        if (producer_id(warp) >= 0) {
            // ------------------------------------------------ TMA producers (alternate stages)
            const uint32_t pid = (uint32_t)producer_id(warp);
            if (lane == 0) {
                uint32_t gs = 0;
                bool ok = true, dep_done = false;
                for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
                    int64_t n0, m0;
                    tile_coords(t, m_tiles, n_tiles, p.wfast, &n0, &m0);
                    const int64_t nr = n0 + kBM * rank;  // this CTA's weight rows
                    const bool src1 = nr >= p.n_split;
                    const CUtensorMap *tw = src1 ? &p.tm_w1 : &p.tm_w0;
                    const int wrow = (int)(src1 ? nr - p.n_split : nr);
                    const int trow = (int)(m0 + kBNHalf * rank);  // this CTA's tokens
                    for (int kt = 0; kt < KT; ++kt) {
                        const uint32_t my = gs++;
                        if (my % kProducers != pid) continue;
                        const int stage = (int)(my % kStages);
                        ok = mbar_wait_cluster(&bars->empty[stage], ((my / kStages) & 1u) ^ 1u, p.status, abort,
                                               peer_abort);
                        if (!ok) break;
                        uint64_t *fb = &bars->full[stage];
                        mbar_arrive_expect_tx(fb, kBStageBytes + kWStageBytes);
                        uint8_t *wdst = wbuf + stage * kWStageBytes;
                        if (p.w_layout == W_KMAJOR)
                            tma_load_2d(wdst, tw, fb, kt * kBK, wrow);  // 128 rows x 128 K bytes
                        else
                            tma_load_2d(wdst, tw, fb, wrow, kt * kBK);  // 128 contraction rows x 128 columns
                        uint8_t *bdst = bbuf + stage * kBStageBytes;
                        if (!dep_done) {  // the tokens come from the preceding kernel: wait for it once
                            pdl_wait();
                            dep_done = true;
                        }
#pragma unroll
                        for (int b = 0; b < kSubs; ++b)
                            tma_load_2d(bdst + b * kTokBox, &p.tm_b, fb, kt * kBK + b * kSub, trow);
                    }
                }
            }
        } else if (warp == 1 && rank == 0) {
            // ------------------------------------------------ pair-MMA issuer (CTA 0)
            if (lane == 0) {
                constexpr uint32_t idesc = idesc_f16(kPairM, kBN, 0, 0, 0);
                uint32_t gs = 0, gsub = 0, chunk = 0;
                bool ok = mbar_wait_cluster(&bars->plan_ready, 0, p.status, abort, peer_abort);
                for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
                    const int csubs =
                        tile_chunk_subs(bars->plan, p, tile_token_index(t, m_tiles, n_tiles, p.wfast), tile_subs);
                    int cpos = 0;  // sub-step within the current chunk (kept incrementally: no division here)
                    for (int kt = 0; kt < KT && ok; ++kt) {
                        const uint32_t my = gs++;
                        const int stage = (int)(my % kStages);
                        // Both CTAs' stage data has landed once their converters publish its sub-steps.
                        const uint32_t b_stage = smem_u32(bbuf + stage * kBStageBytes);
                        for (int sub = 0; sub < kSubs && ok; ++sub) {
                            const uint32_t ms = gsub++;
                            const int tsub = kt * kSubs + sub;  // sub-step within the tile
                            if (cpos == 0) {  // a new chunk: both CTAs' accumulators must have been drained
                                ok = mbar_wait_cluster(&bars->accempty, (chunk & 1u) ^ 1u, p.status, abort,
                                                       peer_abort);
                                if (!ok) break;
                            }
                            const int as = (int)(ms % kAStages);
                            ok = mbar_wait_cluster(&bars->afull[as], (ms / kAStages) & 1u, p.status, abort,
                                                   peer_abort);
                            if (!ok) break;
                            tc_fence_after();
#pragma unroll
                            for (int k16 = 0; k16 < kSub / 16; ++k16) {
                                const uint64_t bdesc =
                                    smem_desc(b_stage + sub * kTokBox + k16 * 32, 16, 1024, kLayoutSw128);
                                mma_pair_ts_f16(tmem + kColAcc, tmem + kColA + as * 32 + k16 * 8, bdesc, idesc,
                                                (cpos > 0 || k16 > 0) ? 1u : 0u);
                            }
                            tc_commit_pair(&bars->aempty[as], 3);
                            if (cpos == csubs - 1 || tsub == tile_subs - 1) {
                                tc_commit_pair(&bars->accfull, 3);
                                ++chunk;
                                cpos = 0;
                            } else {
                                ++cpos;
                            }
                        }
                        tc_commit_pair(&bars->empty[stage], 3);
                    }
                }
                // Let every issued MMA finish before either CTA can release TMEM or shared memory.
                tc_commit_pair(&bars->drain, 1);
                mbar_wait_cluster(&bars->drain, 0, p.status, abort, peer_abort);
            }
        }
    } else if (wg == 1) {
        setmaxnreg_dec<kRegsConv>();
        // ------------------------------------------------ int8 -> fp16 converters (A operand into TMEM)
        const int q = warp & 3;
        const int r = q * 32 + lane;  // TMEM lane = A row of this CTA's half
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t gs = 0, gsub = 0;
        bool ok = true;
        for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
            for (int kt = 0; kt < KT && ok; ++kt) {
                const uint32_t mstage = gs++;
                const int stage = (int)(mstage % kStages);
                const uint8_t *ws = wbuf + stage * kWStageBytes;
                ok = mbar_wait_cluster(&bars->full[stage], (mstage / kStages) & 1u, p.status, abort, peer_abort);
                if (!ok) break;
                for (int sub = 0; sub < kSubs; ++sub) {
                    const uint32_t my = gsub++;
                    const int astage = (int)(my % kAStages);
                    uint32_t a[32];
                    if (p.w_layout == W_KMAJOR) {
                        // Row r: 128 bytes, 128-byte swizzle (16-byte chunk c stored at c ^ (r & 7));
                        // this sub-step is the 64-byte half `sub` of the row.
                        const uint8_t *row = ws + r * 128;
                        uint4 v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            v[c] = *reinterpret_cast<const uint4 *>(row + (((4 * sub + c) ^ (r & 7)) * 16));
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            s8x4_to_f16x4(v[c].x, a[8 * c + 0], a[8 * c + 1]);
                            s8x4_to_f16x4(v[c].y, a[8 * c + 2], a[8 * c + 3]);
                            s8x4_to_f16x4(v[c].z, a[8 * c + 4], a[8 * c + 5]);
                            s8x4_to_f16x4(v[c].w, a[8 * c + 6], a[8 * c + 7]);
                        }
                    } else {
                        // Box [128 contraction rows][128 output columns], 128-byte swizzle:
                        // byte (kr, r) at kr*128 + 16*((r >> 4) ^ (kr & 7)) + (r & 15).
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int kr = sub * kSub + 2 * j;
                            const uint32_t b0 = ws[kr * 128 + 16 * ((r >> 4) ^ (kr & 7)) + (r & 15)];
                            const uint32_t b1 = ws[(kr + 1) * 128 + 16 * ((r >> 4) ^ ((kr + 1) & 7)) + (r & 15)];
                            a[j] = s8pair_to_f16x2(b0 | (b1 << 16));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->empty[stage]);
                    ok = mbar_wait_cluster(&bars->aempty[astage], ((my / kAStages) & 1u) ^ 1u, p.status, abort,
                                           peer_abort);
                    if (!ok) break;
                    tc_fence_after();
                    tmem_st32(lane_addr + kColA + astage * 32, a);
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&bars->afull[astage]), 0));
                }
            }
        }
    } else {
        setmaxnreg_inc<kRegsEpi>();
        pdl_wait();  // scales, L1 sums and the output: only after the preceding kernel completed
        // ------------------------------------------------ chunk plan (epilogue warps, once)
        // Every partial sum of token m's products with int8 weights (|w| <= 128) over a set of K
        // indices is bounded by 128 * sum |q[m][k]| over that set.  A chunk of 2^j aligned 1024-long
        // blocks is therefore exact in fp32 when that bound stays within 2^24 -- block sums of at most
        // 2^17 -- for every token of the tile.  Level 0 (one block) holds for any int8 data; a tile
        // takes its longest level that holds.  Each epilogue thread checks whole token rows and ANDs
        // its verdict into the tile's bits.
        const int nb = (int)(p.K / 1024);
        const bool have_plan = p.row_l1 && p.K % 1024 == 0 && nb <= kPlanMaxBlocks;
        int plan_levels = 0;  // largest j with 2^j <= nb
        while ((2 << plan_levels) <= nb) ++plan_levels;
        if (have_plan) {
            const int et = (warp - 8) * 32 + lane;  // 0 .. 255
            const int64_t mmax = min(p.M, (int64_t)kPlanTiles * kBN);
            for (int64_t m = et; m < mmax; m += 32 * kEpiWarps) {
                int s16[kPlanMaxBlocks];
#pragma unroll
                for (int b2 = 0; b2 < kPlanMaxBlocks; ++b2) s16[b2] = b2 < nb ? __ldg(p.row_l1 + m * p.l1_ld + b2) : 0;
                uint32_t okb = 1u;  // level 0 always holds
#pragma unroll
                for (int j = 1, w = kPlanMaxBlocks / 2; w >= 1; ++j, w >>= 1) {
                    int mx = 0;
#pragma unroll
                    for (int i = 0; i < w; ++i) {
                        s16[i] = s16[2 * i] + s16[2 * i + 1];  // sums of aligned groups of 2^j blocks
                        mx = max(mx, s16[i]);
                    }
                    if (mx <= (1 << 17)) okb |= 1u << j;
                }
                // bit j for j <= plan_levels only if every level below also holds (longer chunks are unions)
                uint32_t pref = 0;
                for (int j = 0; j <= plan_levels && ((okb >> j) & 1u); ++j) pref |= 1u << j;
                atomicAnd(&bars->plan[m / kBN], pref);
            }
        }
        named_bar_sync(1, 32 * kEpiWarps);  // every epilogue thread's verdicts are in
        if (warp == 8 && lane == 0) mbar_arrive(&bars->plan_ready);  // publish the plan to the MMA issuer
        // ------------------------------------------------ epilogue: drain chunks, write outputs
        const int q = warp & 3;
        const int h = (warp >> 2) & 1;  // token half of the tile
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + kColAcc + h * 128;
        uint32_t chunk = 0;
        bool ok = true;
        for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
            int64_t n0, m0;
            tile_coords(t, m_tiles, n_tiles, p.wfast, &n0, &m0);
            n0 += kBM * rank;                      // this CTA's output columns
            const int64_t n = n0 + q * 32 + lane;  // output column owned by this thread
            const bool n_ok = n < p.N;
            float ws = 0.0f, bias = 0.0f;
            if (n_ok && p.epi == EPI_DEQUANT_BF16) {
                ws = n < p.n_split ? __ldg(p.w_scale0 + n) : __ldg(p.w_scale1 + (n - p.n_split));
                if (p.bias) bias = __bfloat162float(p.bias[n]);
            }
            float xs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // x_scale of rows m0 + 128h + 32g + lane
            if (p.epi != EPI_ACC_I32) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int64_t m = m0 + 128 * h + 32 * g + lane;
                    if (m < p.M) xs4[g] = __ldg(p.x_scale + m);
                }
            }
            int32_t tot[128];  // exact running sums for this thread's 128 token columns
#pragma unroll
            for (int i = 0; i < 128; ++i) tot[i] = 0;
            const int csubs =
                tile_chunk_subs(bars->plan, p, tile_token_index(t, m_tiles, n_tiles, p.wfast), tile_subs);
            const int nchunks = (tile_subs + csubs - 1) / csubs;
            for (int c = 0; c < nchunks; ++c) {
                ok = mbar_wait_cluster(&bars->accfull, chunk & 1u, p.status, abort, peer_abort);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t rr[32];
                    tmem_ld32(lane_addr + 32 * j, rr);
                    tc_wait_ld();
                    add_exact_totals(tot + 32 * j, rr);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(lead_accempty);  // this warp is done with the accumulator
                ++chunk;
            }
            if (!ok) break;
            // Debug builds: the pair tile's corner lies inside the output (TMA clips the rest; the second
            // CTA's 128 columns may lie wholly past N in the last tile).
            if (!(GBQ_IN_RANGE(p.status, m0, 1, p.M) && GBQ_IN_RANGE(p.status, n0 - kBM * rank, 1, p.N))) continue;
            if (p.use_tma_out) {
                uint8_t *mine = obuf + (uint32_t)(warp - 8) * 2 * kOutBlock;
                if (p.epi == EPI_ACC_I32)
                    store_tile_tma<16, EPI_ACC_I32>(p, tot, xs4, mine, h, q, lane, n0, m0, ws, bias);
                else if (p.epi == EPI_DEQUANT_BF16)
                    store_tile_tma<32, EPI_DEQUANT_BF16>(p, tot, xs4, mine, h, q, lane, n0, m0, ws, bias);
                else
                    store_tile_tma<16, EPI_ROWSCALE_F32>(p, tot, xs4, mine, h, q, lane, n0, m0, ws, bias);
                continue;
            }
            // Write token rows m0 + 128h + 32j + i of output column n.
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t mb = m0 + 128 * h + 32 * j;
                const float xs_l = xs4[j];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float xs = __shfl_sync(0xffffffffu, xs_l, i);
                    const int64_t m = mb + i;
                    if (!n_ok || m >= p.M) continue;
                    const int32_t acc = tot[32 * j + i];
                    if (p.epi == EPI_ACC_I32) {
                        int32_t *o = reinterpret_cast<int32_t *>(p.out) + m * p.ld_out + n;
                        if (p.reduce_out)
                            atomicAdd(o, acc);
                        else
                            *o = acc;
                    } else if (p.epi == EPI_DEQUANT_BF16) {
                        const float tv = __fmul_rn(__int2float_rn(acc), xs);
                        const float y = __fmaf_rn(tv, ws, bias);
                        reinterpret_cast<__nv_bfloat16 *>(p.out)[m * p.ld_out + n] = __float2bfloat16_rn(y);
                    } else {
                        reinterpret_cast<float *>(p.out)[m * p.ld_out + n] = __fmul_rn(__int2float_rn(acc), xs);
                    }
                }
            }
        }
    }

    if (wg >= 2 && lane == 0 && p.use_tma_out) tma_store_wait_all<0>();  // smem must outlive the stores
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // no CTA leaves while its peer's MMAs, arrivals or stores may touch it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// Co-resident CTA pairs on the current device (cached).
int max_pairs_for_device(int num_sms) {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
    if (cached[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, i8gemm_kernel, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = num_sms / 2;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace

int i8gemm_max_pairs(int num_sms) { return max_pairs_for_device(num_sms); }

int launch_i8gemm(const I8GemmProblem &q, cudaStream_t st) {
    Params p;  // host staging; copied into the launch's parameter buffer
    memset(&p, 0, sizeof(p));
    int rc;
    // Activations: fp16 [M][K], box 64 x 128, 128-byte swizzle (each CTA stages its 128-token half).
    if (q.reduce_out && q.epi != EPI_ACC_I32) return gbq_fail(GBQ_EINVAL, "int8 GEMM: reduce_out needs EPI_ACC_I32");
    const int64_t ld_b = q.ld_b > 0 ? q.ld_b : q.K;
    rc = encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, q.b_f16, (uint64_t)q.K, (uint64_t)q.M,
                        (uint64_t)ld_b * 2, kSub, kBNHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    for (int s = 0; s < 2; ++s) {
        const int8_t *w = s ? q.w1 : q.w0;
        const int64_t rows = s ? q.w_rows_total1 : q.w_rows_total0;
        CUtensorMap *tm = s ? &p.tm_w1 : &p.tm_w0;
        if (q.w_layout == W_KMAJOR)  // [rows][K], box 128 B x 128 rows, 128-byte swizzle
            rc = encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)q.K, (uint64_t)rows,
                                (uint64_t)q.ld_w, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
        else  // [K rows][ld_w]: box 128 B (output columns) x kBK rows, 128-byte swizzle
            rc = encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)q.N, (uint64_t)rows,
                                (uint64_t)q.ld_w, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc) return rc;
    }
    // Output through TMA when its row stride allows (16-byte multiple) and it lies in device memory; an
    // output in pinned host memory (written straight over the chip-to-chip link) takes plain stores.
    {
        const uint32_t esz = q.epi == EPI_DEQUANT_BF16 ? 2u : 4u;
        const CUtensorMapDataType dt = q.epi == EPI_DEQUANT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : q.epi == EPI_ACC_I32    ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        bool out_device = false;
        cudaPointerAttributes pa{};
        if (cudaPointerGetAttributes(&pa, q.out) == cudaSuccess)
            out_device = pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged;
        else
            (void)cudaGetLastError();  // an unknown pointer: plain stores
        p.use_tma_out = (out_device && (q.ld_out * esz) % 16 == 0 && ((uintptr_t)q.out & 15) == 0) ? 1 : 0;
        if (p.use_tma_out) {
            rc = encode_tmap_2d(&p.tm_out, dt, q.out, (uint64_t)q.N, (uint64_t)q.M, (uint64_t)q.ld_out * esz, 32,
                                kOutBlock / (32 * esz), CU_TENSOR_MAP_SWIZZLE_NONE);
            if (rc) return rc;
        }
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
    p.row_l1 = q.row_l1;
    p.l1_ld = q.l1_ld > 0 ? q.l1_ld : q.K / 1024;
    p.reduce_out = q.reduce_out;
    p.wfast = 2 * q.M > q.N ? 1 : 0;  // fp16-coded tokens: 2 M bytes per unit of K against N weight bytes
    p.status = q.status;
    p.w_layout = q.w_layout;
    p.epi = q.epi;

    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(i8gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
        // The per-warpgroup register split (setmaxnreg) must fit in what the block is launched with.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, i8gemm_kernel);
        if (e != cudaSuccess) return gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
        if ((long)fa.numRegs * kThreads < 128L * (kRegsWG0 + kRegsConv + 2 * kRegsEpi))
            return gbq_fail(GBQ_ECUDA, "int8 GEMM: register split exceeds the launch allocation");
        attr = true;
    }
    const int64_t tiles = ((q.M + kBN - 1) / kBN) * ((q.N + kPairM - 1) / kPairM);
    int64_t pairs_max = max_pairs_for_device(q.num_sms);
    if (q.max_pairs > 0 && q.max_pairs < pairs_max) pairs_max = q.max_pairs;
    const int grid = 2 * (int)(tiles < pairs_max ? tiles : pairs_max);
    prof_begin(1, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute lattr[1];
    lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    lattr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = lattr;
    cfg.numAttrs = q.pdl ? 1 : 0;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, i8gemm_kernel, p);
    if (le != cudaSuccess) {
        prof_end(st);
        return gbq_fail(GBQ_ECUDA, cudaGetErrorString(le));
    }
    prof_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return gbq_fail(GBQ_ECUDA, cudaGetErrorString(e));
    return GBQ_OK;
}

}  // namespace gbq
