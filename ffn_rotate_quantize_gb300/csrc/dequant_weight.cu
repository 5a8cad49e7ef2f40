// dequant_weight.cu -- dequant_weight for the H64 (x) H64 rotation (4096 columns per group).
//
// What it computes (PyPI page "xpu-kernels 0.2.0", "The backward: dL/dx,
// weight-only"): the recovered weight in the original basis,
//     W_hat[n, :] = bf16((W8[n, :] * s[n]) R),   R = (H64 (x) H64) / 64 = H4^(x)6 / 64,
// per 4096-long group of a row (the rotation is symmetric, so x R = R x).
//
// Why integer-exact: the unnormalised transform H4^(x)6 has entries +-1, so it
// maps a row of int8 codes to sums of 4096 signed integers of magnitude <= 127.
// Every partial sum of every level stays below 127 * 4096 < 2^24 and is exact
// in fp32 whatever the level order, so the kernel transforms the codes exactly
// and rounds once at the end: W_hat = bf16(fl(v * fl(s[n] / 64))).  That is
// the exact product (W8 s) R rounded to fp32 and then to bf16 (s / 64 is exact
// for every normal s).
//
// Layout: one warp per 4096-long group row at a time (persistent warps stride
// over the rows; a CTA is one warp, so the tile exchange needs only __syncwarp).
// Index bits of an element: X[i][j], element 64 i + j, base-4 digits j01 j23
// j45 i01 i23 i45; lane L holds 128 values.
//   pass 1: the 16-byte chunks L + 32 c (c = 0..7): registers {j0..j3, i3..i5},
//     lanes {j4, j5, i0..i2}; levels j01 (one dp4a per output: the four signed
//     bytes of a word are one base-4 digit), j23 and i45 on packed fp32 pairs;
//     128-bit stores into a 64 x 64 fp32 shared tile.
//   pass 2: registers {j0, j4, j5, i0..i3} (pairs over j0), lanes {j1..j3,
//     i4, i5}: 64-bit tile loads; levels j45, i01, i23; scale; bf16 pairs
//     stored with 32-bit stores (a warp writes four 32-byte runs per store).
// The tile's 16-byte chunks are XOR-swizzled so both passes are free of bank
// conflicts.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace gbq {
namespace {

constexpr int kDqwMinBlocks = 12;  // one-warp CTAs: twelve rows in flight per SM (192 KB of tiles)
constexpr int kDqwK = 4096;
// dp4a accumulator: the int32 result's bits read as fp32 are 1.5 * 2^23 + v for |v| < 2^22.
constexpr int kMagicBits = 0x4B400000;
constexpr float kMagic = 12582912.0f;
// Rows of the printed 4-point factor H4 = J - 2 antidiag as four signed bytes (byte b = H4[a][b]).
constexpr int kH4Row0 = (int)0xFF010101u, kH4Row1 = 0x01FF0101, kH4Row2 = 0x0101FF01, kH4Row3 = 0x010101FF;

// H4 on four pairs whose lanes are independent: out_a = s - 2 x_(3-a), s = x0 + x1 + x2 + x3.
__device__ __forceinline__ void h4_pairs(float2 &x0, float2 &x1, float2 &x2, float2 &x3) {
    const float2 s = __fadd2_rn(__fadd2_rn(x0, x1), __fadd2_rn(x2, x3));
    const float2 m2 = make_float2(-2.0f, -2.0f);
    const float2 y0 = __ffma2_rn(x3, m2, s);
    const float2 y1 = __ffma2_rn(x2, m2, s);
    const float2 y2 = __ffma2_rn(x1, m2, s);
    const float2 y3 = __ffma2_rn(x0, m2, s);
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
}

// Hint: bring [src, src + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Word offset (fp32 units) of X[i][j] in the swizzled tile.
__device__ __forceinline__ int dqw_tile_off(int i, int j) {
    const int c = j >> 2;
    const int pc = c ^ ((c >> 3) << 1) ^ ((i & 1) | (((i >> 4) & 1) << 2));
    return i * 64 + pc * 4 + (j & 3);
}

__device__ __forceinline__ float2 dp4a_pair(uint32_t w, int ra, int rb) {
    return make_float2(__int_as_float(__dp4a((int)w, ra, kMagicBits)), __int_as_float(__dp4a((int)w, rb, kMagicBits)));
}

__global__ void __launch_bounds__(32, kDqwMinBlocks) dqw64_kernel(const int8_t *__restrict__ w8,
                                                                  const float *__restrict__ w_scale,
                                                                  __nv_bfloat16 *__restrict__ out, int64_t rows,
                                                                  int groups, unsigned int *status) {
    __shared__ __align__(16) float tile[64 * 64];
    const int L = threadIdx.x;
    int64_t row = blockIdx.x;
    if (row >= rows) return;
    if (L == 0) bulk_prefetch_l2(w8 + row * kDqwK, kDqwK);
    const float2 unbias = make_float2(-kMagic, -kMagic);
    for (; row < rows; row += gridDim.x) {
        const int64_t next = row + gridDim.x;
        if (L == 0 && next < rows) bulk_prefetch_l2(w8 + next * kDqwK, kDqwK);  // the next row waits in L2
        uint4 ld[8];
        const uint4 *src = reinterpret_cast<const uint4 *>(w8 + row * kDqwK);
        const bool row_ok = GBQ_IN_RANGE(status, row * kDqwK, kDqwK, rows * kDqwK);
#pragma unroll
        for (int c = 0; c < 8; ++c) ld[c] = row_ok ? __ldcs(src + L + 32 * c) : make_uint4(0u, 0u, 0u, 0u);
        const float f = __fmul_rn(__ldg(w_scale + row / groups), 0.015625f);
        // ---- pass 1: level j01 (dp4a), j23 (over the words of a chunk), i45 (over the chunks) ----
        float2 p[8][4][2];  // [c = i3 + 2 i45][q = j23][h]: pair (a = 2h, 2h + 1), a = j01
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t wd[4] = {ld[c].x, ld[c].y, ld[c].z, ld[c].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                p[c][q][0] = __fadd2_rn(dp4a_pair(wd[q], kH4Row0, kH4Row1), unbias);
                p[c][q][1] = __fadd2_rn(dp4a_pair(wd[q], kH4Row2, kH4Row3), unbias);
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) h4_pairs(p[c][0][h], p[c][1][h], p[c][2][h], p[c][3][h]);
#pragma unroll
        for (int i3 = 0; i3 < 2; ++i3)
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int h = 0; h < 2; ++h) h4_pairs(p[i3][q][h], p[i3 + 2][q][h], p[i3 + 4][q][h], p[i3 + 6][q][h]);
        __syncwarp();  // the previous row's pass-2 loads are done
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int i = (L >> 2) + 8 * c;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 16 * (L & 3) + 4 * q;
                *reinterpret_cast<float4 *>(tile + dqw_tile_off(i, j)) =
                    make_float4(p[c][q][0].x, p[c][q][0].y, p[c][q][1].x, p[c][q][1].y);
            }
        }
        __syncwarp();
        // ---- pass 2: registers {j0, j45, i0..i3}; pairs over j0 ----
        const int j13 = 2 * (L & 7), i45 = L >> 3;
        float2 v[4][16];  // [j45][i03]: pair (j0 = 0, 1)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int r = 0; r < 16; ++r)
                v[jj][r] = *reinterpret_cast<const float2 *>(tile + dqw_tile_off(r + 16 * i45, j13 + 16 * jj));
#pragma unroll
        for (int r = 0; r < 16; ++r) h4_pairs(v[0][r], v[1][r], v[2][r], v[3][r]);  // j45
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int i23 = 0; i23 < 4; ++i23)
                h4_pairs(v[jj][4 * i23], v[jj][4 * i23 + 1], v[jj][4 * i23 + 2], v[jj][4 * i23 + 3]);  // i01
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int i01 = 0; i01 < 4; ++i01)
                h4_pairs(v[jj][i01], v[jj][i01 + 4], v[jj][i01 + 8], v[jj][i01 + 12]);  // i23
        if (!row_ok) continue;
        uint32_t *orow = reinterpret_cast<uint32_t *>(out + row * kDqwK);
        const float2 ff = make_float2(f, f);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const __nv_bfloat162 b = __float22bfloat162_rn(__fmul2_rn(v[jj][r], ff));
                orow[((r + 16 * i45) * 64 + j13 + 16 * jj) >> 1] = *reinterpret_cast<const uint32_t *>(&b);
            }
    }
}

}  // namespace

// W_hat for rotations with n = 64 (rows of `groups` 4096-long groups).  rows = N * groups.
cudaError_t launch_dequant_weight64(const int8_t *w8, const float *w_scale, void *out, int64_t N, int groups,
                                    int num_sms, cudaStream_t st, unsigned int *status) {
    const int64_t rows = N * groups;
    if (rows == 0) return cudaSuccess;
    static int per_sm = 0;
    if (per_sm == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dqw64_kernel, 32, 0);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorNotSupported;
    }
    const int64_t resident = (int64_t)per_sm * (num_sms > 0 ? num_sms : 1);
    const unsigned grid = (unsigned)(rows < resident ? rows : resident);
    prof_begin(0, st);
    dqw64_kernel<<<grid, 32, 0, st>>>(w8, w_scale, reinterpret_cast<__nv_bfloat16 *>(out), rows, groups, status);
    prof_end(st);
    return cudaGetLastError();
}

}  // namespace gbq
