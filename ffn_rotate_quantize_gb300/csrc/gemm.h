// gemm.h -- GEMM and elementwise launchers of libgbq (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gbq.h"

namespace gbq {

// Epilogues of the exact int8 GEMM.
enum EpiMode {
    EPI_ACC_I32 = 0,       // out int32 [M, ld_out]: the exact accumulator
    EPI_DEQUANT_BF16 = 1,  // out bf16: bf16(fmaf(fp32(acc) * x_scale[m], w_scale[n], bias[n]))
    EPI_ROWSCALE_F32 = 2,  // out fp32: fp32(acc) * x_scale[m]
};

// Orientation of the int8 weight operand.
enum WLayout {
    W_KMAJOR = 0,  // W8 [N][K]: output index n = W row, contraction along a row (the forward)
    W_NMAJOR = 1,  // W8 [Kc][N]: contraction over W rows, output index = W column (the dx route)
};

struct I8GemmProblem {
    const void *b_f16;        // activations as exact fp16 integers [M][K]
    const int8_t *w0;         // W source for output rows [0, n_split)
    const int8_t *w1;         // W source for output rows [n_split, N) (may equal w0 with n_split = N)
    int64_t ld_w;             // bytes between W rows
    int64_t w_rows_total0, w_rows_total1;  // rows of each source tensor (TMA bounds)
    int64_t M, N, K;
    int64_t n_split;
    int w_layout;
    int epi;
    void *out;
    int64_t ld_out;           // elements
    const float *x_scale;     // [M]
    const float *w_scale0;    // [n_split] (indexed by row within source 0)
    const float *w_scale1;    // [N - n_split]
    const void *bias;         // bf16 [N] or nullptr (EPI_DEQUANT_BF16)
    unsigned int *status;
    int num_sms;
    const int32_t *row_l1;    // optional [M][K/1024]: sum of |q| over each 1024-long block of a token row
    int pdl;                  // launch so the kernel may start while the preceding (quantizer) kernel runs:
                              // it reads the tokens, scales and L1 sums only after that kernel completes
    int64_t ld_b;             // elements between token rows of b_f16 (0: K)
    int64_t l1_ld;            // blocks between token rows of row_l1 (0: K / 1024)
    int max_pairs;            // at most this many co-resident CTA pairs (0: as many as the device holds)
    int reduce_out;           // EPI_ACC_I32 only: add the accumulator into out (exact int32 reduction)
                              // instead of storing it, so launches over parts of K can sum into one buffer
};

// Enqueue the exact int8 GEMM (tcgen05, fp16-coded operands, chunked fp32 -> int32).
int launch_i8gemm(const I8GemmProblem &p, cudaStream_t st);
// CTA pairs of the int8 GEMM that fit the current device at once.
int i8gemm_max_pairs(int num_sms);

// bf16 GEMM dx[M][K] = dy[M][N] @ w[N][K] (fp32 accumulation).
int launch_bf16_gemm_nn(const void *dy, const void *w, void *dx, int64_t M, int64_t N, int64_t K,
                        unsigned int *status, int num_sms, cudaStream_t st);
// bf16 GEMM y[M][N] = x[M][K] @ w[N][K]^T + bias[N] (fp32 accumulation and bias add; bias nullable).
int launch_bf16_gemm_tn(const void *x, const void *w, const void *bias, void *y, int64_t M, int64_t N, int64_t K,
                        unsigned int *status, int num_sms, cudaStream_t st);

// Decode GEMV with the rotation inside (M <= 2, K <= 4096; square n = 16, 32, 64 shapes, see launch_gemv):
// y[m][n] = dequant(sum_k q[m][k] w8[n][k]) from x rotated and quantized in the kernel.
// Returns GBQ_ENOTSUP (nothing launched) for shapes it does not cover.
int launch_gemv(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y, int64_t M,
                int64_t N, int64_t K, int logn, int groups, int num_sms, cudaStream_t st, unsigned int *status);

// Decode GEMV with the generic rotation inside (M <= 2; any descriptor of two or more levels, K <= 49152
// while the tile, the codes and four weight rows fit): the tokens are rotated with the generic rotation's
// level list in every CTA.  GBQ_ENOTSUP (nothing launched) when it does not fit.
bool gemv_gen_fits(int64_t M, int64_t N, int64_t K, int num_sms);
int launch_gemv_gen(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y, int64_t M,
                    int64_t N, int64_t K, int la, int lb, int num_sms, cudaStream_t st, unsigned int *status);

// GEMV (M <= 16) over tokens already quantized: codes int8 [M][K] and row scales fp32 [M] (e.g. in the
// workspace), y[m * ld_y + n] = dequant(sum_k codes[m][k] w8[n][k]).  Launched with programmatic stream
// serialization: it reads the codes and scales only after the preceding kernel completed, w8, w_scale and
// bias before.  GBQ_ENOTSUP (nothing launched) when it does not fit.
bool gemv_codes_fits(int64_t M, int64_t N, int64_t K, int num_sms);
int launch_gemv_codes(const int8_t *codes, const float *scales, const int8_t *w8, const float *w_scale,
                      const void *bias, void *y, int64_t ld_y, int64_t M, int64_t N, int64_t K, int num_sms,
                      cudaStream_t st, unsigned int *status);
// The same over the virtual weight [w8; w8b]: rows [0, n_split) from w8 / w_scale, rows [n_split, N) from
// w8b / w_scale_b (row n - n_split), so y[m][n] covers both (e.g. the FFN's gate | up in one launch).
int launch_gemv_codes2(const int8_t *codes, const float *scales, const int8_t *w8, const float *w_scale,
                       const int8_t *w8b, const float *w_scale_b, int64_t n_split, const void *bias, void *y,
                       int64_t ld_y, int64_t M, int64_t N, int64_t K, int num_sms, cudaStream_t st,
                       unsigned int *status);

// Elementwise helpers.
cudaError_t launch_dequant(const int32_t *acc, int64_t ld_acc, const float *xs, const float *ws, const void *bias,
                           void *y, int64_t ld_y, int64_t M, int64_t N, cudaStream_t st, unsigned int *status = nullptr);
cudaError_t launch_s8_to_f16(const int8_t *q, void *out, int64_t n, cudaStream_t st, unsigned int *status = nullptr);
cudaError_t launch_scale_rows_s8(const int8_t *w8, const float *s, void *w, int64_t N, int64_t K, cudaStream_t st,
                                 unsigned int *status = nullptr);

size_t gemm_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t H);       // minimum
size_t gemm_workspace_size_pref(int op, int64_t M, int64_t N, int64_t K, int64_t H);  // what gbq_workspace_size reports

// Launch timing hooks (abi.cu): bracket one kernel launch on stream st.
void prof_begin(int kind, cudaStream_t st);
void prof_end(cudaStream_t st);

// Shared with abi.cu.
int encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
int gbq_fail(int code, const char *msg);
// gbq_linear's size and rotation checks, then the device set-up (nothing else; no pointer is read).
int linear_args_check(const char *what, int64_t M, int64_t N, int64_t K, gbq_rot rot);
// Per-device set-up of gbq_linear_noalloc's static scratch (noalloc.cu), run by the library's device
// set-up with `dev` current: looks up the array's device address once.
int noalloc_setup_current(int dev);

}  // namespace gbq
