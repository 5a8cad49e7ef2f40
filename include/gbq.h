/*
 * gbq.h -- C ABI of libgbq: rotated INT8 linear layers, a SwiGLU FFN and the
 * input-gradient backward, as hand-written CUDA for GB300 (sm_103a).
 *
 * The method is the one on the PyPI page "xpu-kernels 0.2.0"
 * (pypi.org/project/xpu-kernels/0.2.0): ConvRot Kronecker-Hadamard rotation
 * of the activation, per-token INT8 quantization, an int8 x int8 -> int32
 * GEMM against a weight stored pre-rotated, and a dequant epilogue.
 *
 * Conventions (shared by every entry point):
 *   - All tensors are row-major and contiguous unless a leading dimension
 *     (ld_*) is given.  Sizes are int64_t.  bf16 tensors are passed as
 *     void* holding IEEE bfloat16 values.
 *   - Every pointer is a DEVICE pointer owned by the caller (for example a
 *     torch tensor's data_ptr()).  The library never allocates, frees or
 *     keeps a reference to caller memory after the call returns, and no
 *     entry point allocates device memory (all scratch comes from the
 *     caller's `workspace`, sized by gbq_workspace_size()).
 *   - Pointers must be 16-byte aligned; K (the contraction length) must be
 *     a multiple of 64 for GEMM entry points.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work; nothing is synchronised.  Use gbq_sync().
 *   - Return value: 0 on success, a negative GBQ_E* code otherwise, with a
 *     human-readable message in gbq_last_error() (thread-local).  On an
 *     argument error nothing is launched.  No kernel traps: a device-side
 *     wait that exceeds its iteration limit records a code that
 *     gbq_device_status() returns.
 *
 * Rotation descriptor: R = I_groups (x) (H_a (x) H_b) / sqrt(a*b) with
 * K = a*b*groups.  H_n = H4^(x)j for n = 4^j (H4 as printed in the page's
 * "Algorithm: fused ConvRot rotation"), H_n = H2 (x) H4^(x)j for n = 2*4^j
 * (H2 on the most significant index bit; the page is silent there).
 * a = b = 1 is the identity.  Any powers of two a, b >= 1 with a*b*groups = K
 * are accepted (a != b included).  a = b in {16, 32, 64, 128} with at most
 * 64, 32, 8, 2 groups run the square kernels; every other shape runs one
 * generic kernel, which needs K % 16 == 0 and K <= 49152 (GBQ_ENOTSUP
 * otherwise).  Where both could serve a descriptor they give identical values:
 * the levels of a descriptor (H4/2 on a base-4 digit of the group index, or an
 * unnormalised H2 on one bit, whose factor is removed once at the end: an exact
 * halving for two of them, a multiplication by fl(sqrt(1/2)) for one) run in one
 * fixed order with the same fp32 operations in every kernel.
 * R is symmetric and orthogonal, so rotating x and the weight rows by the
 * same R leaves x @ W^T unchanged.
 */
#ifndef GBQ_H
#define GBQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gbq_rot {
    int32_t a;      /* Hadamard factor on the high index part (power of two) */
    int32_t b;      /* Hadamard factor on the low, contiguous index part     */
    int32_t groups; /* number of contiguous blocks of a*b columns            */
} gbq_rot;

#define GBQ_OK 0
#define GBQ_EINVAL (-22)      /* bad argument: null/misaligned pointer, bad size, bad rotation */
#define GBQ_ENOSPC (-28)      /* workspace below the minimum (see gbq_workspace_size) */
#define GBQ_ENODEV (-19)      /* no usable sm_103 device */
#define GBQ_ECUDA (-5)        /* a CUDA runtime call or launch failed */
#define GBQ_ENOTSUP (-95)     /* valid but unsupported combination (e.g. rotation shape) */

/* Device-status bits reported by gbq_device_status(). */
#define GBQ_DEV_WAIT_TIMEOUT 0x1u /* an mbarrier wait hit its iteration limit */
#define GBQ_DEV_BOUNDS 0x2u       /* debug build only (GBQ_DEBUG_BOUNDS): a kernel computed a global   */
                                  /* memory access outside its tensor; the access was skipped       */

/* ---- library / device ------------------------------------------------ */

/* Selects nothing, checks that the current device is an sm_103 GPU and sets up
 * per-device state (device status word, driver entry point for TMA
 * descriptors, a second stream, and the 16 MiB static scratch of
 * gbq_linear_noalloc).  Called implicitly by every entry point; safe to call
 * again.  Call it once at start-up, before any stream capture. */
int gbq_init(void);
/* Name of the current device ("" before a successful gbq_init). */
const char *gbq_device_name(void);
/* Message for the last failing call on this host thread ("" if none). */
const char *gbq_last_error(void);
/* Waits for `stream`, then copies the device status word to *status and
 * clears it (0 = no kernel recorded an error since the last read). */
int gbq_device_status(void *stream, uint32_t *status);
/* cudaStreamSynchronize(stream), with the error mapped to a GBQ code. */
int gbq_sync(void *stream);

/* ---- workspace sizing ------------------------------------------------- */

enum gbq_op {
    GBQ_OP_LINEAR = 1,      /* gbq_linear / gbq_linear_acc (M,N,K)        */
    GBQ_OP_INT8_GEMM = 2,   /* gbq_int8_gemm (M,N,K)                     */
    GBQ_OP_FFN = 3,         /* gbq_ffn_fused (M, d=K, H)                 */
    GBQ_OP_LINEAR_DX_INT8 = 4 /* gbq_linear_dx_int8 (M,N,K)             */
};
/* Bytes of device workspace to pass to the entry point for `op` at these sizes.
 * The calls accept less, down to a minimum (linear / linear_acc / int8_gemm:
 * M*K*2 + M*4; ffn: those of x and of the hidden h plus g|u; linear_dx_int8:
 * M*N*2 + M*4 + M*K*4; each term rounded up to 256 bytes) and reject a smaller
 * workspace with GBQ_ENOSPC.  For linear, linear_acc, ffn and linear_dx_int8
 * the reported size adds, per quantized token row, one int32 per 1024-long block
 * of the contraction (the sum of the row's |codes| over the block): the int8
 * GEMM then gives each 256-token tile the longest exact fp32 chunk of 2^j
 * aligned blocks whose sums stay within 2^17 for all of its tokens; with the
 * minimum it uses 1024-long chunks throughout.  The results are identical. */
size_t gbq_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t H);

/* ---- rotate + quantize (activation side) ------------------------------ */

/*
 * q, x_scale = quantize(R x) per row ("Use from C": bf16 [M,K] -> int8 [M,K]
 * + fp32 [M] row scales; "Algorithm: fused ConvRot rotation").
 * x: bf16 [M,K].  q: int8 [M,K].  x_scale: fp32 [M].
 * Per row, in fp32: v = R x_m; amax = max|v|; s = amax/127;
 * q = clamp(rne(v/s), -127, 127); a row with s == 0 gets q = 0.
 */
int gbq_quantize_act(const void *x, int8_t *q, float *x_scale, int64_t M, int64_t K,
                     gbq_rot rot, void *stream);

/*
 * The activation fused into the quantizer ("Use from Python":
 * quantize_act(x2, act)): h = silu(g) * u in fp32 from bf16 g, u [M,H], then
 * q, h_scale = quantize(R h) as in gbq_quantize_act.
 */
int gbq_quantize_act_glu(const void *g, const void *u, int8_t *q, float *h_scale,
                         int64_t M, int64_t H, gbq_rot rot, void *stream);

/*
 * "dequant_act_quantize" ("Use from Python"): from the int32 gate and up
 * accumulators (leading dimension ld_acc), g = bf16(acc_g*x_scale*s_gate),
 * u = bf16(acc_u*x_scale*s_up), h = silu(g)*u, then quantize(R h).
 * Bit-identical to gbq_dequant + gbq_quantize_act_glu.
 */
int gbq_dequant_act_quantize(const int32_t *acc_g, const int32_t *acc_u, int64_t ld_acc,
                             const float *x_scale, const float *s_gate, const float *s_up,
                             int8_t *q, float *h_scale, int64_t M, int64_t H, gbq_rot rot,
                             void *stream);

/* ---- weight preparation ---------------------------------------------- */

/*
 * w8, w_scale = prepare_weight(w) ("Use from Python": bf16 [N,K] -> int8 +
 * fp32 [N], once).  The rotation is baked into the rows: W8 = quantize(W R^T)
 * with the same per-row quantizer as gbq_quantize_act.
 */
int gbq_prepare_weight(const void *w, int8_t *w8, float *w_scale, int64_t N, int64_t K,
                       gbq_rot rot, void *stream);

/* ---- linear layer ----------------------------------------------------- */

/*
 * acc = int8 GEMM of pre-quantized operands: acc[m,n] = sum_k q[m,k] w8[n,k]
 * (the page's torch._int_mm step).  q int8 [M,K], w8 int8 [N,K], acc int32
 * [M,N] with leading dimension ld_acc.  Exact.  Workspace: GBQ_OP_INT8_GEMM.
 */
int gbq_int8_gemm(const int8_t *q, const int8_t *w8, int32_t *acc, int64_t ld_acc,
                  int64_t M, int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                  void *stream);

/*
 * acc, x_scale = linear_acc(x, w8) ("Use from Python": int32 [M,N], no bf16
 * round trip).  x bf16 [M,K]; acc int32 [M,N] (ld_acc); x_scale fp32 [M].
 * Workspace: GBQ_OP_LINEAR.
 */
int gbq_linear_acc(const void *x, const int8_t *w8, int32_t *acc, int64_t ld_acc,
                   float *x_scale, int64_t M, int64_t N, int64_t K, gbq_rot rot,
                   void *workspace, size_t ws_bytes, void *stream);

/*
 * y = dequant(acc) ("API": out = acc * x_scale[m] * w_scale[n] + bias[n]).
 * acc int32 [M,N] (ld_acc), y bf16 [M,N] (ld_y; a column slice of a wider
 * output is allowed, the page's dequant_slice).  bias bf16 [N] or NULL.
 * Per element: t = fp32(acc) * x_scale[m]; y = bf16(fmaf(t, w_scale[n], bias[n])).
 */
int gbq_dequant(const int32_t *acc, int64_t ld_acc, const float *x_scale,
                const float *w_scale, const void *bias, void *y, int64_t ld_y,
                int64_t M, int64_t N, void *stream);

/*
 * y = linear(x, w8, w_scale, bias) ("Use from Python": bf16 [..,K] -> bf16
 * [..,N]); rotate+quantize, int8 GEMM and the dequant epilogue fused in the
 * GEMM.  Bit-identical to gbq_dequant(gbq_linear_acc(x)).  M = 1..16 runs a
 * GEMV (weight streaming): with the rotation inside for M <= 2 and a = b in
 * {16, 32, 64}, K <= 4096, and for every other descriptor (not the identity)
 * while M * K <= 8192; else over codes the rotation kernels write into the
 * workspace first (any descriptor, while M * K codes and four weight rows fit
 * in shared memory; at N = 4096: K <= 44032 at M = 1, 27520 at M = 4, 11008
 * at M = 16); larger M or K runs the GEMM (same values).  Workspace:
 * GBQ_OP_LINEAR.
 * At K = 4096 (a = b = 64, one group) the decode kernel is launched with
 * programmatic stream serialization: it may start while the kernel before it on
 * the stream is still running, but reads none of its inputs (x, w8, w_scale,
 * bias) before that kernel has completed, so x may be that kernel's output;
 * consecutive decode calls overlap (the next one's weight is fetched into L2
 * meanwhile).  Results do not depend on the overlap.
 * y may also be pinned host memory (cudaHostAlloc / cudaHostRegister): the
 * kernels then write it directly over the chip-to-chip link with plain
 * stores (no TMA).  On GB300 that is slower than a device y followed by a
 * copy, so it serves convenience, not speed.
 */
int gbq_linear(const void *x, const int8_t *w8, const float *w_scale, const void *bias,
               void *y, int64_t M, int64_t N, int64_t K, gbq_rot rot, void *workspace,
               size_t ws_bytes, void *stream);

/*
 * y = linear(x, w8, w_scale, bias) with no workspace argument: the same
 * computation and kernels as gbq_linear, with the scratch taken from a 16 MiB
 * static device array inside the library instead of a caller workspace.  It is
 * outside the method; it exists for callers that cannot allocate device memory
 * at the point of the call (a plugin inside a framework that owns all device
 * memory through its own pool, or a latency-critical loop that cannot afford
 * cudaMalloc's implicit synchronisation).
 * Limit: M*K*2 + M*4 bytes (each part rounded up to 256) must fit in 16 MiB,
 * e.g. M*K <= ~8.3 million; larger calls return GBQ_ENOSPC and launch nothing.
 * Sizes and the rotation are checked first, exactly as by gbq_linear.
 * The array is reserved, and its device address looked up (cudaGetSymbolAddress
 * with the device current), by the library's per-device set-up: gbq_init() or
 * the first call of any entry point on that device.  That set-up can therefore
 * fail with GBQ_ECUDA when the device lacks the 16 MiB; run it (gbq_init) at
 * start-up, before any stream capture.  Every device set up this way holds the
 * 16 MiB until the process exits; calls after the set-up allocate nothing.
 * All calls share the one array and it keeps the last call's contents (nothing
 * needs clearing: each call writes all the scratch it reads); calls that overlap
 * on the GPU -- on different streams, or from different host threads -- race
 * on it.
 */
int gbq_linear_noalloc(const void *x, const int8_t *w8, const float *w_scale, const void *bias,
                       void *y, int64_t M, int64_t N, int64_t K, gbq_rot rot, void *stream);

/* ---- SwiGLU FFN ------------------------------------------------------- */

/*
 * y = down(quantize(R_h(silu(gate(x)) * up(x)))) -- the page's fused MLP
 * (MUL_MAT + MUL_MAT + GLU/SWIGLU, then the down projection) with
 * "dequant_act_quantize" as its middle.
 * x bf16 [M,d]; wg8, wu8 int8 [H,d] with s_gate, s_up fp32 [H] (prepared with
 * rot_d); wd8 int8 [d,H] with s_down fp32 [d] (prepared with rot_h);
 * y bf16 [M,d].  No biases.  Bit-identical to the unfused chain
 * linear_acc -> dequant -> quantize_act_glu -> linear.
 * Workspace: GBQ_OP_FFN with (M, K=d, H).
 */
int gbq_ffn_fused(const void *x, const int8_t *wg8, const float *s_gate, const int8_t *wu8,
                  const float *s_up, const int8_t *wd8, const float *s_down, void *y,
                  int64_t M, int64_t d, int64_t H, gbq_rot rot_d, gbq_rot rot_h,
                  void *workspace, size_t ws_bytes, void *stream);

/* ---- backward dL/dx ---------------------------------------------------- */

/*
 * w = dequant_weight(w8, w_scale) ("The backward": recover W once).
 * w8 int8 [N,K], w_scale fp32 [N] -> w bf16 [N,K] = bf16((w8[n,:]*s[n]) R),
 * i.e. un-rotated back to the original basis (with rot = identity the
 * literal w8*s).  Memory-bound.
 */
int gbq_dequant_weight(const int8_t *w8, const float *w_scale, void *w, int64_t N, int64_t K,
                       gbq_rot rot, void *stream);

/*
 * dx = dy @ w ("The backward": bf16 GEMM, no transpose, no bias).
 * dy bf16 [M,N], w bf16 [N,K], dx bf16 [M,K]; fp32 accumulation.
 * N must be a multiple of 64, K a multiple of 16.
 */
int gbq_linear_dx(const void *dy, const void *w, void *dx, int64_t M, int64_t N, int64_t K,
                  void *stream);

/*
 * dx = linear_dx_int8(dy, w8, w_scale) ("The backward"): dy'[m,n] =
 * dy[m,n]*s[n]; per-row int8 quantize of dy' (no rotation) -> qd, t;
 * acc[m,k] = sum_n qd[m,n] w8[n,k] (exact); dx = bf16((fp32(acc)*t[m]) R).
 * dy bf16 [M,N]; w8 int8 [N,K]; w_scale fp32 [N]; dx bf16 [M,K].
 * Workspace: GBQ_OP_LINEAR_DX_INT8.
 */
int gbq_linear_dx_int8(const void *dy, const int8_t *w8, const float *w_scale, void *dx,
                       int64_t M, int64_t N, int64_t K, gbq_rot rot, void *workspace,
                       size_t ws_bytes, void *stream);

/* ---- rotate-only bf16 path --------------------------------------------- */

/*
 * xr = bf16(R x) ("Use from C": the BF16 path needs only the rotation).
 * x, xr bf16 [M,K].
 */
int gbq_rotate_bf16(const void *x, void *xr, int64_t M, int64_t K, gbq_rot rot, void *stream);

/*
 * y = x @ w^T + bias: the bf16 linear layer of the rotate-only path ("Use from
 * C": the BF16 comparator rotates the activation with gbq_rotate_bf16 and
 * multiplies it by the weight stored pre-rotated in bf16, w = bf16(W R); since
 * R is orthogonal, (x R)(W R)^T = x W^T up to the bf16 roundings).
 * x bf16 [M,K] (activation, K contiguous); w bf16 [N,K] (K contiguous);
 * bias bf16 [N] or NULL; y bf16 [M,N].  fp32 accumulation on the tensor cores,
 * bias added in fp32, one rounding to bf16.  K must be a multiple of 64; M >= 0
 * (M = 0 launches nothing), N >= 1 (any N; rows of y start 16-byte aligned only
 * when N % 8 == 0, otherwise the epilogue stores element by element).
 * x, w, y must be 16-byte aligned; bias needs bf16 alignment only.  All buffers
 * caller-owned; nothing is allocated.
 */
int gbq_linear_bf16(const void *x, const void *w, const void *bias, void *y, int64_t M, int64_t N,
                    int64_t K, void *stream);

/* ---- kernel timing ------------------------------------------------------ */

/* Kernel classes for gbq_prof_read(). */
enum gbq_kernel {
    GBQ_K_ROTATE = 0,   /* rotate(+quantize) kernels            */
    GBQ_K_I8GEMM = 1,   /* exact int8 tensor-core GEMM          */
    GBQ_K_BF16GEMM = 2, /* bf16 tensor-core GEMMs (linear_dx,   */
                        /* linear_bf16)                         */
    GBQ_K_GEMV = 3,     /* decode GEMV                          */
    GBQ_K_ELEMWISE = 4  /* dequant / operand coding / scaling   */
};
/* on != 0: from now on every kernel launch of the library is bracketed by a
 * pair of CUDA events recorded on the launch's stream (up to 8192 launches;
 * later ones are not timed).  Clears the previous record.  The events are
 * created once per process on the first enable.  on == 0 stops recording. */
int gbq_prof_enable(int on);
/* Synchronises the recorded events and returns, for kernel class `kind`, the
 * number of timed launches and the sum of their durations in milliseconds. */
int gbq_prof_read(int kind, int *launches, double *total_ms);

#ifdef __cplusplus
}
#endif

#endif /* GBQ_H */
