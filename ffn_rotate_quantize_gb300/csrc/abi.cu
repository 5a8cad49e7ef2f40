// abi.cu -- the extern "C" boundary of libgbq: argument checks, error reporting,
// per-device set-up and dispatch to the kernels.  No entry point allocates
// device memory; scratch comes from the caller's workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/gbq.h"
#include "gemm.h"
#include "kernels.h"

using namespace gbq;

namespace {

thread_local char g_err[1024] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    if (e == cudaErrorNotSupported) return fail(GBQ_ENOTSUP, "%s: unsupported shape or rotation for this kernel", what);
    return fail(GBQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The device status word: kernels OR GBQ_DEV_* bits into it.
__device__ unsigned int g_status_word;

struct DevState {
    // Set (release) once every other field is in place; read (acquire) without the lock.
    std::atomic<bool> ready{false};
    unsigned int *status = nullptr;
    int sms = 0;
    char name[256] = "";
    // A second stream and fork/join events for work the library splits over two streams (created once);
    // fork_mu keeps one call's record/wait sequence from interleaving with another's.
    cudaStream_t aux = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_entry = nullptr, ev_zero = nullptr;
    std::mutex fork_mu;
};
constexpr int kMaxDevices = 64;
DevState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
thread_local char g_name_out[256] = "";

int init_current(DevState **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GBQ_ENODEV, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(GBQ_ENODEV, "device index %d out of range", dev);
    DevState &d = g_dev[dev];
    if (d.ready.load(std::memory_order_acquire)) {
        *out = &d;
        return GBQ_OK;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        if (!(prop.major == 10 && prop.minor == 3))
            return fail(GBQ_ENODEV, "device %d (%s) is sm_%d%d; libgbq is built for sm_103a only", dev, prop.name,
                        prop.major, prop.minor);
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(GBQ_ECUDA, "cuTensorMapEncodeTiled entry point unavailable");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        // The static scratch of gbq_linear_noalloc: its module is loaded (and its memory reserved)
        // here, at the device's set-up, not inside a later call.
        int rc = noalloc_setup_current(dev);
        if (rc != GBQ_OK) return rc;
        e = cudaStreamCreateWithFlags(&d.aux, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_join, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_entry, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_zero, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "creating the library's auxiliary stream");
        d.status = static_cast<unsigned int *>(p);
        d.sms = prop.multiProcessorCount;
        snprintf(d.name, sizeof(d.name), "%s", prop.name);
        d.ready.store(true, std::memory_order_release);
    }
    *out = &d;
    return GBQ_OK;
}

bool a16(const void *p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

#define REQUIRE(cond, ...)                                   \
    do {                                                     \
        if (!(cond)) return fail(GBQ_EINVAL, __VA_ARGS__);   \
    } while (0)

#define INIT(dptr)                           \
    DevState *dptr = nullptr;                \
    do {                                     \
        int rc_ = init_current(&dptr);       \
        if (rc_ != GBQ_OK) return rc_;       \
    } while (0)

int ilog2(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

// A validated rotation descriptor and the kernel family that serves it.
struct RotSel {
    int logn;    // 0: identity; 4..7: a = b = 2^logn, the square kernels; -1: the generic kernel
    int la, lb;  // log2 a, log2 b
    int a, b, groups;
};

// Validates a rotation descriptor for row length K.  Any powers of two a, b >= 1 with a*b*groups = K
// are accepted.  a = b in {16, 32, 64, 128} with few enough groups for one CTA per row go to the
// square kernels; every other shape (a != b, factors 2..8 or above 128, many groups) to the generic
// kernel, which needs K % 16 == 0 and K <= kGenMaxK (GBQ_ENOTSUP otherwise).  Both produce the same
// values for a descriptor they can both serve.
int check_rot(gbq_rot r, int64_t K, RotSel *sel) {
    REQUIRE(r.a >= 1 && r.b >= 1 && r.groups >= 1, "rotation (a=%d, b=%d, groups=%d): all must be >= 1", r.a, r.b,
            r.groups);
    REQUIRE((r.a & (r.a - 1)) == 0 && (r.b & (r.b - 1)) == 0, "rotation a=%d, b=%d: must be powers of two", r.a, r.b);
    REQUIRE((int64_t)r.a * r.b * r.groups == K, "rotation a*b*groups = %lld != K = %lld",
            (long long)r.a * r.b * r.groups, (long long)K);
    sel->la = ilog2(r.a);
    sel->lb = ilog2(r.b);
    sel->a = r.a;
    sel->b = r.b;
    sel->groups = r.groups;
    if (r.a == 1 && r.b == 1) {
        sel->logn = 0;
        return GBQ_OK;
    }
    if (r.a == r.b && sel->la >= 4 && sel->la <= 7 &&
        (int64_t)rotq_row_threads(sel->la, 1) * r.groups <= (sel->la >= 6 ? 256 : 512)) {
        sel->logn = sel->la;
        return GBQ_OK;
    }
    if (!rotg_fits(K))
        return fail(GBQ_ENOTSUP,
                    "rotation (a=%d, b=%d, groups=%d) over K=%lld: this shape is served for K %% 16 == 0 and "
                    "K <= %lld only",
                    r.a, r.b, r.groups, (long long)K, (long long)kGenMaxK);
    sel->logn = -1;
    return GBQ_OK;
}

// Rotate(+quantize) rows of an input through the right kernel.
int run_rotq(const char *what, const RotSel &rot, int in_kind, int out_kind, RotArgs a, cudaStream_t st) {
    cudaError_t e;
    DevState *d = nullptr;
    int rc = init_current(&d);
    if (rc != GBQ_OK) return rc;
    a.status = d->status;
    a.num_sms = d->sms;
    if (rot.logn == 0 && in_kind == IN_BF16 && out_kind != OUT_BF16) {
        REQUIRE(a.K % 8 == 0, "%s: identity rotation needs K %% 8 == 0 (K=%lld)", what, (long long)a.K);
        IdArgs ia{a.in0, nullptr, a.ld_in, a.out, a.out_scale, a.M, a.K, nullptr, d->status, d->sms};
        e = launch_quant_identity(out_kind, ia, st);
    } else if (rot.logn > 0) {
        a.G = rot.groups;
        if (out_kind == OUT_BF16)
            e = launch_rotb(rot.logn, in_kind, a, st);
        else
            e = launch_rotq(rot.logn, in_kind, out_kind, a, st);
        // A shape the square kernels cannot stage (shared memory): the generic kernel gives the same values.
        if (e == cudaErrorNotSupported && rotg_fits(a.K)) e = launch_rotg(in_kind, out_kind, a, rot.la, rot.lb, st);
    } else {
        e = launch_rotg(in_kind, out_kind, a, rot.la, rot.lb, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    return GBQ_OK;
}

}  // namespace

// Tensor-map encoder shared with the GEMM launchers (gemm.h).
namespace gbq {
int encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    if (!g_encode) return fail(GBQ_ECUDA, "tensor-map encoder not initialised");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GBQ_ECUDA, "cuTensorMapEncodeTiled failed (%d) for %llux%llu, stride %llu, box %ux%u", (int)r,
                    (unsigned long long)inner, (unsigned long long)outer, (unsigned long long)row_stride_bytes,
                    box_inner, box_outer);
    return GBQ_OK;
}
int gbq_fail(int code, const char *msg) { return fail(code, "%s", msg); }

// ---- launch timing: library-owned event pairs, recorded only while enabled.
namespace {
constexpr int kProfMax = 8192;
bool g_prof_on = false;
int g_prof_n = 0;
int g_prof_kind[kProfMax];
cudaEvent_t g_prof_ev[2][kProfMax];
bool g_prof_created = false;
std::mutex g_prof_mu;
}  // namespace

void prof_begin(int kind, cudaStream_t st) {
    if (!g_prof_on) return;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (g_prof_n >= kProfMax) return;
    g_prof_kind[g_prof_n] = kind;
    cudaEventRecord(g_prof_ev[0][g_prof_n], st);
}
void prof_end(cudaStream_t st) {
    if (!g_prof_on) return;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (g_prof_n >= kProfMax) return;
    cudaEventRecord(g_prof_ev[1][g_prof_n], st);
    ++g_prof_n;
}
}  // namespace gbq

// ============================================================ entry points
extern "C" {

int gbq_init(void) {
    DevState *d = nullptr;
    return init_current(&d);
}

const char *gbq_device_name(void) {
    int dev = -1;
    g_name_out[0] = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices &&
        g_dev[dev].ready.load(std::memory_order_acquire))
        snprintf(g_name_out, sizeof(g_name_out), "%s", g_dev[dev].name);
    return g_name_out;
}

const char *gbq_last_error(void) { return g_err; }

int gbq_sync(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return GBQ_OK;
}

int gbq_device_status(void *stream, uint32_t *status) {
    REQUIRE(status != nullptr, "gbq_device_status: status is NULL");
    INIT(d);
    cudaStream_t st = (cudaStream_t)stream;
    unsigned int host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, d->status, sizeof(host), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(d->status, 0, sizeof(unsigned int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "gbq_device_status");
    *status = host;
    return GBQ_OK;
}

int gbq_prof_enable(int on) {
    INIT(d);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (on && !g_prof_created) {
        for (int i = 0; i < 2; ++i)
            for (int j = 0; j < kProfMax; ++j) {
                cudaError_t e = cudaEventCreate(&g_prof_ev[i][j]);
                if (e != cudaSuccess) return cuda_fail(e, "gbq_prof_enable");
            }
        g_prof_created = true;
    }
    g_prof_n = 0;
    g_prof_on = on != 0;
    return GBQ_OK;
}

int gbq_prof_read(int kind, int *launches, double *total_ms) {
    REQUIRE(launches && total_ms, "gbq_prof_read: NULL output");
    std::lock_guard<std::mutex> lock(g_prof_mu);
    int n = 0;
    double ms = 0.0;
    for (int i = 0; i < g_prof_n; ++i) {
        if (g_prof_kind[i] != kind) continue;
        cudaError_t e = cudaEventSynchronize(g_prof_ev[1][i]);
        float t = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, g_prof_ev[0][i], g_prof_ev[1][i]);
        if (e != cudaSuccess) return cuda_fail(e, "gbq_prof_read");
        ms += t;
        ++n;
    }
    *launches = n;
    *total_ms = ms;
    return GBQ_OK;
}

size_t gbq_workspace_size(int op, int64_t M, int64_t N, int64_t K, int64_t H) {
    return gemm_workspace_size_pref(op, M, N, K, H);
}

int gbq_quantize_act(const void *x, int8_t *q, float *x_scale, int64_t M, int64_t K, gbq_rot rot, void *stream) {
    REQUIRE(M >= 0 && K >= 1, "gbq_quantize_act: bad sizes M=%lld K=%lld", (long long)M, (long long)K);
    RotSel rs{};
    int rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(x) && a16(q) && a16(x_scale), "gbq_quantize_act: pointers must be non-NULL and 16-byte aligned");
    INIT(d);
    RotArgs a{};
    a.in0 = x;
    a.ld_in = K;
    a.out = q;
    a.out_scale = x_scale;
    a.M = M;
    a.K = K;
    return run_rotq("gbq_quantize_act", rs, IN_BF16, OUT_S8, a, (cudaStream_t)stream);
}

int gbq_prepare_weight(const void *w, int8_t *w8, float *w_scale, int64_t N, int64_t K, gbq_rot rot,
                       void *stream) {
    REQUIRE(N >= 0 && K >= 1, "gbq_prepare_weight: bad sizes N=%lld K=%lld", (long long)N, (long long)K);
    RotSel rs{};
    int rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (N == 0) return GBQ_OK;
    REQUIRE(a16(w) && a16(w8) && a16(w_scale), "gbq_prepare_weight: pointers must be non-NULL and 16-byte aligned");
    INIT(d);
    RotArgs a{};
    a.in0 = w;
    a.ld_in = K;
    a.out = w8;
    a.out_scale = w_scale;
    a.M = N;
    a.K = K;
    return run_rotq("gbq_prepare_weight", rs, IN_BF16, OUT_S8, a, (cudaStream_t)stream);
}

int gbq_quantize_act_glu(const void *g, const void *u, int8_t *q, float *h_scale, int64_t M, int64_t H,
                         gbq_rot rot, void *stream) {
    REQUIRE(M >= 0 && H >= 1, "gbq_quantize_act_glu: bad sizes M=%lld H=%lld", (long long)M, (long long)H);
    RotSel rs{};
    int rc = check_rot(rot, H, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(g) && a16(u) && a16(q) && a16(h_scale),
            "gbq_quantize_act_glu: pointers must be non-NULL and 16-byte aligned");
    INIT(d);
    RotArgs a{};
    a.in0 = g;
    a.in1 = u;
    a.ld_in = H;
    a.out = q;
    a.out_scale = h_scale;
    a.M = M;
    a.K = H;
    return run_rotq("gbq_quantize_act_glu", rs, IN_GLU_BF16, OUT_S8, a, (cudaStream_t)stream);
}

int gbq_dequant_act_quantize(const int32_t *acc_g, const int32_t *acc_u, int64_t ld_acc, const float *x_scale,
                             const float *s_gate, const float *s_up, int8_t *q, float *h_scale, int64_t M, int64_t H,
                             gbq_rot rot, void *stream) {
    REQUIRE(M >= 0 && H >= 1 && ld_acc >= H, "gbq_dequant_act_quantize: bad sizes M=%lld H=%lld ld_acc=%lld",
            (long long)M, (long long)H, (long long)ld_acc);
    RotSel rs{};
    int rc = check_rot(rot, H, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(acc_g) && a16(acc_u) && a16(x_scale) && a16(s_gate) && a16(s_up) && a16(q) && a16(h_scale),
            "gbq_dequant_act_quantize: pointers must be non-NULL and 16-byte aligned");
    REQUIRE(ld_acc % 4 == 0, "gbq_dequant_act_quantize: ld_acc must be a multiple of 4");
    INIT(d);
    RotArgs a{};
    a.in0 = acc_g;
    a.in1 = acc_u;
    a.in_scale = x_scale;
    a.col_scale0 = s_gate;
    a.col_scale1 = s_up;
    a.ld_in = ld_acc;
    a.out = q;
    a.out_scale = h_scale;
    a.M = M;
    a.K = H;
    return run_rotq("gbq_dequant_act_quantize", rs, IN_ACC_GLU, OUT_S8, a, (cudaStream_t)stream);
}

int gbq_rotate_bf16(const void *x, void *xr, int64_t M, int64_t K, gbq_rot rot, void *stream) {
    REQUIRE(M >= 0 && K >= 1, "gbq_rotate_bf16: bad sizes M=%lld K=%lld", (long long)M, (long long)K);
    RotSel rs{};
    int rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(x) && a16(xr), "gbq_rotate_bf16: pointers must be non-NULL and 16-byte aligned");
    INIT(d);
    if (rs.logn == 0) {
        cudaError_t e = cudaMemcpyAsync(xr, x, (size_t)(M * K * 2), cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
        return e == cudaSuccess ? GBQ_OK : cuda_fail(e, "gbq_rotate_bf16");
    }
    RotArgs a{};
    a.in0 = x;
    a.ld_in = K;
    a.out = xr;
    a.M = M;
    a.K = K;
    return run_rotq("gbq_rotate_bf16", rs, IN_BF16, OUT_BF16, a, (cudaStream_t)stream);
}

int gbq_dequant_weight(const int8_t *w8, const float *w_scale, void *w, int64_t N, int64_t K, gbq_rot rot,
                       void *stream) {
    REQUIRE(N >= 0 && K >= 1, "gbq_dequant_weight: bad sizes N=%lld K=%lld", (long long)N, (long long)K);
    RotSel rs{};
    int rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (N == 0) return GBQ_OK;
    REQUIRE(a16(w8) && a16(w_scale) && a16(w), "gbq_dequant_weight: pointers must be non-NULL and 16-byte aligned");
    INIT(d);
    if (rs.logn == 0) {
        REQUIRE(K % 16 == 0, "gbq_dequant_weight: identity rotation needs K %% 16 == 0");
        cudaError_t e = launch_scale_rows_s8(w8, w_scale, w, N, K, (cudaStream_t)stream, d->status);
        return e == cudaSuccess ? GBQ_OK : cuda_fail(e, "gbq_dequant_weight");
    }
    if (rot.a == 64 && rot.b == 64) {  // integer-exact two-pass kernel
        cudaError_t e = launch_dequant_weight64(w8, w_scale, w, N, rot.groups, d->sms, (cudaStream_t)stream, d->status);
        return e == cudaSuccess ? GBQ_OK : cuda_fail(e, "gbq_dequant_weight");
    }
    RotArgs a{};
    a.in0 = w8;
    a.in_scale = w_scale;
    a.ld_in = K;
    a.out = w;
    a.M = N;
    a.K = K;
    return run_rotq("gbq_dequant_weight", rs, IN_S8_ROWSCALE, OUT_BF16, a, (cudaStream_t)stream);
}

}  // extern "C"

// ============================================================ GEMM-backed entry points
namespace {

struct Ws {
    uint8_t *p;
    size_t left;
    void *take(size_t bytes) {
        bytes = (bytes + 255) & ~(size_t)255;
        if (bytes > left) return nullptr;
        void *r = p;
        p += bytes;
        left -= bytes;
        return r;
    }
};

int check_gemm_sizes(const char *what, int64_t M, int64_t N, int64_t K) {
    REQUIRE(M >= 0 && N >= 1 && K >= 64, "%s: bad sizes M=%lld N=%lld K=%lld", what, (long long)M, (long long)N,
            (long long)K);
    REQUIRE(K % 64 == 0, "%s: K=%lld must be a multiple of 64", what, (long long)K);
    REQUIRE(K <= 131072, "%s: K=%lld exceeds 131072 (int32 accumulator bound)", what, (long long)K);
    REQUIRE(M < (1ll << 31) && N < (1ll << 31), "%s: sizes exceed 2^31", what);
    return GBQ_OK;
}

int check_ws(const char *what, int op, void *workspace, size_t ws_bytes, int64_t M, int64_t N, int64_t K, int64_t H) {
    const size_t need = gemm_workspace_size(op, M, N, K, H);
    if (ws_bytes < need)
        return fail(GBQ_ENOSPC, "%s: workspace %zu bytes < %zu needed", what, ws_bytes, need);
    REQUIRE(need == 0 || ((uintptr_t)workspace & 255u) == 0, "%s: workspace must be 256-byte aligned", what);
    return GBQ_OK;
}

// Quantize x into the f16-coded GEMM operand.
int quantize_f16q(const char *what, const void *x, int64_t ld, void *qf16, float *xs, int64_t M, int64_t K,
                  const RotSel &rot, cudaStream_t st, int32_t *l1 = nullptr) {
    RotArgs a{};
    a.in0 = x;
    a.ld_in = ld;
    a.out = qf16;
    a.out_scale = xs;
    a.out_l1 = l1;
    a.M = M;
    a.K = K;
    return run_rotq(what, rot, IN_BF16, OUT_F16Q, a, st);
}

I8GemmProblem gemm_problem(DevState *d, const void *b_f16, const int8_t *w8, int64_t M, int64_t N, int64_t K,
                           int epi, void *out, int64_t ld_out, const float *xs, const float *ws, const void *bias) {
    I8GemmProblem g{};
    g.b_f16 = b_f16;
    g.w0 = w8;
    g.w1 = w8;
    g.ld_w = K;
    g.w_rows_total0 = N;
    g.w_rows_total1 = N;
    g.M = M;
    g.N = N;
    g.K = K;
    g.n_split = N;
    g.w_layout = W_KMAJOR;
    g.epi = epi;
    g.out = out;
    g.ld_out = ld_out;
    g.x_scale = xs;
    g.w_scale0 = ws;
    g.w_scale1 = ws;
    g.bias = bias;
    g.status = d->status;
    g.num_sms = d->sms;
    return g;
}

}  // namespace

namespace gbq {
// The argument checks of gbq_linear that need no pointer, then the device set-up (gbq_linear_noalloc
// runs them before its own scratch checks, so a bad argument gets the same code as from gbq_linear).
int linear_args_check(const char *what, int64_t M, int64_t N, int64_t K, gbq_rot rot) {
    int rc = check_gemm_sizes(what, M, N, K);
    if (rc) return rc;
    RotSel rs{};
    rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    DevState *d = nullptr;
    return init_current(&d);
}
}  // namespace gbq

extern "C" {

int gbq_int8_gemm(const int8_t *q, const int8_t *w8, int32_t *acc, int64_t ld_acc, int64_t M, int64_t N, int64_t K,
                  void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_gemm_sizes("gbq_int8_gemm", M, N, K);
    if (rc) return rc;
    REQUIRE(ld_acc >= N, "gbq_int8_gemm: ld_acc=%lld < N=%lld", (long long)ld_acc, (long long)N);
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(q) && a16(w8) && a16(acc), "gbq_int8_gemm: pointers must be non-NULL and 16-byte aligned");
    rc = check_ws("gbq_int8_gemm", GBQ_OP_INT8_GEMM, workspace, ws_bytes, M, N, K, 0);
    if (rc) return rc;
    INIT(d);
    cudaStream_t st = (cudaStream_t)stream;
    Ws w{(uint8_t *)workspace, ws_bytes};
    void *qf = w.take((size_t)M * K * 2);
    cudaError_t e = launch_s8_to_f16(q, qf, M * K, st, d->status);
    if (e != cudaSuccess) return cuda_fail(e, "gbq_int8_gemm (operand coding)");
    I8GemmProblem g = gemm_problem(d, qf, w8, M, N, K, EPI_ACC_I32, acc, ld_acc, nullptr, nullptr, nullptr);
    return launch_i8gemm(g, st);
}

int gbq_linear_acc(const void *x, const int8_t *w8, int32_t *acc, int64_t ld_acc, float *x_scale, int64_t M,
                   int64_t N, int64_t K, gbq_rot rot, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_gemm_sizes("gbq_linear_acc", M, N, K);
    if (rc) return rc;
    RotSel rs{};
    rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    REQUIRE(ld_acc >= N, "gbq_linear_acc: ld_acc < N");
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(x) && a16(w8) && a16(acc) && a16(x_scale),
            "gbq_linear_acc: pointers must be non-NULL and 16-byte aligned");
    rc = check_ws("gbq_linear_acc", GBQ_OP_LINEAR, workspace, ws_bytes, M, N, K, 0);
    if (rc) return rc;
    INIT(d);
    cudaStream_t st = (cudaStream_t)stream;
    Ws w{(uint8_t *)workspace, ws_bytes};
    void *qf = w.take((size_t)M * K * 2);
    (void)w.take((size_t)M * 4);                      // (gbq_linear's x_scale slot)
    int32_t *l1 = (int32_t *)w.take((size_t)M * 4 * ((K + 1023) / 1024));  // block L1 norms: preferred size only
    if (!rotq_writes_l1(rs.logn, rs.groups)) l1 = nullptr;
    rc = quantize_f16q("gbq_linear_acc", x, K, qf, x_scale, M, K, rs, st, l1);
    if (rc) return rc;
    I8GemmProblem g = gemm_problem(d, qf, w8, M, N, K, EPI_ACC_I32, acc, ld_acc, nullptr, nullptr, nullptr);
    g.row_l1 = l1;
    g.pdl = 1;  // directly after the quantizer launch
    return launch_i8gemm(g, st);
}

int gbq_dequant(const int32_t *acc, int64_t ld_acc, const float *x_scale, const float *w_scale, const void *bias,
                void *y, int64_t ld_y, int64_t M, int64_t N, void *stream) {
    REQUIRE(M >= 0 && N >= 1 && ld_acc >= N && ld_y >= N, "gbq_dequant: bad sizes");
    if (M == 0) return GBQ_OK;
    REQUIRE(acc && x_scale && w_scale && y, "gbq_dequant: pointers must be non-NULL");
    REQUIRE(((uintptr_t)acc & 3) == 0 && ((uintptr_t)x_scale & 3) == 0 && ((uintptr_t)w_scale & 3) == 0 &&
                ((uintptr_t)y & 1) == 0 && ((uintptr_t)bias & 1) == 0,
            "gbq_dequant: pointers must be aligned to their element size");
    INIT(d);
    cudaError_t e = launch_dequant(acc, ld_acc, x_scale, w_scale, bias, y, ld_y, M, N, (cudaStream_t)stream, d->status);
    return e == cudaSuccess ? GBQ_OK : cuda_fail(e, "gbq_dequant");
}

int gbq_linear(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y, int64_t M, int64_t N,
               int64_t K, gbq_rot rot, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_gemm_sizes("gbq_linear", M, N, K);
    if (rc) return rc;
    RotSel rs{};
    rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(x) && a16(w8) && a16(w_scale) && a16(y) && (bias == nullptr || a16(bias)),
            "gbq_linear: pointers must be non-NULL (bias may be NULL) and 16-byte aligned");
    rc = check_ws("gbq_linear", GBQ_OP_LINEAR, workspace, ws_bytes, M, N, K, 0);
    if (rc) return rc;
    INIT(d);
    cudaStream_t st = (cudaStream_t)stream;
    // Decode and small batches: for one or two tokens a GEMV with the rotation inside (the square kernels'
    // for the shapes they cover, else the generic rotation's); otherwise, up to 16 tokens, the rotation
    // kernels quantize x into the workspace and a GEMV streams the weight over those codes.  Every route
    // has the same codes, scales and epilogue as the GEMM route below.
    if (M <= 4 && rs.logn > 0) {
        rc = launch_gemv(x, w8, w_scale, bias, y, M, N, K, rs.logn, rs.groups, d->sms, st, d->status);
        if (rc != GBQ_ENOTSUP) return rc;
    }
    // The generic rotation inside: faster than the rotation kernels + codes GEMV while a CTA rotates at
    // most 8192 values (measured: K = 2048 as 32x64, one token, 5.8 vs 6.9 us; K = 8192 as 64x128, 21.3 vs
    // 22.3 us, two tokens 27.9 vs 23.9 us; K = 16384 as 128x128, 48.9 vs 46.0 us).
    if (M * K <= 8192 && rs.logn != 0 && gemv_gen_fits(M, N, K, d->sms)) {
        rc = launch_gemv_gen(x, w8, w_scale, bias, y, M, N, K, rs.la, rs.lb, d->sms, st, d->status);
        if (rc != GBQ_ENOTSUP) return rc;
    }
    if (gemv_codes_fits(M, N, K, d->sms)) {
        Ws wc{(uint8_t *)workspace, ws_bytes};
        int8_t *codes = (int8_t *)wc.take((size_t)M * K);
        float *xs_c = (float *)wc.take((size_t)M * 4);
        RotArgs a{};
        a.in0 = x;
        a.ld_in = K;
        a.out = codes;
        a.out_scale = xs_c;
        a.M = M;
        a.K = K;
        rc = run_rotq("gbq_linear (GEMV codes)", rs, IN_BF16, OUT_S8, a, st);
        if (rc) return rc;
        return launch_gemv_codes(codes, xs_c, w8, w_scale, bias, y, N, M, N, K, d->sms, st, d->status);
    }
    Ws w{(uint8_t *)workspace, ws_bytes};
    void *qf = w.take((size_t)M * K * 2);
    float *xs = (float *)w.take((size_t)M * 4);
    int32_t *l1 = (int32_t *)w.take((size_t)M * 4 * ((K + 1023) / 1024));  // block L1 norms: preferred size only
    if (!rotq_writes_l1(rs.logn, rs.groups)) l1 = nullptr;
    rc = quantize_f16q("gbq_linear", x, K, qf, xs, M, K, rs, st, l1);
    if (rc) return rc;
    I8GemmProblem g = gemm_problem(d, qf, w8, M, N, K, EPI_DEQUANT_BF16, y, N, xs, w_scale, bias);
    g.row_l1 = l1;
    g.pdl = 1;  // directly after the quantizer launch
    return launch_i8gemm(g, st);
}

int gbq_ffn_fused(const void *x, const int8_t *wg8, const float *s_gate, const int8_t *wu8, const float *s_up,
                  const int8_t *wd8, const float *s_down, void *y, int64_t M, int64_t d, int64_t H, gbq_rot rot_d,
                  gbq_rot rot_h, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_gemm_sizes("gbq_ffn_fused (gate/up)", M, 2 * H, d);
    if (rc) return rc;
    rc = check_gemm_sizes("gbq_ffn_fused (down)", M, d, H);
    if (rc) return rc;
    REQUIRE(H % 128 == 0, "gbq_ffn_fused: H=%lld must be a multiple of 128", (long long)H);
    RotSel rsd{}, rsh{};
    rc = check_rot(rot_d, d, &rsd);
    if (rc) return rc;
    rc = check_rot(rot_h, H, &rsh);
    if (rc) return rc;
    if (rsh.logn == 0 && !rotg_fits(H))
        return fail(GBQ_ENOTSUP, "gbq_ffn_fused: identity hidden rotation needs H <= %lld", (long long)kGenMaxK);
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(x) && a16(wg8) && a16(s_gate) && a16(wu8) && a16(s_up) && a16(wd8) && a16(s_down) && a16(y),
            "gbq_ffn_fused: pointers must be non-NULL and 16-byte aligned");
    rc = check_ws("gbq_ffn_fused", GBQ_OP_FFN, workspace, ws_bytes, M, 0, d, H);
    if (rc) return rc;
    INIT(dv);
    cudaStream_t st = (cudaStream_t)stream;
    if (gemv_codes_fits(M, 2 * H, d, dv->sms) && gemv_codes_fits(M, d, H, dv->sms)) {
        // Decode and small batches: the same four steps with int8 codes and weight-streaming GEMVs in
        // place of the GEMMs (the same codes, scales and epilogues, so the same bits).
        Ws wc{(uint8_t *)workspace, ws_bytes};
        int8_t *cx = (int8_t *)wc.take((size_t)M * d * 2);  // the slots of the GEMM route below
        float *cxs = (float *)wc.take((size_t)M * 4);
        uint8_t *cgu = (uint8_t *)wc.take((size_t)M * 2 * H * 2);
        int8_t *ch = (int8_t *)wc.take((size_t)M * H * 2);
        float *chs = (float *)wc.take((size_t)M * 4);
        RotArgs a{};
        a.in0 = x;
        a.ld_in = d;
        a.out = cx;
        a.out_scale = cxs;
        a.M = M;
        a.K = d;
        rc = run_rotq("gbq_ffn_fused (x codes)", rsd, IN_BF16, OUT_S8, a, st);
        if (rc) return rc;
        // g | u in bf16, row stride 2H (no bias): one GEMV over the virtual weight [W_gate; W_up]
        rc = launch_gemv_codes2(cx, cxs, wg8, s_gate, wu8, s_up, H, nullptr, cgu, 2 * H, M, 2 * H, d, dv->sms, st,
                                dv->status);
        if (rc) return rc;
        RotArgs ah{};
        ah.in0 = cgu;
        ah.in1 = cgu + H * 2;
        ah.ld_in = 2 * H;
        ah.out = ch;
        ah.out_scale = chs;
        ah.M = M;
        ah.K = H;
        rc = run_rotq("gbq_ffn_fused (h codes)", rsh, IN_GLU_BF16, OUT_S8, ah, st);
        if (rc) return rc;
        return launch_gemv_codes(ch, chs, wd8, s_down, nullptr, y, d, M, d, H, dv->sms, st, dv->status);
    }
    Ws w{(uint8_t *)workspace, ws_bytes};
    void *qx = w.take((size_t)M * d * 2);
    float *xs = (float *)w.take((size_t)M * 4);
    void *gu = w.take((size_t)M * 2 * H * 2);
    void *qh = w.take((size_t)M * H * 2);
    float *hs = (float *)w.take((size_t)M * 4);
    int32_t *l1x = (int32_t *)w.take((size_t)M * 4 * ((d + 1023) / 1024));  // block L1 norms: preferred size only
    int32_t *l1h = (int32_t *)w.take((size_t)M * 4 * ((H + 1023) / 1024));
    if (!rotq_writes_l1(rsd.logn, rsd.groups)) l1x = nullptr;
    if (!rotq_writes_l1(rsh.logn, rsh.groups)) l1h = nullptr;
    // 1) rotate + quantize x over d
    rc = quantize_f16q("gbq_ffn_fused (x)", x, d, qx, xs, M, d, rsd, st, l1x);
    if (rc) return rc;
    // 2) gate and up GEMMs in one launch over the virtual weight [W_gate; W_up],
    //    dequantized to bf16 g | u (row stride 2H)
    I8GemmProblem g = gemm_problem(dv, qx, wg8, M, 2 * H, d, EPI_DEQUANT_BF16, gu, 2 * H, xs, s_gate, nullptr);
    g.w1 = wu8;
    g.w_rows_total0 = H;
    g.w_rows_total1 = H;
    g.n_split = H;
    g.w_scale1 = s_up;
    g.row_l1 = l1x;
    g.pdl = 1;
    rc = launch_i8gemm(g, st);
    if (rc) return rc;
    // 3) h = silu(g) * u, rotate over H, quantize
    RotArgs a{};
    a.in0 = gu;
    a.in1 = (const uint8_t *)gu + H * 2;
    a.ld_in = 2 * H;
    a.out = qh;
    a.out_scale = hs;
    a.out_l1 = l1h;
    a.M = M;
    a.K = H;
    rc = run_rotq("gbq_ffn_fused (h)", rsh, IN_GLU_BF16, OUT_F16Q, a, st);
    if (rc) return rc;
    // 4) down GEMM + dequant
    I8GemmProblem gd = gemm_problem(dv, qh, wd8, M, d, H, EPI_DEQUANT_BF16, y, d, hs, s_down, nullptr);
    gd.row_l1 = l1h;
    gd.pdl = 1;
    return launch_i8gemm(gd, st);
}

int gbq_linear_dx(const void *dy, const void *w, void *dx, int64_t M, int64_t N, int64_t K, void *stream) {
    REQUIRE(M >= 0 && N >= 64 && K >= 16, "gbq_linear_dx: bad sizes M=%lld N=%lld K=%lld", (long long)M,
            (long long)N, (long long)K);
    REQUIRE(N % 64 == 0 && K % 16 == 0, "gbq_linear_dx: N must be a multiple of 64 and K of 16");
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(dy) && a16(w) && a16(dx), "gbq_linear_dx: pointers must be non-NULL and 16-byte aligned");
    INIT(d);
    return launch_bf16_gemm_nn(dy, w, dx, M, N, K, d->status, d->sms, (cudaStream_t)stream);
}

int gbq_linear_bf16(const void *x, const void *w, const void *bias, void *y, int64_t M, int64_t N, int64_t K,
                    void *stream) {
    REQUIRE(M >= 0 && N >= 1 && K >= 64, "gbq_linear_bf16: bad sizes M=%lld N=%lld K=%lld", (long long)M,
            (long long)N, (long long)K);
    REQUIRE(K % 64 == 0, "gbq_linear_bf16: K must be a multiple of 64");
    REQUIRE(N <= ((int64_t)1 << 31) && K <= ((int64_t)1 << 31) && M <= ((int64_t)1 << 31),
            "gbq_linear_bf16: sizes beyond 2^31");
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(x) && a16(w) && a16(y), "gbq_linear_bf16: x, w, y must be non-NULL and 16-byte aligned");
    REQUIRE(((uintptr_t)bias & 1) == 0, "gbq_linear_bf16: bias must be 2-byte aligned");
    INIT(d);
    return launch_bf16_gemm_tn(x, w, bias, y, M, N, K, d->status, d->sms, (cudaStream_t)stream);
}

int gbq_linear_dx_int8(const void *dy, const int8_t *w8, const float *w_scale, void *dx, int64_t M, int64_t N,
                       int64_t K, gbq_rot rot, void *workspace, size_t ws_bytes, void *stream) {
    // The GEMM contracts over N (W8's rows) and produces K output columns.
    int rc = check_gemm_sizes("gbq_linear_dx_int8", M, K, N);
    if (rc) return rc;
    REQUIRE(K % 16 == 0, "gbq_linear_dx_int8: K must be a multiple of 16");
    RotSel rs{};
    rc = check_rot(rot, K, &rs);
    if (rc) return rc;
    if (M == 0) return GBQ_OK;
    REQUIRE(a16(dy) && a16(w8) && a16(w_scale) && a16(dx),
            "gbq_linear_dx_int8: pointers must be non-NULL and 16-byte aligned");
    rc = check_ws("gbq_linear_dx_int8", GBQ_OP_LINEAR_DX_INT8, workspace, ws_bytes, M, N, K, 0);
    if (rc) return rc;
    INIT(d);
    cudaStream_t st = (cudaStream_t)stream;
    Ws w{(uint8_t *)workspace, ws_bytes};
    void *qd = w.take((size_t)M * N * 2);
    float *t = (float *)w.take((size_t)M * 4);
    float *dxr = (float *)w.take((size_t)M * K * 4);
    int32_t *l1 = (int32_t *)w.take((size_t)M * 4 * ((N + 1023) / 1024));  // block L1 norms: preferred size only
    if (rs.logn == 0 && !rotg_fits(K))
        return fail(GBQ_ENOTSUP, "gbq_linear_dx_int8: identity rotation needs K <= %lld", (long long)kGenMaxK);
    // A long contraction splits in two halves run side by side on two streams, each GEMM on half the CTA
    // pairs: the 256 x 256 tiles then fill the SMs in about twice as many waves of half-length tiles
    // (M = K = 4096: 6.7 waves of halves against 3.4 of whole tiles, whose last wave leaves most SMs idle).
    // Each half adds its exact int32 sums into the (zeroed) accumulator; the rotation applies t[m].
    const bool split = N >= 8192 && N % 2048 == 0;
    int32_t *acc = reinterpret_cast<int32_t *>(dxr);  // the same workspace bytes, read as int32 when split
    cudaError_t e;
    std::unique_lock<std::mutex> fork_lock(d->fork_mu, std::defer_lock);
    if (split) {
        // The accumulator is cleared on the second stream while the quantizer runs on this one (after
        // everything enqueued on this stream before the call, which may still use the workspace).
        fork_lock.lock();
        e = cudaEventRecord(d->ev_entry, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(d->aux, d->ev_entry, 0);
        if (e == cudaSuccess) e = cudaMemsetAsync(acc, 0, (size_t)M * K * 4, d->aux);
        if (e == cudaSuccess) e = cudaEventRecord(d->ev_zero, d->aux);
        if (e != cudaSuccess) return cuda_fail(e, "gbq_linear_dx_int8 (clear the accumulator)");
    }
    // 1) dy' = dy * s[n] (column scale), per-row quantize, no rotation
    IdArgs ia{dy, w_scale, N, qd, t, M, N, l1, d->status, d->sms};
    e = launch_quant_identity(OUT_F16Q, ia, st);
    if (e != cudaSuccess) {
        if (split) (void)cudaStreamWaitEvent(st, d->ev_zero, 0);  // the caller's stream stays after the clear
        return cuda_fail(e, "gbq_linear_dx_int8 (quantize dy)");
    }
    RotArgs a{};
    a.ld_in = K;
    a.out = dx;
    a.M = M;
    a.K = K;
    if (!split) {
        // 2) acc[m, k] = sum_n qd[m, n] w8[n, k]; dx_rot = fp32(acc) * t[m]
        I8GemmProblem g = gemm_problem(d, qd, w8, M, K, N, EPI_ROWSCALE_F32, dxr, K, t, nullptr, nullptr);
        g.w_layout = W_NMAJOR;
        g.ld_w = K;
        g.w_rows_total0 = N;
        g.w_rows_total1 = N;
        g.row_l1 = l1;
        g.pdl = 1;  // directly after the quantizer launch
        rc = launch_i8gemm(g, st);
        if (rc) return rc;
        // 3) dx = bf16(dx_rot R)
        a.in0 = dxr;
        return run_rotq("gbq_linear_dx_int8 (rotate dx)", rs, IN_F32, OUT_BF16, a, st);
    }
    // 2) acc[m, k] += sum over each half of n of qd[m, n] w8[n, k], the halves on two streams
    const int64_t nh = N / 2;
    const int nb = (int)((N + 1023) / 1024);
    int half_pairs = i8gemm_max_pairs(d->sms) / 2;
    if (half_pairs < 1) half_pairs = 1;
    I8GemmProblem g0 = gemm_problem(d, qd, w8, M, K, nh, EPI_ACC_I32, acc, K, nullptr, nullptr, nullptr);
    g0.w_layout = W_NMAJOR;
    g0.ld_w = K;
    g0.w_rows_total0 = nh;
    g0.w_rows_total1 = nh;
    g0.ld_b = N;
    g0.row_l1 = l1;
    g0.l1_ld = nb;
    g0.reduce_out = 1;
    g0.max_pairs = half_pairs;
    g0.pdl = 0;  // the fork's event record sits between the quantizer and this launch
    I8GemmProblem g1 = g0;
    g1.b_f16 = reinterpret_cast<const uint16_t *>(qd) + nh;
    g1.w0 = w8 + nh * K;
    g1.w1 = g1.w0;
    g1.row_l1 = l1 ? l1 + nh / 1024 : nullptr;
    {
        e = cudaEventRecord(d->ev_fork, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(d->aux, d->ev_fork, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, d->ev_zero, 0);
        if (e != cudaSuccess) return cuda_fail(e, "gbq_linear_dx_int8 (fork)");
        rc = launch_i8gemm(g0, st);
        if (rc == GBQ_OK) rc = launch_i8gemm(g1, d->aux);
        // the join is recorded even after a failed launch, so that the auxiliary stream never runs ahead
        e = cudaEventRecord(d->ev_join, d->aux);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, d->ev_join, 0);
        fork_lock.unlock();
        if (rc) return rc;
        if (e != cudaSuccess) return cuda_fail(e, "gbq_linear_dx_int8 (join)");
    }
    // 3) dx = bf16((fp32(acc) * t[m]) R)
    a.in0 = acc;
    a.in_scale = t;
    return run_rotq("gbq_linear_dx_int8 (rotate dx)", rs, IN_ACC_ROWSCALE, OUT_BF16, a, st);
}

}  // extern "C"
