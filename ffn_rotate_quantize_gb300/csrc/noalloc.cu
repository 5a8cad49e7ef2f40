// noalloc.cu -- gbq_linear_noalloc: the rotated-INT8 linear layer with its
// scratch in a static device array instead of a caller workspace.
//
// gbq_linear needs scratch for the quantized activations (fp16-coded int8
// codes, M*K*2 bytes) and their per-row scales (M*4 bytes).  Normally the
// caller passes that scratch as `workspace`.  Some callers cannot allocate
// device memory at the point of the call: a plugin running inside a host
// framework that owns all device memory through its own pool and forbids
// direct cudaMalloc, or a latency-critical loop where cudaMalloc's implicit
// device-wide synchronisation is not acceptable.  This entry point serves
// them: the scratch is a file-scope static __device__ array.
//
// The library's kernels live in separately compiled modules, which CUDA loads
// lazily: this array's module (and its 16 MiB) is loaded by the first lookup of
// the array's address.  That lookup is part of the library's per-device set-up
// (gbq_init, or the first call of any entry point on the device), so no call of
// gbq_linear_noalloc after the set-up reserves device memory.
#include <stdio.h>

#include <atomic>

#include "../../include/gbq.h"
#include "gemm.h"

namespace {

// Every device that sets the library up holds this array until exit.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::atomic<void *> g_scratch_addr[kMaxDev];

}  // namespace

namespace gbq {

// The host-side symbol g_noalloc_scratch is only a stand-in for the device array; its device
// address comes from cudaGetSymbolAddress with the device current.  Called once per device by the
// library's device set-up (under its lock).
int noalloc_setup_current(int dev) {
    if (dev < 0 || dev >= kMaxDev) return gbq_fail(GBQ_ENODEV, "gbq_linear_noalloc: device index out of range");
    if (g_scratch_addr[dev].load(std::memory_order_acquire)) return GBQ_OK;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "device set-up: reserving gbq_linear_noalloc's 16 MiB static scratch (cudaGetSymbolAddress) "
                 "failed: %s",
                 cudaGetErrorString(e));
        return gbq_fail(GBQ_ECUDA, msg);
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
    return GBQ_OK;
}

}  // namespace gbq

extern "C" int gbq_linear_noalloc(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y,
                                  int64_t M, int64_t N, int64_t K, gbq_rot rot, void *stream) {
    // gbq_linear's own size and rotation checks and the device set-up come first, so a bad argument
    // returns the same code as from gbq_linear.
    int rc = gbq::linear_args_check("gbq_linear_noalloc", M, N, K, rot);
    if (rc != GBQ_OK) return rc;
    // An empty batch needs no scratch: gbq_linear launches nothing, as for every other entry point.
    if (M == 0) return gbq_linear(x, w8, w_scale, bias, y, M, N, K, rot, nullptr, 0, stream);
    const size_t need = gbq::gemm_workspace_size(GBQ_OP_LINEAR, M, N, K, 0);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gbq_linear_noalloc: M=%lld, K=%lld needs %zu bytes of scratch; the static scratch holds %zu "
                 "bytes (M*K*2 + M*4, each rounded up to 256, must fit); use gbq_linear with a workspace",
                 (long long)M, (long long)K, need, kNoAllocScratchBytes);
        return gbq::gbq_fail(GBQ_ENOSPC, msg);
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return gbq::gbq_fail(GBQ_ENODEV, "gbq_linear_noalloc: no current CUDA device");
    void *scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!scratch) return gbq::gbq_fail(GBQ_ECUDA, "gbq_linear_noalloc: the device's static scratch is not set up");
    // The scratch needs no clearing: the quantizer writes every code and scale that the GEMM (or the
    // GEMV) reads afterwards, and the per-block sums that do not fit are simply not used.
    return gbq_linear(x, w8, w_scale, bias, y, M, N, K, rot, scratch, kNoAllocScratchBytes, stream);
}
