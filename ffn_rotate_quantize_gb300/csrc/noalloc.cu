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
// them: the scratch is a file-scope static __device__ array, reserved when the
// library is loaded on a device and kept until the process exits.
#include <stdio.h>

#include <mutex>

#include "../../include/gbq.h"
#include "gemm.h"

namespace {

// Every device that loads the library holds this array until exit.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void *g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of the static scratch for the current device.  The host-side
// symbol is only a stand-in; the real address comes from cudaGetSymbolAddress,
// called once per device with that device current.
int scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return gbq::gbq_fail(GBQ_ENODEV, "gbq_linear_noalloc: no current CUDA device");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof(msg), "gbq_linear_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return gbq::gbq_fail(GBQ_ECUDA, msg);
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GBQ_OK;
}

}  // namespace

extern "C" int gbq_linear_noalloc(const void *x, const int8_t *w8, const float *w_scale, const void *bias, void *y,
                                  int64_t M, int64_t N, int64_t K, gbq_rot rot, void *stream) {
    if (M < 0 || N < 0 || K < 0) return gbq::gbq_fail(GBQ_EINVAL, "gbq_linear_noalloc: negative size");
    const size_t need = gbq::gemm_workspace_size(GBQ_OP_LINEAR, M, N, K, 0);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gbq_linear_noalloc: M=%lld, K=%lld needs %zu bytes of scratch; the static scratch holds %zu "
                 "bytes (M*K*2 + M*4, each rounded up to 256, must fit); use gbq_linear with a workspace",
                 (long long)M, (long long)K, need, kNoAllocScratchBytes);
        return gbq::gbq_fail(GBQ_ENOSPC, msg);
    }
    // An empty batch needs no scratch: gbq_linear checks the arguments and launches nothing, as for
    // every other entry point (no device work at all, so it also holds where no device is present).
    if (M == 0) return gbq_linear(x, w8, w_scale, bias, y, M, N, K, rot, nullptr, 0, stream);
    void *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != GBQ_OK) return rc;
    // The scratch needs no clearing: the quantizer writes every code and scale
    // that the GEMM (or the GEMV) reads afterwards.
    return gbq_linear(x, w8, w_scale, bias, y, M, N, K, rot, scratch, kNoAllocScratchBytes, stream);
}
