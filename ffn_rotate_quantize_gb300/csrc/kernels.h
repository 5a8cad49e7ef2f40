// kernels.h -- host-side launchers of the libgbq kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rotate_impl.cuh"

namespace gbq {

void prof_begin(int kind, cudaStream_t st);
void prof_end(cudaStream_t st);

// Per-row identity "rotation" quantizer (R = I), optional per-column scale on the input.
struct IdArgs {
    const void *in;           // bf16 [M, ld_in]
    const float *col_scale;   // fp32 [K] or nullptr
    int64_t ld_in;
    void *out;                // int8 or f16-coded int [M, K]
    float *out_scale;         // fp32 [M]
    int64_t M, K;
    int32_t *out_l1;          // [M][ceil(K/1024)] sums of |code| over 1024-long blocks, or nullptr
    unsigned int *status = nullptr;  // device status word; with num_sms > 0 it enables the streaming
    int num_sms = 0;                 // kernel for long rows (8192 <= K <= 16384)
};

// Launch a rotate(+quantize) kernel.  Returns cudaErrorNotSupported for a
// combination that has no instantiation or does not fit one CTA.
cudaError_t launch_rotq(int logn, int in_kind, int out_kind, RotArgs a, cudaStream_t st);   // OUT_S8 / OUT_F16Q
cudaError_t launch_rotb(int logn, int in_kind, RotArgs a, cudaStream_t st);                 // OUT_BF16
cudaError_t launch_quant_identity(int out_kind, IdArgs a, cudaStream_t st);
// W_hat = bf16((W8 * s) R) for n = 64 (N rows of `groups` 4096-long groups), integer-exact transform.
cudaError_t launch_dequant_weight64(const int8_t *w8, const float *w_scale, void *out, int64_t N, int groups,
                                    int num_sms, cudaStream_t st, unsigned int *status = nullptr);

// The rotation for every descriptor (rotate_g.cu): any powers of two a = 2^la, b = 2^lb
// (la = lb = 0: the identity, quantization or conversion only), rows of K values with
// K % 16 == 0 and K <= kGenMaxK.  Bit-identical to the square kernels where both apply.
constexpr int64_t kGenMaxK = 49152;
bool rotg_fits(int64_t K);
cudaError_t launch_rotg(int in_kind, int out_kind, const RotArgs &a, int la, int lb, cudaStream_t st);

// Whether the rotate+quantize launch for this rotation fills RotArgs::out_l1 (the three-pass
// kernels: a = b = 64 or 128, one group per row); elsewhere out_l1 is left untouched.
inline bool rotq_writes_l1(int logn, int groups) { return (logn == 6 || logn == 7) && groups == 1; }

// Threads of one rotq launch row (G groups of n/CPT threads).
inline int rotq_row_threads(int logn, int G) {
    const int n = 1 << logn;
    const int cpt = logn >= 7 ? 1 : 2;
    return G * (n / cpt);
}

}  // namespace gbq
