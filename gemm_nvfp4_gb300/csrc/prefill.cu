// prefill.cu -- products for N > 16 tokens (prefill).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

size_t prefill_workspace_bytes(int64_t N, int64_t M, int64_t K, int n_weights)
{
    (void)N; (void)M; (void)K;
    return (size_t)kGemvMaxCtas * kGemvPartialFloatsPerCta * n_weights * 4;
}

// Interim: 16-token slices through the skinny kernel.
cudaError_t launch_prefill(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                           const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                           int out_bf16, void *workspace, int num_sms, cudaStream_t stream)
{
    const size_t esize = out_bf16 ? 2 : 4;
    for (int64_t n0 = 0; n0 < N; n0 += 16) {
        const int n = (int)std::min<int64_t>(16, N - n0);
        cudaError_t e = launch_gemv(x + n0 * K, n, M, K, codes, scales, ts, n_weights,
                                    static_cast<char *>(y) + n0 * M * esize, out_bf16, workspace, num_sms, stream);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace nvfp4
