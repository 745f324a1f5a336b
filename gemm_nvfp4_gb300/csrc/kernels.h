// kernels.h -- launch interface between the C ABI (nvfp4_abi.cu) and the
// kernel translation units.  Internal to libnvfp4.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace nvfp4 {

// Runs `set` once for each device it is called on (the current device) and
// returns that device's result.  Function attributes such as the dynamic
// shared-memory limit belong to each device's context, so a process that
// drives several GPUs must set them on every one.
constexpr int kMaxDevices = 64;
template <class F>
cudaError_t once_per_device(std::once_flag (&flags)[kMaxDevices], cudaError_t (&results)[kMaxDevices], F &&set)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::call_once(flags[dev], [&] { results[dev] = set(); });
    return results[dev];
}

// Byte offset of the device status word inside the workspace of every product
// call (skinny, gate/up, prefill; NVFP4 and FP6).  A tensor-core kernel whose
// bounded pipeline wait runs out stores a nonzero code there (atomicExch) and
// returns; no kernel ever clears it, so it stays set until the caller clears
// it (nvfp4_device_status).  Codes: 1..7 prefill, 11..25 skinny, and
// kStatusSelftest for the wait-timeout self-test.
constexpr size_t kStatusWordOffset = 128;
constexpr uint32_t kStatusSelftest = 127;

// One thread waits on a shared-memory barrier that nothing completes; after
// the bounded wait gives up it records kStatusSelftest in the status word.
cudaError_t launch_wait_timeout_selftest(void *workspace, cudaStream_t stream);

// Partial maxima written by the amax kernel of the quantiser.
constexpr int kQuantPartials = 1024;
// Largest grid of the skinny kernel (sizes its split-K workspace).
constexpr int kGemvMaxCtas = 1024;
// Split-K partials of one CTA: 2 slots x 16 rows x 16 tokens fp32.
constexpr int64_t kGemvPartialFloatsPerCta = 2 * 16 * 16;

cudaError_t launch_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, void *workspace, int num_sms, cudaStream_t stream);
cudaError_t launch_quantize_bf16(const uint16_t *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                 float *tensor_scale, void *workspace, int num_sms, cudaStream_t stream);
cudaError_t launch_fp6_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                int num_sms, cudaStream_t stream);
cudaError_t launch_fp6_quantize_bf16(const uint16_t *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                     int num_sms, cudaStream_t stream);
cudaError_t launch_import_blocked_scales(const uint8_t *blocked, int64_t M, int64_t K, uint8_t *scales,
                                         cudaStream_t stream);

// n_weights = 1: y = x . W^T; n_weights = 2: h = silu(x . Wg^T) * (x . Wu^T)
// with codes/scales/ts[0] = gate, [1] = up.
cudaError_t launch_gemv(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                        const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                        int out_bf16, void *workspace, int num_sms, cudaStream_t stream);

int64_t gemv_grid(int64_t M, int64_t K, int num_sms);

// FP6 E2M3 weights (codes [M][3K/4], UE8M0 scales [M][K/128], K % 128 == 0):
// the skinny product for N = 1..16 on the warp-level MMA kernel of gemv.cu
// (split-K partials in the workspace, gemv_mma_workspace_bytes), and the
// tensor-core prefill for larger N.
size_t gemv_mma_workspace_bytes(int n_weights);
cudaError_t launch_gemv_fp6(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                            const uint8_t *const *scales, int n_weights, void *y, int out_bf16, void *workspace,
                            int num_sms, cudaStream_t stream);
cudaError_t launch_skinny_tc_fp6(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                                 const uint8_t *const *scales, int n_weights, void *y, int out_bf16,
                                 void *workspace, int num_sms, cudaStream_t stream);
cudaError_t launch_prefill_fp6(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                               const uint8_t *const *scales, int n_weights, void *y, int out_bf16,
                               void *workspace, int num_sms, cudaStream_t stream);

}  // namespace nvfp4

namespace nvfp4 {

size_t prefill_workspace_bytes(int64_t N, int64_t M, int64_t K, int n_weights, int fmt);

cudaError_t launch_prefill(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                           const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                           int out_bf16, void *workspace, int num_sms, cudaStream_t stream);

}  // namespace nvfp4

namespace nvfp4 {

// Skinny tcgen05 path (gemv_tc.cu), used when skinny_tc_supported(M, K).
constexpr int kSkinnyTcMaxCtas = 256;
bool skinny_tc_supported(int64_t M, int64_t K);
size_t skinny_tc_workspace_bytes(int64_t M, int64_t K, int n_weights);
cudaError_t launch_skinny_tc(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                             const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                             int out_bf16, void *workspace, int num_sms, cudaStream_t stream);

// Workspace of the skinny product for any K (tcgen05 path or the mma.sync path).
size_t skinny_workspace_bytes(int64_t M, int64_t K, int n_weights);

}  // namespace nvfp4

namespace nvfp4 {

// Host-side argument checks of nvfp4_gemv_skinny (everything but the
// workspace): returns an nvfp4_status; *nothing_to_do is set when the call is
// valid but enqueues nothing (N == 0 or M == 0).
int check_skinny_call(const uint16_t *x, int64_t N, const uint8_t *codes, const uint8_t *scales,
                      const float *tensor_scale, int64_t M, int64_t K, const void *y, int out_dtype,
                      bool *nothing_to_do);

}  // namespace nvfp4
