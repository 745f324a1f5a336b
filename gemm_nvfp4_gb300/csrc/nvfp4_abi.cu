// nvfp4_abi.cu -- the C ABI of libnvfp4.so (declared in include/nvfp4.h):
// argument checks on the host, workspace sizes, and dispatch by N to the
// skinny kernel (N <= 16) or the tensor-core prefill kernel (N > 16), the
// per-shape dispatch of bw24 README, NVFP4 decode path (one entry point per
// operation, the library picks the kernel from the shape).
#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/nvfp4.h"
#include "kernels.h"

namespace {

using namespace nvfp4;

constexpr int kMaxSkinnyN = 16;
static_assert(kStatusWordOffset == NVFP4_STATUS_WORD_OFFSET, "status word offset differs from the header");

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Streaming multiprocessors of the current device (cached per device id).
int current_num_sms(int *out)
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) {
            *out = v;
            return NVFP4_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return NVFP4_ERR_CUDA;
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return NVFP4_OK;
}

size_t skinny_ws(int64_t M, int64_t K, int n_weights) { return skinny_workspace_bytes(M, K, n_weights); }

bool size_ok(int64_t a, int64_t b) { return a >= 0 && b >= 0 && (b == 0 || a <= (INT64_C(1) << 62) / b); }

// Shared checks of the three product calls.
int check_product(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *codes,
                  const uint8_t *scales, const float *ts, const void *y, int out_dtype)
{
    if (N < 0 || M < 0 || K < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0 || !size_ok(N, K) || !size_ok(M, K) || !size_ok(N, M))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || M == 0)
        return NVFP4_OK;
    if (!y || !aligned(y, 16))
        return NVFP4_ERR_INVALID_ARG;
    if (K == 0)
        return NVFP4_OK;
    if (!x || !codes || !scales || !ts)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 16) || !aligned(ts, 4))
        return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

int check_workspace(const void *ws, size_t have, size_t need)
{
    if (have < need)
        return NVFP4_ERR_WORKSPACE;
    if (need > 0 && (!ws || !aligned(ws, 16)))
        return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

int zero_output(void *y, int64_t N, int64_t M, int out_dtype, cudaStream_t s)
{
    const size_t bytes = (size_t)N * (size_t)M * (out_dtype == NVFP4_OUT_BF16 ? 2 : 4);
    return cudaMemsetAsync(y, 0, bytes, s) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int run_products(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                 const uint8_t *const *scales, const float *const *ts, int n_weights, void *y, int out_dtype,
                 void *ws, cudaStream_t stream)
{
    int sms = 0;
    int rc = current_num_sms(&sms);
    if (rc != NVFP4_OK)
        return rc;
    // N <= 16: one skinny launch.  Larger N: tensor-core prefill.
    if (N <= kMaxSkinnyN) {
        cudaError_t e = launch_gemv(x, (int)N, M, K, codes, scales, ts, n_weights, y,
                                    out_dtype == NVFP4_OUT_BF16, ws, sms, stream);
        return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
    }
    cudaError_t e = launch_prefill(x, N, M, K, codes, scales, ts, n_weights, y, out_dtype == NVFP4_OUT_BF16,
                                   ws, sms, stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace

namespace nvfp4 {

int check_skinny_call(const uint16_t *x, int64_t N, const uint8_t *codes, const uint8_t *scales,
                      const float *tensor_scale, int64_t M, int64_t K, const void *y, int out_dtype,
                      bool *nothing_to_do)
{
    *nothing_to_do = false;
    int rc = check_product(x, N, M, K, codes, scales, tensor_scale, y, out_dtype);
    if (rc != NVFP4_OK)
        return rc;
    if (N < 1 || N > kMaxSkinnyN) {
        *nothing_to_do = N == 0;
        return N == 0 ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED_SHAPE;
    }
    *nothing_to_do = M == 0;
    return NVFP4_OK;
}

}  // namespace nvfp4

extern "C" {

const char *nvfp4_status_string(int status)
{
    switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG: null, negative, misaligned or unknown argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE: K % 16 != 0, N out of range or size overflow";
    case NVFP4_ERR_WORKSPACE: return "NVFP4_ERR_WORKSPACE: workspace smaller than nvfp4_workspace_bytes()";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA: a CUDA call or kernel launch failed";
    case NVFP4_ERR_DEVICE_TIMEOUT:
        return "NVFP4_ERR_DEVICE_TIMEOUT: a kernel's bounded pipeline wait gave up; outputs since the status "
               "word was last cleared are undefined";
    default: return "NVFP4 unknown status";
    }
}

int nvfp4_version(void) { return 100; }

size_t nvfp4_workspace_bytes(int op, int64_t N, int64_t M, int64_t K)
{
    if (N < 0 || M < 0 || K < 0 || K % 16 != 0)
        return 0;
    switch (op) {
    case NVFP4_OP_QUANTIZE: return (size_t)kQuantPartials * 4;
    case NVFP4_OP_GEMV_SKINNY: return (N >= 1 && N <= kMaxSkinnyN) ? skinny_ws(M, K, 1) : 0;
    case NVFP4_OP_GATEUP_SWIGLU: return N <= kMaxSkinnyN ? skinny_ws(M, K, 2) : prefill_workspace_bytes(N, M, K, 2, 0);
    case NVFP4_OP_GEMM_PREFILL: return N <= kMaxSkinnyN ? skinny_ws(M, K, 1) : prefill_workspace_bytes(N, M, K, 1, 0);
    case NVFP4_OP_FP6_GEMM:
    case NVFP4_OP_FP6_GATEUP_SWIGLU: {
        if (K % 128 != 0)
            return 0;
        const int nw = op == NVFP4_OP_FP6_GEMM ? 1 : 2;
        if (N > kMaxSkinnyN)
            return prefill_workspace_bytes(N, M, K, nw, 1);
        return skinny_tc_supported(M, K) ? skinny_tc_workspace_bytes(M, K, nw) : gemv_mma_workspace_bytes(nw);
    }
    default: return 0;
    }
}

int nvfp4_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales, float *tensor_scale,
                   void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    if (M < 0 || K < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0 || !size_ok(M, K))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!tensor_scale || !aligned(tensor_scale, 4))
        return NVFP4_ERR_INVALID_ARG;
    if (M * K > 0 && (!w || !codes || !scales || !aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 16)))
        return NVFP4_ERR_INVALID_ARG;
    int rc = check_workspace(workspace, workspace_bytes, nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE, 0, M, K));
    if (rc != NVFP4_OK)
        return rc;
    int sms = 0;
    rc = current_num_sms(&sms);
    if (rc != NVFP4_OK)
        return rc;
    cudaError_t e = launch_quantize(w, M, K, codes, scales, tensor_scale, workspace, sms, (cudaStream_t)stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int nvfp4_quantize_bf16(const uint16_t *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                        float *tensor_scale, void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    if (M < 0 || K < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0 || !size_ok(M, K))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!tensor_scale || !aligned(tensor_scale, 4))
        return NVFP4_ERR_INVALID_ARG;
    if (M * K > 0 && (!w || !codes || !scales || !aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 16)))
        return NVFP4_ERR_INVALID_ARG;
    int rc = check_workspace(workspace, workspace_bytes, nvfp4_workspace_bytes(NVFP4_OP_QUANTIZE, 0, M, K));
    if (rc != NVFP4_OK)
        return rc;
    int sms = 0;
    rc = current_num_sms(&sms);
    if (rc != NVFP4_OK)
        return rc;
    cudaError_t e = launch_quantize_bf16(w, M, K, codes, scales, tensor_scale, workspace, sms, (cudaStream_t)stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

size_t nvfp4_blocked_scale_bytes(int64_t M, int64_t K)
{
    if (M < 0 || K < 0 || K % 16 != 0 || !size_ok(M, K))
        return 0;
    return (size_t)((M + 127) / 128) * (size_t)((K / 16 + 3) / 4) * 512;
}

int nvfp4_import_blocked_scales(const uint8_t *blocked, int64_t M, int64_t K, uint8_t *scales,
                                nvfp4_stream_t stream)
{
    if (M < 0 || K < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0 || !size_ok(M, K))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || K == 0)
        return NVFP4_OK;
    if (!blocked || !scales || !aligned(blocked, 16) || !aligned(scales, 16))
        return NVFP4_ERR_INVALID_ARG;
    cudaError_t e = launch_import_blocked_scales(blocked, M, K, scales, (cudaStream_t)stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// FP6 E2M3 block-scaled weights
// ---------------------------------------------------------------------------

static int fp6_check_quantize(const void *w, int64_t M, int64_t K, const uint8_t *codes, const uint8_t *scales)
{
    if (M < 0 || K < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 128 != 0 || !size_ok(M, K))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M * K > 0 && (!w || !codes || !scales || !aligned(w, 16) || !aligned(codes, 16) || !aligned(scales, 16)))
        return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

int nvfp4_fp6_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                       nvfp4_stream_t stream)
{
    int rc = fp6_check_quantize(w, M, K, codes, scales);
    if (rc != NVFP4_OK || M * K == 0)
        return rc;
    int sms = 0;
    if ((rc = current_num_sms(&sms)) != NVFP4_OK)
        return rc;
    cudaError_t e = launch_fp6_quantize(w, M, K, codes, scales, sms, (cudaStream_t)stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int nvfp4_fp6_quantize_bf16(const uint16_t *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                            nvfp4_stream_t stream)
{
    int rc = fp6_check_quantize(w, M, K, codes, scales);
    if (rc != NVFP4_OK || M * K == 0)
        return rc;
    int sms = 0;
    if ((rc = current_num_sms(&sms)) != NVFP4_OK)
        return rc;
    cudaError_t e = launch_fp6_quantize_bf16(w, M, K, codes, scales, sms, (cudaStream_t)stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

static int fp6_products(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                        const uint8_t *const *scales, int n_weights, void *y, int out_dtype, void *ws,
                        size_t ws_bytes, cudaStream_t stream)
{
    if (N < 0 || M < 0 || K < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 128 != 0 || !size_ok(N, K) || !size_ok(M, K) || !size_ok(N, M))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || M == 0)
        return NVFP4_OK;
    if (!y || !aligned(y, 16))
        return NVFP4_ERR_INVALID_ARG;
    if (K > 0) {
        if (!x || !aligned(x, 16))
            return NVFP4_ERR_INVALID_ARG;
        for (int i = 0; i < n_weights; ++i)
            if (!codes[i] || !scales[i] || !aligned(codes[i], 16) || !aligned(scales[i], 16))
                return NVFP4_ERR_INVALID_ARG;
    }
    const int op = n_weights == 1 ? NVFP4_OP_FP6_GEMM : NVFP4_OP_FP6_GATEUP_SWIGLU;
    int rc = check_workspace(ws, ws_bytes, nvfp4_workspace_bytes(op, N, M, K));
    if (rc != NVFP4_OK)
        return rc;
    if (K == 0)
        return zero_output(y, N, M, out_dtype, stream);
    int sms = 0;
    if ((rc = current_num_sms(&sms)) != NVFP4_OK)
        return rc;
    const int bf16 = out_dtype == NVFP4_OUT_BF16;
    cudaError_t e;
    if (N > kMaxSkinnyN)
        e = launch_prefill_fp6(x, N, M, K, codes, scales, n_weights, y, bf16, ws, sms, stream);
    else if (skinny_tc_supported(M, K))
        e = launch_skinny_tc_fp6(x, (int)N, M, K, codes, scales, n_weights, y, bf16, ws, sms, stream);
    else
        e = launch_gemv_fp6(x, (int)N, M, K, codes, scales, n_weights, y, bf16, ws, sms, stream);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int nvfp4_fp6_gemm(const uint16_t *x, int64_t N, const uint8_t *codes, const uint8_t *scales, int64_t M, int64_t K,
                   void *y, int out_dtype, void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    const uint8_t *c[1] = {codes};
    const uint8_t *s[1] = {scales};
    return fp6_products(x, N, M, K, c, s, 1, y, out_dtype, workspace, workspace_bytes, (cudaStream_t)stream);
}

int nvfp4_fp6_gateup_swiglu(const uint16_t *x, int64_t N, const uint8_t *gate_codes, const uint8_t *gate_scales,
                            const uint8_t *up_codes, const uint8_t *up_scales, int64_t M, int64_t K, void *h,
                            int out_dtype, void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    const uint8_t *c[2] = {gate_codes, up_codes};
    const uint8_t *s[2] = {gate_scales, up_scales};
    return fp6_products(x, N, M, K, c, s, 2, h, out_dtype, workspace, workspace_bytes, (cudaStream_t)stream);
}

int nvfp4_gemv_skinny(const uint16_t *x, int64_t N, const uint8_t *codes, const uint8_t *scales,
                      const float *tensor_scale, int64_t M, int64_t K, void *y, int out_dtype, void *workspace,
                      size_t workspace_bytes, nvfp4_stream_t stream)
{
    bool nothing = false;
    int rc = nvfp4::check_skinny_call(x, N, codes, scales, tensor_scale, M, K, y, out_dtype, &nothing);
    if (rc != NVFP4_OK || nothing)
        return rc;
    rc = check_workspace(workspace, workspace_bytes, nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, N, M, K));
    if (rc != NVFP4_OK)
        return rc;
    if (K == 0)
        return zero_output(y, N, M, out_dtype, (cudaStream_t)stream);
    const uint8_t *c[1] = {codes};
    const uint8_t *s[1] = {scales};
    const float *t[1] = {tensor_scale};
    return run_products(x, N, M, K, c, s, t, 1, y, out_dtype, workspace, (cudaStream_t)stream);
}

int nvfp4_gateup_swiglu(const uint16_t *x, int64_t N, const uint8_t *gate_codes, const uint8_t *gate_scales,
                        const float *gate_tensor_scale, const uint8_t *up_codes, const uint8_t *up_scales,
                        const float *up_tensor_scale, int64_t M, int64_t K, void *h, int out_dtype,
                        void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    int rc = check_product(x, N, M, K, gate_codes, gate_scales, gate_tensor_scale, h, out_dtype);
    if (rc != NVFP4_OK)
        return rc;
    rc = check_product(x, N, M, K, up_codes, up_scales, up_tensor_scale, h, out_dtype);
    if (rc != NVFP4_OK)
        return rc;
    if (N == 0 || M == 0)
        return NVFP4_OK;
    rc = check_workspace(workspace, workspace_bytes, nvfp4_workspace_bytes(NVFP4_OP_GATEUP_SWIGLU, N, M, K));
    if (rc != NVFP4_OK)
        return rc;
    if (K == 0)  // g = u = 0 -> h = silu(0) * 0 = 0
        return zero_output(h, N, M, out_dtype, (cudaStream_t)stream);
    const uint8_t *c[2] = {gate_codes, up_codes};
    const uint8_t *s[2] = {gate_scales, up_scales};
    const float *t[2] = {gate_tensor_scale, up_tensor_scale};
    return run_products(x, N, M, K, c, s, t, 2, h, out_dtype, workspace, (cudaStream_t)stream);
}

int nvfp4_gemm_prefill(const uint16_t *x, int64_t N, const uint8_t *codes, const uint8_t *scales,
                       const float *tensor_scale, int64_t M, int64_t K, void *y, int out_dtype, void *workspace,
                       size_t workspace_bytes, nvfp4_stream_t stream)
{
    int rc = check_product(x, N, M, K, codes, scales, tensor_scale, y, out_dtype);
    if (rc != NVFP4_OK)
        return rc;
    if (N == 0 || M == 0)
        return NVFP4_OK;
    rc = check_workspace(workspace, workspace_bytes, nvfp4_workspace_bytes(NVFP4_OP_GEMM_PREFILL, N, M, K));
    if (rc != NVFP4_OK)
        return rc;
    if (K == 0)
        return zero_output(y, N, M, out_dtype, (cudaStream_t)stream);
    const uint8_t *c[1] = {codes};
    const uint8_t *s[1] = {scales};
    const float *t[1] = {tensor_scale};
    return run_products(x, N, M, K, c, s, t, 1, y, out_dtype, workspace, (cudaStream_t)stream);
}

// Status word checks shared by the two calls below: a workspace that holds it.
static int check_status_workspace(const void *workspace, size_t workspace_bytes)
{
    if (!workspace || !aligned(workspace, 16) || workspace_bytes < kStatusWordOffset + sizeof(uint32_t))
        return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

int nvfp4_device_status(const void *workspace, size_t workspace_bytes, int clear, uint32_t *code,
                        nvfp4_stream_t stream)
{
    int rc = check_status_workspace(workspace, workspace_bytes);
    if (rc != NVFP4_OK)
        return rc;
    uint8_t *word = const_cast<uint8_t *>(reinterpret_cast<const uint8_t *>(workspace)) + kStatusWordOffset;
    uint32_t v = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (clear && v != 0 && cudaMemsetAsync(word, 0, sizeof(v), s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (code)
        *code = v;
    return v == 0 ? NVFP4_OK : NVFP4_ERR_DEVICE_TIMEOUT;
}

int nvfp4_selftest_wait_timeout(void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    int rc = check_status_workspace(workspace, workspace_bytes);
    if (rc != NVFP4_OK)
        return rc;
    return launch_wait_timeout_selftest(workspace, (cudaStream_t)stream) == cudaSuccess ? NVFP4_OK
                                                                                        : NVFP4_ERR_CUDA;
}

}  // extern "C"
