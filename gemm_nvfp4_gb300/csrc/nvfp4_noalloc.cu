// nvfp4_noalloc.cu -- the skinny product for callers that cannot allocate
// device memory.
//
// nvfp4_gemv_skinny needs a caller-provided workspace for the partial sums of
// rows whose K range is split across thread blocks.  Some callers have no way
// to provide one at the point of the call: a plain C or Fortran host program
// that links the library but owns no device allocator, code that must not call
// cudaMalloc because it synchronises the whole device (a latency-critical
// decode loop), or code running where allocation is not allowed at all.  For
// them this file keeps the scratch in the library's own device memory: a
// fixed, file-scope __device__ array of NVFP4_NOALLOC_SCRATCH_BYTES that every
// GPU loading the library holds until the process exits.
//
// Host code cannot use the array's name as a device pointer (in host code it
// names a host-side stand-in), so the device address is looked up with
// cudaGetSymbolAddress with the device current.  The lookup is cached per
// device together with the identity of the CUDA context it was made in: after
// cudaDeviceReset (or from another context) the module is loaded again and
// the array may sit at a new address, so a changed context repeats the lookup.
//
// The array also holds the device status word and the split-K counters of the
// skinny kernels, like any skinny workspace.  The caller never sees its
// address, so nvfp4_noalloc_status reads (and clears) that word, and on clear
// zero-fills the whole array, which restores the counters a timed-out call may
// have left behind; nvfp4_noalloc_selftest_wait_timeout runs the bounded-wait
// self-test against it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = NVFP4_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; keeps the last call's contents.  Static
// device memory starts zero-filled when the module loads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct CachedAddress {
    unsigned long long ctx_id;
    void *address;
};
CachedAddress g_scratch[kMaxDevices];  // per device: context id and device address of the array

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current CUDA context (0 if unknown).
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device.  The first call
// in a context does the set-up (a host-side symbol lookup that allocates
// nothing); later calls in the same context reuse it.
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_CUDA;
    // 0 when no context is current yet: the lookup below creates the device's
    // primary context, and the id is read again after it
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    CachedAddress &c = g_scratch[dev];
    if (c.address == nullptr || ctx == 0 || c.ctx_id != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return NVFP4_ERR_CUDA;
        c.address = p;
        c.ctx_id = current_context_id();
    }
    *out = c.address;
    return NVFP4_OK;
}

}  // namespace

extern "C" int nvfp4_gemv_skinny_noalloc(const uint16_t *x, int64_t N, const uint8_t *codes,
                                         const uint8_t *scales, const float *tensor_scale, int64_t M,
                                         int64_t K, void *y, int out_dtype, nvfp4_stream_t stream)
{
    // The same host checks as nvfp4_gemv_skinny come first, so a bad argument
    // gives the same status and touches no CUDA state.
    bool nothing = false;
    int rc = nvfp4::check_skinny_call(x, N, codes, scales, tensor_scale, M, K, y, out_dtype, &nothing);
    if (rc != NVFP4_OK || nothing)
        return rc;
    // Problems whose scratch would not fit the fixed array are refused before
    // anything runs.
    if (nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, N, M, K) > kScratchBytes)
        return NVFP4_ERR_WORKSPACE;
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != NVFP4_OK)
        return rc;
    return nvfp4_gemv_skinny(x, N, codes, scales, tensor_scale, M, K, y, out_dtype, scratch, kScratchBytes,
                             stream);
}

extern "C" int nvfp4_noalloc_status(int clear, uint32_t *code, nvfp4_stream_t stream)
{
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != NVFP4_OK)
        return rc;
    uint32_t v = 0;
    cudaStream_t s = (cudaStream_t)stream;
    const uint8_t *word = reinterpret_cast<const uint8_t *>(scratch) + nvfp4::kStatusWordOffset;
    if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    // A failed call can leave split-K counters set as well as the word:
    // zero-fill the whole array, its state when the library was loaded.
    if (clear && v != 0 && cudaMemsetAsync(scratch, 0, kScratchBytes, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (code)
        *code = v;
    return v == 0 ? NVFP4_OK : NVFP4_ERR_DEVICE_TIMEOUT;
}

extern "C" int nvfp4_noalloc_selftest_wait_timeout(nvfp4_stream_t stream)
{
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != NVFP4_OK)
        return rc;
    return nvfp4::launch_wait_timeout_selftest(scratch, (cudaStream_t)stream) == cudaSuccess ? NVFP4_OK
                                                                                              : NVFP4_ERR_CUDA;
}
