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
// cudaGetSymbolAddress once per device, with that device current, on the first
// call made on that device, and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"

namespace {

constexpr size_t kScratchBytes = NVFP4_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; keeps the last call's contents.  Static
// device memory starts zero-filled when the module loads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_address[kMaxDevices];  // device address of g_noalloc_scratch per device

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return NVFP4_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" int nvfp4_gemv_skinny_noalloc(const uint16_t *x, int64_t N, const uint8_t *codes,
                                         const uint8_t *scales, const float *tensor_scale, int64_t M,
                                         int64_t K, void *y, int out_dtype, nvfp4_stream_t stream)
{
    // Problems whose scratch would not fit the fixed array are refused before
    // anything runs.
    if (nvfp4_workspace_bytes(NVFP4_OP_GEMV_SKINNY, N, M, K) > kScratchBytes)
        return NVFP4_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != NVFP4_OK)
        return rc;
    return nvfp4_gemv_skinny(x, N, codes, scales, tensor_scale, M, K, y, out_dtype, scratch, kScratchBytes,
                             stream);
}
