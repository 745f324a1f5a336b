// quantize.cu -- fp32 weights -> NVFP4 (E2M1 codes, E4M3 block scales, fp32
// tensor scale), bit-exact with the recipe:
//   ts    = amax / 2688                           (fp32 division)
//   q     = (block_amax / 6) / ts                 (two fp32 divisions, in order)
//   scale = E4M3 round-to-nearest-even of q, saturating at 448
//   d     = e4m3(scale) * ts                      (one fp32 rounding)
//   code  = E2M1 round-to-nearest-even of w / d   (fp32 division), clamp +-6;
//           d == 0 gives code 0.
// NVFP4 is the format both engines on the pages stream (bw24 README, NVFP4 /
// Q4_0 decode path; qwentin README, "Why it's interesting", E2M1 4-bit mode),
// and qwentin quantises and packs on the GPU through its C ABI (qwentin README,
// converter section).
//
// Two kernels, both HBM-bound (4 B read per weight; 0.5625 B written):
//   1. amax_partial: per-block max of |w| bit patterns (integer max on the
//      non-negative float bits is exact and order independent) -> workspace.
//   2. quantize_blocks: every CTA reduces the partial maxima itself (no
//      atomics, no host sync, no workspace initialisation), derives ts, and
//      quantises 16-element blocks, two threads per block.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
amax_partial_kernel(const float4 *__restrict__ w, int64_t n_vec4, uint32_t *__restrict__ partial)
{
    uint32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 v = __ldcs(w + i);
        m = max(m, __float_as_uint(v.x) & 0x7FFFFFFFu);
        m = max(m, __float_as_uint(v.y) & 0x7FFFFFFFu);
        m = max(m, __float_as_uint(v.z) & 0x7FFFFFFFu);
        m = max(m, __float_as_uint(v.w) & 0x7FFFFFFFu);
    }
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __shared__ uint32_t red[kQuantThreads / 32];
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int i = 0; i < kQuantThreads / 32; ++i)
            r = max(r, red[i]);
        partial[blockIdx.x] = r;
    }
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_blocks_kernel(const float *__restrict__ w, int64_t n_half_blocks,
                       const uint32_t *__restrict__ partial, int n_partial,
                       uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                       float *__restrict__ tensor_scale)
{
    // Tensor amax from the partial maxima (every CTA does the same reduction).
    __shared__ float s_ts;
    if (threadIdx.x < 32) {
        uint32_t m = 0;
        for (int i = threadIdx.x; i < n_partial; i += 32)
            m = max(m, partial[i]);
        for (int o = 16; o > 0; o >>= 1)
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (threadIdx.x == 0) {
            float ts = __fdiv_rn(__uint_as_float(m), 2688.0f);
            s_ts = ts;
            if (blockIdx.x == 0)
                *tensor_scale = ts;
        }
    }
    __syncthreads();
    const float ts = s_ts;

    // Two threads per 16-element block; each holds 8 consecutive weights.  The
    // loop runs warp-uniformly so the pair shuffle always has all 32 lanes.
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x - lane); base < n_half_blocks;
         base += stride) {
        const int64_t hb = base + lane;
        const bool active = hb < n_half_blocks;  // n_half_blocks is even: pairs are active together
        float v[8];
        float amax = 0.0f;
        if (active) {
            const float4 *p = reinterpret_cast<const float4 *>(w + hb * 8);
            float4 a = __ldcs(p), b = __ldcs(p + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                amax = fmaxf(amax, fabsf(v[j]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        if (!active)
            continue;

        uint32_t sb = 0;
        if (ts > 0.0f) {
            float q = __fdiv_rn(__fdiv_rn(amax, 6.0f), ts);
            sb = f32_to_e4m3_satfinite(q);
        }
        const float d = __fmul_rn(e4m3_to_f32(sb), ts);

        uint32_t packed = 0;
        if (d != 0.0f) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo = __fdiv_rn(v[2 * j], d);
                float hi = __fdiv_rn(v[2 * j + 1], d);
                packed |= f32x2_to_e2m1x2(lo, hi) << (8 * j);
            }
        }
        reinterpret_cast<uint32_t *>(codes)[hb] = packed;
        if ((hb & 1) == 0)
            scales[hb >> 1] = (uint8_t)sb;
    }
}

cudaError_t launch_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, void *workspace, int num_sms, cudaStream_t stream)
{
    const int64_t n = M * K;
    uint32_t *partial = reinterpret_cast<uint32_t *>(workspace);
    int64_t want = (n / 4 + kQuantThreads * 8 - 1) / (kQuantThreads * 8);
    int grid_a = (int)std::min<int64_t>(std::max<int64_t>(want, 1), kQuantPartials);
    amax_partial_kernel<<<grid_a, kQuantThreads, 0, stream>>>(reinterpret_cast<const float4 *>(w), n / 4,
                                                               partial);
    const int64_t n_half = n / 8;
    int64_t blocks_b = (n_half + kQuantThreads - 1) / kQuantThreads;
    int grid_b = (int)std::min<int64_t>(std::max<int64_t>(blocks_b, 1), (int64_t)num_sms * 8);
    quantize_blocks_kernel<<<grid_b, kQuantThreads, 0, stream>>>(w, n_half, partial, grid_a, codes, scales,
                                                                  tensor_scale);
    return cudaGetLastError();
}

}  // namespace nvfp4
