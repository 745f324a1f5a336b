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
// The same recipe runs on bf16 input (values widened exactly to fp32).
//
// Two kernels, both HBM-bound (4 B, or 2 B for bf16, read per weight;
// 0.5625 B written):
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

// Input element types.  A bf16 value is exactly the fp32 value whose bits are
// its 16 bits followed by 16 zero bits, so both inputs feed the same fp32
// recipe below and give identical NVFP4 for the same values.
template <typename T> struct Src;

template <> struct Src<float> {
    static constexpr int kPer16B = 4;  // elements per 16-byte vector
    // Largest |value| bit pattern of one 16-byte vector (non-negative float
    // bits order like the values, so an integer max is exact).
    static __device__ __forceinline__ uint32_t amax_bits(uint4 v)
    {
        return max(max(v.x & 0x7FFFFFFFu, v.y & 0x7FFFFFFFu), max(v.z & 0x7FFFFFFFu, v.w & 0x7FFFFFFFu));
    }
    // Eight consecutive values starting at element 8 * hb: loaded raw (so
    // several half blocks can be in flight), then widened to fp32.
    static constexpr int kUnroll = 2;  // half blocks in flight per thread
    struct Raw {
        uint4 a, b;
    };
    static __device__ __forceinline__ Raw load_raw(const float *w, int64_t hb)
    {
        const uint4 *p = reinterpret_cast<const uint4 *>(w + hb * 8);
        return Raw{__ldcs(p), __ldcs(p + 1)};
    }
    static __device__ __forceinline__ void widen(const Raw &r, float v[8])
    {
        v[0] = __uint_as_float(r.a.x); v[1] = __uint_as_float(r.a.y);
        v[2] = __uint_as_float(r.a.z); v[3] = __uint_as_float(r.a.w);
        v[4] = __uint_as_float(r.b.x); v[5] = __uint_as_float(r.b.y);
        v[6] = __uint_as_float(r.b.z); v[7] = __uint_as_float(r.b.w);
    }
};

template <> struct Src<uint16_t> {
    static constexpr int kPer16B = 8;
    static __device__ __forceinline__ uint32_t half_bits(uint32_t word)
    {
        // the two bf16 values of a word as |fp32| bit patterns
        return max((word << 16) & 0x7FFF0000u, word & 0x7FFF0000u);
    }
    static __device__ __forceinline__ uint32_t amax_bits(uint4 v)
    {
        return max(max(half_bits(v.x), half_bits(v.y)), max(half_bits(v.z), half_bits(v.w)));
    }
    static constexpr int kUnroll = 4;  // half blocks in flight per thread (16 bytes each)
    struct Raw {
        uint4 a;
    };
    static __device__ __forceinline__ Raw load_raw(const uint16_t *w, int64_t hb)
    {
        return Raw{__ldcs(reinterpret_cast<const uint4 *>(w + hb * 8))};
    }
    static __device__ __forceinline__ void widen(const Raw &r, float v[8])
    {
        const uint32_t words[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(words[j] << 16);
            v[2 * j + 1] = __uint_as_float(words[j] & 0xFFFF0000u);
        }
    }
};

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
amax_partial_kernel(const uint4 *__restrict__ w, int64_t n_vec, uint32_t *__restrict__ partial)
{
    uint32_t m = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
         i += (int64_t)gridDim.x * blockDim.x)
        m = max(m, Src<T>::amax_bits(__ldcs(w + i)));
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

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
quantize_blocks_kernel(const T *__restrict__ w, int64_t n_half_blocks,
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
    // Each thread loads U half blocks (one grid stride apart) before it
    // quantises any, so U loads per thread are in flight.
    constexpr int U = Src<T>::kUnroll;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x - lane); base < n_half_blocks;
         base += stride * U) {
        typename Src<T>::Raw raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t hb = base + u * stride + lane;
            if (hb < n_half_blocks)
                raw[u] = Src<T>::load_raw(w, hb);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t hb = base + u * stride + lane;
            const bool active = hb < n_half_blocks;  // n_half_blocks is even: pairs are active together
            float v[8];
            float amax = 0.0f;
            if (active) {
                Src<T>::widen(raw[u], v);
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
}

template <typename T>
static cudaError_t quantize_any(const T *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                float *tensor_scale, void *workspace, int num_sms, cudaStream_t stream)
{
    const int64_t n = M * K;
    uint32_t *partial = reinterpret_cast<uint32_t *>(workspace);
    const int64_t n_vec = n / Src<T>::kPer16B;  // K % 16 == 0: whole vectors
    int64_t want = (n_vec + kQuantThreads * 8 - 1) / (kQuantThreads * 8);
    int grid_a = (int)std::min<int64_t>(std::max<int64_t>(want, 1), kQuantPartials);
    amax_partial_kernel<T><<<grid_a, kQuantThreads, 0, stream>>>(reinterpret_cast<const uint4 *>(w), n_vec,
                                                                  partial);
    const int64_t n_half = n / 8;
    int64_t blocks_b = (n_half + kQuantThreads - 1) / kQuantThreads;
    // four CTAs of 256 threads fit an SM at this kernel's register count:
    // one resident round, each thread looping over its half blocks
    int grid_b = (int)std::min<int64_t>(std::max<int64_t>(blocks_b, 1), (int64_t)num_sms * 4);
    quantize_blocks_kernel<T><<<grid_b, kQuantThreads, 0, stream>>>(w, n_half, partial, grid_a, codes, scales,
                                                                     tensor_scale);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, void *workspace, int num_sms, cudaStream_t stream)
{
    return quantize_any<float>(w, M, K, codes, scales, tensor_scale, workspace, num_sms, stream);
}

cudaError_t launch_quantize_bf16(const uint16_t *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                 float *tensor_scale, void *workspace, int num_sms, cudaStream_t stream)
{
    return quantize_any<uint16_t>(w, M, K, codes, scales, tensor_scale, workspace, num_sms, stream);
}

// ---------------------------------------------------------------------------
// FP6 E2M3 quantiser (block-scaled variant, one UE8M0 scale per 128 k).
//
//   shared = max(floor(log2(block amax)) - 2, -127)   (-127 for a zero block)
//   scale byte = shared + 127
//   code = nearest E2M3 value to w / 2^shared, ties to the even code,
//          saturating at 7.5, sign kept
// One warp per 128-element block, four consecutive elements per lane; the
// codes form a little-endian 6-bit stream per row (4 codes = 3 bytes), which
// the warp assembles with shuffles into 24 aligned 32-bit stores.  One pass:
// no tensor-wide amax.  HBM-bound: 4 B (fp32) or 2 B (bf16) read and 0.7578 B
// written per weight.

// E2M3 code of an fp32 value.  On [0, 2) the grid step is 1/8 and the code
// magnitude is the step count, on [2, 4) the step is 1/4 (code 8 + 4a), on
// [4, 7.5] 1/2 (code 16 + 2a); the scalings by 8, 4, 2 are exact, rintf rounds
// half to even, which on each range is the even code.  7.5 and above -> 31.
NVFP4_DEVINL uint32_t f32_to_e2m3(float q)
{
    const float a = fabsf(q);
    uint32_t mag;
    if (a >= 7.5f)
        mag = 31u;
    else if (a < 2.0f)
        mag = (uint32_t)rintf(a * 8.0f);
    else if (a < 4.0f)
        mag = (uint32_t)rintf(a * 4.0f) + 8u;
    else
        mag = (uint32_t)rintf(a * 2.0f) + 16u;
    return mag | ((__float_as_uint(q) >> 26) & 0x20u);
}

template <typename T> struct Src4;  // four consecutive elements of one lane
template <> struct Src4<float> {
    static __device__ __forceinline__ void load(const float *w, int64_t i, float v[4])
    {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(w + i));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
};
template <> struct Src4<uint16_t> {
    static __device__ __forceinline__ void load(const uint16_t *w, int64_t i, float v[4])
    {
        const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(w + i));
        v[0] = __uint_as_float(a.x << 16); v[1] = __uint_as_float(a.x & 0xFFFF0000u);
        v[2] = __uint_as_float(a.y << 16); v[3] = __uint_as_float(a.y & 0xFFFF0000u);
    }
};

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
fp6_quantize_kernel(const T *__restrict__ w, int64_t n_blocks, uint8_t *__restrict__ codes,
                    uint8_t *__restrict__ scales)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kQuantThreads / 32);
    for (int64_t blk = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5); blk < n_blocks;
         blk += warps) {
        float v[4];
        Src4<T>::load(w, blk * 128 + 4 * lane, v);
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = max(m, __float_as_uint(v[j]) & 0x7FFFFFFFu);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        // floor(log2(amax)) from the bit pattern (normal or subnormal amax)
        int shared = -127;
        if (m != 0) {
            const int e = (int)(m >> 23);
            const int fl = e != 0 ? e - 127 : (31 - __clz((int)m)) - 149;
            shared = max(fl - 2, -127);
        }
        // 2^-shared is a normal fp32 (-shared <= 127), and w * 2^-shared is the
        // same correctly rounded real number as w / 2^shared.
        const float inv = __uint_as_float((uint32_t)(127 - shared) << 23);
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            packed |= f32_to_e2m3(__fmul_rn(v[j], inv)) << (6 * j);
        // 24 bits per lane -> word l of the block's 96 bytes holds bytes
        // 4l .. 4l+3, which start at byte (4l) % 3 of lane (4l) / 3.
        const int src = min((4 * lane) / 3, 30);
        const int off = (4 * lane) % 3;
        const uint32_t va = __shfl_sync(0xFFFFFFFFu, packed, src);
        const uint32_t vb = __shfl_sync(0xFFFFFFFFu, packed, src + 1);
        const uint32_t word = (va >> (8 * off)) | (vb << (24 - 8 * off));
        if (lane < 24)
            reinterpret_cast<uint32_t *>(codes + blk * 96)[lane] = word;
        if (lane == 0)
            scales[blk] = (uint8_t)(shared + 127);
    }
}

template <typename T>
static cudaError_t fp6_quantize_any(const T *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                    int num_sms, cudaStream_t stream)
{
    const int64_t n_blocks = M * (K / 128);
    const int64_t want = (n_blocks + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
    const int grid = (int)std::min<int64_t>(std::max<int64_t>(want, 1), (int64_t)num_sms * 16);
    fp6_quantize_kernel<T><<<grid, kQuantThreads, 0, stream>>>(w, n_blocks, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_fp6_quantize(const float *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                int num_sms, cudaStream_t stream)
{
    return fp6_quantize_any<float>(w, M, K, codes, scales, num_sms, stream);
}

cudaError_t launch_fp6_quantize_bf16(const uint16_t *w, int64_t M, int64_t K, uint8_t *codes, uint8_t *scales,
                                     int num_sms, cudaStream_t stream)
{
    return fp6_quantize_any<uint16_t>(w, M, K, codes, scales, num_sms, stream);
}

// ---------------------------------------------------------------------------
// Import of block scales from the blocked (128 x 4) layout.
//
// Blocked layout: 128-row x 4-scale-column blocks, row-major over
// (ceil(M/128), ceil(S/4)) with S = K/16; inside a block, scale (r, c) at byte
// (r % 32) * 16 + (r / 32) * 4 + c.  Entries past M or S are padding.
//
// One CTA per (128-row block, chunk of kImportBlocks scale-column blocks): the
// chunk is contiguous in the blocked buffer (read with 16-byte loads into
// shared memory), and its 128 output row segments are written with 16-byte
// stores when rows start on 16-byte boundaries (S % 16 == 0; the output
// buffer itself is 16-byte aligned by the call's contract), else with 4-byte
// stores where rows start on 4-byte boundaries, else byte by byte.
// HBM-bound: every byte read and written once.
constexpr int kImportThreads = 256;
constexpr int kImportBlocks = 16;  // 4-column blocks per CTA: 64 columns, 8 KB

__global__ void __launch_bounds__(kImportThreads)
import_blocked_scales_kernel(const uint8_t *__restrict__ blocked, int64_t M, int64_t S, int64_t nb,
                             int64_t n_chunks, uint8_t *__restrict__ scales)
{
    __shared__ __align__(16) uint32_t tile[kImportBlocks * 128];
    const int64_t mb = blockIdx.x / n_chunks;
    const int64_t kb0 = (blockIdx.x % n_chunks) * kImportBlocks;
    const int nblk = (int)(nb - kb0 < kImportBlocks ? nb - kb0 : kImportBlocks);
    const uint4 *src = reinterpret_cast<const uint4 *>(blocked + (mb * nb + kb0) * 512);
    for (int i = threadIdx.x; i < nblk * 32; i += kImportThreads)
        reinterpret_cast<uint4 *>(tile)[i] = __ldcs(src + i);
    __syncthreads();

    if ((S & 15) == 0) {
        // Rows start on 16-byte boundaries: piece p = (row r, 16 scale
        // columns q of the chunk) is four words, one from each of four
        // consecutive blocks, written with one 16-byte store; a warp's 32
        // pieces cover 8 rows x 64 contiguous bytes.
        for (int p = threadIdx.x; p < 128 * (kImportBlocks / 4); p += kImportThreads) {
            const int r = p / (kImportBlocks / 4), q = p % (kImportBlocks / 4);
            const int64_t m = mb * 128 + r;
            const int64_t c = kb0 * 4 + 16 * q;
            if (m >= M || c >= S || 4 * q >= nblk)
                continue;
            const int w = (r & 31) * 4 + (r >> 5);  // word of row r inside a block
            const uint4 v = make_uint4(tile[(4 * q + 0) * 128 + w], tile[(4 * q + 1) * 128 + w],
                                       tile[(4 * q + 2) * 128 + w], tile[(4 * q + 3) * 128 + w]);
            *reinterpret_cast<uint4 *>(scales + m * S + c) = v;
        }
        return;
    }
    // Other S: thread t writes row t / 2, scale columns [32 * (t % 2), +32) of the chunk.
    const int r = threadIdx.x >> 1;
    const int64_t m = mb * 128 + r;
    if (m >= M)
        return;
    const int64_t c0 = kb0 * 4 + (threadIdx.x & 1) * 32;
    uint8_t *row = scales + m * S;
    const int widx = (r & 31) * 4 + (r >> 5);  // word of row r inside a block
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t c = c0 + 4 * j;
        if (c >= S)
            break;
        const int blk = (int)(c / 4 - kb0);
        const uint32_t word = tile[blk * 128 + widx];
        if ((S & 3) == 0) {
            *reinterpret_cast<uint32_t *>(row + c) = word;
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (c + b < S)
                    row[c + b] = (uint8_t)(word >> (8 * b));
        }
    }
}

cudaError_t launch_import_blocked_scales(const uint8_t *blocked, int64_t M, int64_t K, uint8_t *scales,
                                         cudaStream_t stream)
{
    const int64_t S = K / 16;
    const int64_t nb = (S + 3) / 4;
    const int64_t n_chunks = (nb + kImportBlocks - 1) / kImportBlocks;
    const int64_t grid = ((M + 127) / 128) * n_chunks;
    if (grid > 0x7FFFFFFF)
        return cudaErrorInvalidConfiguration;
    import_blocked_scales_kernel<<<(unsigned)grid, kImportThreads, 0, stream>>>(blocked, M, S, nb, n_chunks,
                                                                               scales);
    return cudaGetLastError();
}

}  // namespace nvfp4
