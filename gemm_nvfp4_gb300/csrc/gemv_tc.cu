// gemv_tc.cu -- skinny NVFP4 x bf16 products (N = 1..16 tokens) on the
// tcgen05 tensor cores, for K a multiple of 256.
//
// What it computes is the decode matvec / batched verify of the pages (bw24
// README, NVFP4 decode path and speculative decoding sections; qwentin README,
// "Highlights", verify reading each weight once for the whole draft tree):
//   y[n][m] = ts * sum_k e2m1(code[m][k]) * e4m3(scale[m][k/16]) * x[n][k].
//
// Why this shape on GB300: measured on the GB300s used here, the integer and
// half-precision ALU instructions issue at 16 lanes/clk/SMSP and legacy
// mma.sync tops out near 200 TFLOP/s, so a register-dequant + mma.sync kernel
// cannot keep up with HBM.  Here the CUDA cores only dequantise (one hardware
// E2M1 -> f16x2 conversion and one f16x2 scale multiply per two weights) into
// tensor memory, and tcgen05.mma (A from TMEM, B from shared memory) does the
// products:
//
//   prep kernel  x (bf16) -> x' = x * 2^s_n in f16 for each token n, with s_n
//                chosen so max|x'_n| is in [2^15, 2^16).  If any element of
//                any token is not exact in f16, the call falls back to bf16
//                operands (slower dequant, same exact products).  Also zeroes
//                the split-K counters.
//   main kernel  one CTA per SM, stream-K over units (tile of 128 rows,
//                128 k) so every SM streams the same bytes:
//     warp 0     TMA: code tile [128 rows][64 B] (64-byte swizzle) and scale
//                tile [128 rows][16 B] per unit into an 8-deep ring.  It does
//                not depend on the prep kernel, so it starts streaming weights
//                while the previous kernel and the prep kernel still run.
//     warp 2     TMA: activation tile [16 tokens][128 k] (128-byte swizzle).
//     warps 3-10 dequantise: thread = weight row = TMEM lane; codes and scales
//                from shared memory -> f16x2 (or bf16x2) -> tcgen05.st into a
//                TMEM ring of A operands; group 0 also runs the epilogue.
//     warp 1     allocates TMEM; one thread issues tcgen05.mma kind::f16
//                (M=128, N=16, K=16, A in TMEM) into a double-buffered fp32
//                accumulator in TMEM.
//   A tile split across CTAs is finished by the last CTA to arrive (counter in
//   the workspace), which adds the partials in CTA order: deterministic.
//
// Every product is exact in the fp32 accumulator (f16 operands: at most 6 and
// 8 significant bits; bf16 fallback likewise).  All waits are bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace sk {

constexpr int BM = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int BKU = 256;         // k per unit (one code box per matrix)
constexpr int kScaleUnits = 4;   // units covered by one scale box (1024 k)
constexpr int NTOK = 16;         // MMA N (tokens, padded)
// Warp roles: 0..3 MMA issuers (one per SM sub-partition), 4 and 5 code
// producers (even / odd units), 6 scale producer, 7 activation producer,
// 8..23 dequantisers (four groups of four warps, one warp per TMEM lane
// quarter).  Several producer threads are used because one thread issuing TMA
// copies back to back tops out well below HBM bandwidth on GB300, while two to
// four issuing threads reach it.  Several MMA issuers are used because a
// thread issuing tcgen05.mma competes for issue slots with the dequantiser
// warps of its sub-partition; N = 16 MMAs are short, so issue rate matters.
constexpr int kMmaWarps = 4;
constexpr int kFirstDqWarp = 8;
constexpr int kDqWarps = 16;
constexpr int kThreads = (kFirstDqWarp + kDqWarps) * 32;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kEpiThreads = 128;     // the first dequantiser group
constexpr int kCodeBox = BM * 128;   // 16 KB: 128 rows x 128 code bytes (256 k), 128-byte swizzle
constexpr int kScaleBox = BM * 64;   // 8 KB: 128 rows x 64 scale bytes (1024 k), 64-byte swizzle
constexpr int kXUnit = NTOK * BKU * 2;  // 8 KB: activation image of one unit
constexpr uint32_t kTmemCols = 512;

template <int NW>
struct Cfg {
    // The code ring holds most of the shared memory: with ~4 us of loaded
    // DRAM latency, every SM needs well over 100 KB of weights in flight.
    static constexpr int kCStages = NW == 1 ? 10 : 5;  // code ring (units)
    static constexpr int kSStages = 2;                  // scale ring (kScaleUnits units each)
    static constexpr int kXStages = NW == 1 ? 4 : 3;   // activation ring (units, from L2)
    // One unit = kSubs TMEM A sub-stages of 128 columns.  Group g of the
    // dequantisers fills columns [col0(g), +kGroupCols) of sub-stage sub(g).
    //   NW = 1: 1 sub-stage of 256 k; group g fills k [64g, 64g+64) (32 columns).
    //   NW = 2: 2 sub-stages of 128 k x 2 matrices; group g fills matrix g/2,
    //           sub-stage g%2 (64 columns).
    static constexpr int kSubs = NW;
    static constexpr int kSubK = BKU / kSubs;
    static constexpr int kAFullCount = kDqWarps / kSubs;  // one arrival per dequantiser warp
    static constexpr int kAStages = 3;                 // TMEM A ring (128 columns each)
    static constexpr int kACols = 128;
    // Independent accumulation chains per matrix: issuer q accumulates matrix
    // q / kChains over the K steps kk = q % kChains (mod kChains) into its own
    // chain; the epilogue adds the chains in a fixed order.
    static constexpr int kChains = kMmaWarps / NW;
    static constexpr int kDCols = 16 * NW * kChains;   // one accumulator buffer
    static constexpr size_t kSmemBytes = (size_t)kCStages * NW * kCodeBox + (size_t)kSStages * NW * kScaleBox +
                                         (size_t)kXStages * kXUnit + 1024 + 1024;
    static_assert(kAStages * kACols + 2 * kDCols <= (int)kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Args {
    int N;
    int64_t M, K;
    int C;            // units per tile
    int64_t T;        // tiles
    int64_t total;    // T * C
    int P;            // CTAs
    const float *ts[2];
    const float *factor;   // [16] 2^-s_n
    const int *flags;      // [16] 1 if token n is not exact in f16
    uint32_t *counters;    // [T][128] per-row arrival counters
    float *partial;        // [P][2][NW][16][128]
    const uint8_t *x_img;  // [C][8 KB] f16 activation image (shared-memory layout)
    uint32_t *err;
    void *y;
    int out_bf16;
};

// Workspace layout (bytes): header 256 (factor[16], flags[16], err), per-row
// counters, the f16 activation image, split-K partials.
struct WsLayout {
    size_t counters, ximg, partial, total;
};

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(int64_t M, int64_t K, int nw)
{
    WsLayout w;
    const int64_t T = (M + BM - 1) / BM;
    const int64_t C = (K + BKU - 1) / BKU;
    w.counters = 256;
    w.ximg = w.counters + round_up((size_t)T * BM * 4, 1024);
    w.partial = w.ximg + (size_t)C * kXUnit;
    w.total = w.partial + (size_t)kSkinnyTcMaxCtas * 2 * nw * NTOK * BM * 4;
    return w;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

// Four E2M1 pairs (one code word, k = 0..7) -> f16x2 in natural k order.
NVFP4_DEVINL void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4])
{
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
        " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
        " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

NVFP4_DEVINL uint32_t f16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// bf16 path (fallback): exact bf16 values e2m1 * scale * 2^-8, natural order.
NVFP4_DEVINL void e2m1x8_to_bf16x2(uint32_t w, uint32_t mult, uint32_t (&o)[4])
{
    constexpr uint32_t kMag = 0x01C001C0u;
    const uint32_t te = w & 0x08080808u;
    const uint32_t to = w & 0x80808080u;
    const uint32_t p0 = bf16x2_mul(((w << 6) & kMag) | ((te << 12) & ~kMag), mult);
    const uint32_t p1 = bf16x2_mul(((w << 2) & kMag) | ((to << 8) & ~kMag), mult);
    const uint32_t p2 = bf16x2_mul(((w >> 2) & kMag) | ((te << 4) & ~kMag), mult);
    const uint32_t p3 = bf16x2_mul(((w >> 6) & kMag) | (to & ~kMag), mult);
    o[0] = prmt(p0, p1, 0x5410);
    o[1] = prmt(p2, p3, 0x5410);
    o[2] = prmt(p0, p1, 0x7632);
    o[3] = prmt(p2, p3, 0x7632);
}

NVFP4_DEVINL uint32_t bf16_scale_mult(uint32_t byte)
{
    return f32_to_bf16x2_bcast(__fmul_rn(e4m3_to_f32(byte & 0xFF), 0x1p118f));
}

// Dequantise one 16-byte chunk of codes (32 k) with its two scale bytes into
// 16 words (f16x2 or bf16x2), natural k order.
NVFP4_DEVINL void dequant_chunk(uint4 c, uint32_t sc2, int mode, uint32_t *out)
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    if (mode == 0) {
        const uint32_t s2 = e4m3x2_to_f16x2((uint16_t)(sc2 & 0xFFFF));  // {s0, s1}
        const uint32_t sb[2] = {prmt(s2, s2, 0x1010), prmt(s2, s2, 0x3232)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t o[4];
            e2m1x8_to_f16x2(w[q], o);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                out[4 * q + e] = f16x2_mul(o[e], sb[q >> 1]);
        }
    } else {
        const uint32_t mb[2] = {bf16_scale_mult(sc2 & 0xFF), bf16_scale_mult((sc2 >> 8) & 0xFF)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t o[4];
            e2m1x8_to_bf16x2(w[q], mb[q >> 1], o);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                out[4 * q + e] = o[e];
        }
    }
}

// Stream-K partition in 32-bit arithmetic (the host keeps total * P < 2^31):
// CTA b owns units [b * total / P, (b + 1) * total / P).
NVFP4_DEVINL int cta_of(uint32_t q, uint32_t total, uint32_t P) { return (int)(((q + 1) * P - 1) / total); }
NVFP4_DEVINL uint32_t cta_lo(uint32_t b, uint32_t total, uint32_t P) { return b * total / P; }

NVFP4_DEVINL uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

NVFP4_DEVINL void fail(const Args &a, uint32_t code) { atomicExch(a.err, code); }

NVFP4_DEVINL int load_mode(const Args &a)
{
    int f = 0;
    for (int n = 0; n < a.N; ++n)
        f |= a.flags[n];
    return f ? 1 : 0;
}

NVFP4_DEVINL float silu_mul(float g, float u) { return __fdiv_rn(g, 1.0f + expf(-g)) * u; }

NVFP4_DEVINL void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(tc::smem_addr(dst)), "l"(src), "r"(bytes), "r"(tc::smem_addr(bar))
                 : "memory");
}


// ---------------------------------------------------------------------------
// prep kernel: activation images + per-token power of two + exactness flags
// ---------------------------------------------------------------------------

// Byte offset of element (token n, k) in the activation image: units of 256 k,
// each 4 sub-boxes of [16 tokens][64 k] with the 128-byte swizzle applied, so a
// unit is copied to shared memory verbatim and read by the MMA as a K-major
// 128-byte-swizzled operand.
NVFP4_DEVINL int64_t ximg_offset(int n, int64_t k)
{
    const int64_t u = k / BKU;
    const int kl = (int)(k % BKU);
    const int sb = kl >> 6, c = (kl >> 3) & 7, e = kl & 7;
    return u * kXUnit + sb * (NTOK * 128) + n * 128 + ((c ^ (n & 7)) << 4) + e * 2;
}

constexpr int kPrepThreads = 512;
constexpr int kPrepCache = 4;  // 16-byte chunks per thread kept in registers between the passes

// One block per token n < N: per-token power of two s (max|x| * 2^s in
// [2^15, 2^16)), the f16 image of x * 2^s in the shared-memory layout of the
// main kernel, and the exactness flag (any element not exact in f16 after the
// scaling -> the call uses bf16 operands and reads x itself).  All blocks also
// zero the split-K row counters.
__global__ void __launch_bounds__(kPrepThreads) skinny_prep_kernel(const uint16_t *__restrict__ x, int N, int64_t K,
                                                                   uint8_t *__restrict__ ximg, float *factor,
                                                                   int *flags, uint32_t *counters, int64_t T,
                                                                   uint32_t *err)
{
    tc::griddep_launch_dependents();
    tc::griddep_wait();  // x may come from the previous kernel; the workspace may be in use by it
    const int n = blockIdx.x;
    const int tid = threadIdx.x;
    for (int64_t i = (int64_t)n * kPrepThreads + tid; i < T * BM; i += (int64_t)N * kPrepThreads)
        counters[i] = 0;
    if (n == 0 && tid == 0)
        *err = 0;
    __shared__ uint32_t red[kPrepThreads / 32];
    __shared__ int bad;
    const uint16_t *xr = x + (int64_t)n * K;
    uint4 cache[kPrepCache];
    uint32_t m = 0;
    auto vmax = [&](const uint4 &v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m = max(m, w[i] & 0x7FFFu);
            m = max(m, (w[i] >> 16) & 0x7FFFu);
        }
    };
#pragma unroll
    for (int c = 0; c < kPrepCache; ++c) {
        const int64_t k = ((int64_t)c * kPrepThreads + tid) * 8;
        cache[c] = k < K ? ldg_v4(xr + k) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < kPrepCache; ++c)
        vmax(cache[c]);
    for (int64_t k = ((int64_t)kPrepCache * kPrepThreads + tid) * 8; k < K; k += kPrepThreads * 8)
        vmax(ldg_v4(xr + k));
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((tid & 31) == 0)
        red[tid >> 5] = m;
    if (tid == 0)
        bad = 0;
    __syncthreads();
    m = 0;
    for (int i = 0; i < kPrepThreads / 32; ++i)
        m = max(m, red[i]);
    // Non-finite, subnormal-only or extreme rows go to the bf16 mode.
    int flag = 0, s = 0;
    if (m >= 0x7F80u || (m != 0 && (m >> 7) == 0)) {
        flag = 1;
    } else if (m != 0) {
        s = 15 - ((int)(m >> 7) - 127);
        if (s > 120 || s < -120)
            flag = 1;
    }
    int local_bad = 0;
    if (!flag) {
        const float scale = __int_as_float((s + 127) << 23);
        auto convert = [&](const uint4 &v, int64_t k) {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __uint_as_float(w[i] << 16) * scale;
                const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * scale;
                const __half hl = __float2half_rn(lo), hh = __float2half_rn(hi);
                local_bad |= (__half2float(hl) != lo) | (__half2float(hh) != hi);
                out[i] = (uint32_t)__half_as_ushort(hl) | ((uint32_t)__half_as_ushort(hh) << 16);
            }
            *reinterpret_cast<uint4 *>(ximg + ximg_offset(n, k)) = make_uint4(out[0], out[1], out[2], out[3]);
        };
#pragma unroll
        for (int c = 0; c < kPrepCache; ++c) {
            const int64_t k = ((int64_t)c * kPrepThreads + tid) * 8;
            if (k < K)
                convert(cache[c], k);
        }
        for (int64_t k = ((int64_t)kPrepCache * kPrepThreads + tid) * 8; k < K; k += kPrepThreads * 8)
            convert(ldg_v4(xr + k), k);
    }
    if (local_bad)
        atomicOr(&bad, 1);
    __syncthreads();
    flag |= bad;
    if (tid == 0) {
        factor[n] = flag ? 1.0f : __int_as_float((127 - s) << 23);
        flags[n] = flag;
    }
}

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------

// Epilogue of one tile segment for thread row r: whole tiles are written
// directly; split tiles publish this row's partial and the last CTA to arrive
// for the row (per-row counter) adds all partials of the row in CTA order.
// fac[mi][n] (shared memory): tensor scale times the activation factor.
template <int NW>
__device__ __noinline__ void epilogue(const Args &a, const float *fac, const float (&v)[NW][16], int tile, int j,
                                      int u, int first_tile, int b, int r)
{
    constexpr int kMaxSplit = 8;  // partials loaded together by the last arriver
    const uint32_t total = (uint32_t)a.total, P = (uint32_t)a.P, C = (uint32_t)a.C;
    const int64_t m = (int64_t)tile * BM + r;
    const bool whole = (j == a.C - 1) && (u - j >= (int)cta_lo(b, total, P));
    float acc[NW][NTOK];
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
#pragma unroll
        for (int n = 0; n < NTOK; ++n)
            acc[mi][n] = v[mi][n];
    if (!whole) {
        const int slot = (tile == first_tile) ? 0 : 1;
        float *mine = a.partial + ((size_t)b * 2 + slot) * NW * NTOK * BM + r;
#pragma unroll
        for (int mi = 0; mi < NW; ++mi)
#pragma unroll
            for (int n = 0; n < NTOK; ++n)
                if (n < a.N)
                    mine[(mi * NTOK + n) * BM] = acc[mi][n];
        const int b_lo = cta_of((uint32_t)tile * C, total, P);
        const int b_hi = cta_of(((uint32_t)tile + 1) * C - 1, total, P);
        // acq_rel: publishes this thread's partial (release) and, for the last
        // arriver, makes the other CTAs' partials of this row visible (acquire).
        const uint32_t old = atom_add_acq_rel(&a.counters[(size_t)tile * BM + r], 1u);
        if (old != (uint32_t)(b_hi - b_lo))
            return;  // another CTA finishes this row
        // Sum the partials of CTAs b_lo..b_hi in CTA order, kMaxSplit CTAs per
        // round, all loads of a round in flight together.
#pragma unroll
        for (int mi = 0; mi < NW; ++mi)
#pragma unroll
            for (int n = 0; n < NTOK; ++n)
                acc[mi][n] = 0.0f;
        for (int b0 = b_lo; b0 <= b_hi; b0 += kMaxSplit) {
            const float *src[kMaxSplit];
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q) {
                const int bb = b0 + q <= b_hi ? b0 + q : b_hi;
                const int sl = ((int)(cta_lo((uint32_t)bb, total, P) / C) == tile) ? 0 : 1;
                src[q] = a.partial + ((size_t)bb * 2 + sl) * NW * NTOK * BM + r;
            }
#pragma unroll
            for (int mi = 0; mi < NW; ++mi)
#pragma unroll
                for (int n = 0; n < NTOK; ++n) {
                    if (n < a.N) {
                        float pv[kMaxSplit];
#pragma unroll
                        for (int q = 0; q < kMaxSplit; ++q)
                            pv[q] = __ldcg(src[q] + (mi * NTOK + n) * BM);
#pragma unroll
                        for (int q = 0; q < kMaxSplit; ++q)
                            if (b0 + q <= b_hi)
                                acc[mi][n] += pv[q];
                    }
                }
        }
    }
    if (m >= a.M)
        return;
#pragma unroll
    for (int n = 0; n < NTOK; ++n) {
        if (n < a.N) {
            float val;
            if (NW == 1)
                val = acc[0][n] * fac[n];
            else
                val = silu_mul(acc[0][n] * fac[n], acc[NW - 1][n] * fac[NTOK + n]);
            const int64_t idx = (int64_t)n * a.M + m;
            if (a.out_bf16)
                reinterpret_cast<uint16_t *>(a.y)[idx] = f32_to_bf16(val);
            else
                reinterpret_cast<float *>(a.y)[idx] = val;
        }
    }
}

struct IssuerArgs {
    const uint8_t *x_ring;
    uint64_t *x_full, *x_empty, *a_full, *a_empty, *d_full, *d_empty;
    uint32_t tmem_a, tmem_d;
    int n_units, j_lo;
};

// One MMA issuer (warp q, lane 0): matrix q / kChains, accumulator chain
// q % kChains, K steps kk = chain (mod kChains) of every sub-stage - four MMAs
// per sub-stage in both configurations.  The descriptor and TMEM offsets of
// those MMAs are computed once, so each MMA costs a few issue slots (the
// issuing thread shares its sub-partition with ALU-bound dequantisers).  One
// copy of the loop serves all issuers: per-issuer specialisations multiply the
// kernel's code size and starve the dequantisers' instruction fetch.
template <int NW>
NVFP4_DEVINL void mma_issuer(const Args &a, const IssuerArgs &p, int q)
{
    using C = Cfg<NW>;
    constexpr int kPerSub = C::kSubK / 16 / C::kChains;
    static_assert(kPerSub == 4, "four MMAs per issuer and sub-stage");
    const int mi = q / C::kChains;
    const int chain = q % C::kChains;
    uint32_t boff[C::kSubs][kPerSub], aoff[kPerSub];
#pragma unroll
    for (int t = 0; t < kPerSub; ++t) {
        const int kk = chain + C::kChains * t;
        aoff[t] = (uint32_t)(mi * 64 + kk * 8);
#pragma unroll
        for (int sub = 0; sub < C::kSubs; ++sub) {
            const int kl = sub * C::kSubK + kk * 16;  // k within the unit
            // B: 64-k sub-box kl / 64 of the activation unit (16 rows x 128 B,
            // 128-byte swizzle), 32-byte step kl % 64 inside it; descriptor
            // addresses are in 16-byte units.
            boff[sub][t] = (uint32_t)((kl >> 6) * (NTOK * 128 / 16) + 2 * ((kl >> 4) & 3));
        }
    }
    const uint32_t idesc = tc::idesc_f16kind(BM, NTOK, (uint32_t)load_mode(a));
    int j = p.j_lo;
    int seg = -1;
    int sx = 0, sa = 0;
    uint32_t phx = 0, pha = 0;
    for (int i = 0; i < p.n_units; ++i) {
        const bool first = (i == 0) || j == 0;
        const bool last = (i == p.n_units - 1) || j == a.C - 1;
        if (first) {
            ++seg;
            if (!tc::mbar_wait(&p.d_empty[seg & 1], (((uint32_t)seg >> 1) & 1) ^ 1)) {
                fail(a, 13);
                return;
            }
        }
        if (!tc::mbar_wait(&p.x_full[sx], phx)) {
            fail(a, 14);
            return;
        }
        const uint64_t bdesc0 = tc::smem_desc_sw128(p.x_ring + (size_t)sx * kXUnit);
        const uint32_t dcol = p.tmem_d + (uint32_t)(seg & 1) * C::kDCols + (uint32_t)(chain * NW + mi) * 16;
#pragma unroll
        for (int sub = 0; sub < C::kSubs; ++sub) {
            if (!tc::mbar_wait(&p.a_full[sa], pha)) {
                fail(a, 15);
                return;
            }
            tc::fence_after_sync();
            const uint32_t acol = p.tmem_a + (uint32_t)(sa * C::kACols);
#pragma unroll
            for (int t = 0; t < kPerSub; ++t)
                tc::mma_f16_ts(dcol, acol + aoff[t], bdesc0 + boff[sub][t], idesc,
                               (first && sub == 0 && t == 0) ? 0u : 1u);
            tc::mma_commit(&p.a_empty[sa]);
            if (++sa == C::kAStages) {
                sa = 0;
                pha ^= 1;
            }
        }
        tc::mma_commit(&p.x_empty[sx]);
        if (++sx == C::kXStages) {
            sx = 0;
            phx ^= 1;
        }
        if (last)
            tc::mma_commit(&p.d_full[seg & 1]);
        if (++j == a.C)
            j = 0;
    }
}

template <int NW>
__global__ void __launch_bounds__(kThreads, 1)
skinny_tc_kernel(const __grid_constant__ CUtensorMap m_codes0, const __grid_constant__ CUtensorMap m_codes1,
                 const __grid_constant__ CUtensorMap m_scales0, const __grid_constant__ CUtensorMap m_scales1,
                 const __grid_constant__ CUtensorMap m_x, Args a)
{
    using C = Cfg<NW>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *c_ring = smem;                                                   // [kCStages][NW][16 KB]
    uint8_t *s_ring = c_ring + (size_t)C::kCStages * NW * kCodeBox;           // [kSStages][NW][16 KB]
    uint8_t *x_ring = s_ring + (size_t)C::kSStages * NW * kScaleBox;          // [kXStages][8 KB]
    uint64_t *bars = reinterpret_cast<uint64_t *>(x_ring + (size_t)C::kXStages * kXUnit);
    uint64_t *c_full = bars;
    uint64_t *c_empty = c_full + C::kCStages;
    uint64_t *s_full = c_empty + C::kCStages;
    uint64_t *s_empty = s_full + C::kSStages;
    uint64_t *x_full = s_empty + C::kSStages;
    uint64_t *x_empty = x_full + C::kXStages;
    uint64_t *a_full = x_empty + C::kXStages;
    uint64_t *a_empty = a_full + C::kAStages;
    uint64_t *d_full = a_empty + C::kAStages;
    uint64_t *d_empty = d_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(d_empty + 2);
    float *fac_s = reinterpret_cast<float *>(tmem_slot + 4);  // [NW][16] epilogue factors

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const int64_t lo = (int64_t)b * a.total / a.P;
    const int64_t hi = (int64_t)(b + 1) * a.total / a.P;

    if (threadIdx.x == 0) {
        // Let the next kernel in the stream be scheduled as soon as SMs free up;
        // it waits for this grid's completion before it reads anything we write.
        tc::griddep_launch_dependents();
        // Consumers arrive once per warp (lane 0 after __syncwarp): hundreds
        // of per-thread arrivals on one mbarrier serialise in shared memory.
        for (int s = 0; s < C::kCStages; ++s) {
            tc::mbar_init(&c_full[s], 1);
            tc::mbar_init(&c_empty[s], kDqWarps);
        }
        for (int s = 0; s < C::kSStages; ++s) {
            tc::mbar_init(&s_full[s], 1);
            tc::mbar_init(&s_empty[s], kDqWarps);
        }
        for (int s = 0; s < C::kXStages; ++s) {
            tc::mbar_init(&x_full[s], 1);
            tc::mbar_init(&x_empty[s], kMmaWarps);
        }
        for (int s = 0; s < C::kAStages; ++s) {
            tc::mbar_init(&a_full[s], C::kAFullCount);
            tc::mbar_init(&a_empty[s], kMmaWarps);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&d_full[s], kMmaWarps);
            tc::mbar_init(&d_empty[s], kEpiThreads / 32);
        }
        tc::fence_mbar_init();
        tc::prefetch_tensormap(&m_codes0);
        tc::prefetch_tensormap(&m_scales0);
        if (NW == 2) {
            tc::prefetch_tensormap(&m_codes1);
            tc::prefetch_tensormap(&m_scales1);
        }
    }
    if (warp == 0)
        tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_a = tmem;
    const uint32_t tmem_d = tmem + C::kAStages * C::kACols;

    // Every role walks the CTA's units lo..hi-1 with incremental (tile, j)
    // and ring (stage, phase) counters: no 64-bit division in the loops.
    const int n_units = (int)(hi - lo);
    const int64_t tile_lo = lo / a.C;
    const int j_lo = (int)(lo - tile_lo * a.C);

    if (warp == 4 || warp == 5) {
        // ---- code producers: even units (warp 4) and odd units (warp 5) ----
        if (lane == 0) {
            const int par = warp - 4;
            int64_t tile = tile_lo;
            int j = j_lo + par;
            if (j >= a.C) {
                j -= a.C;
                ++tile;
            }
            for (int i = par; i < n_units; i += 2) {
                const int s = i % C::kCStages;
                const uint32_t ph = (uint32_t)(i / C::kCStages) & 1;
                if (!tc::mbar_wait(&c_empty[s], ph ^ 1)) {
                    fail(a, 11);
                    break;
                }
                uint8_t *st = c_ring + (size_t)s * NW * kCodeBox;
                tc::mbar_arrive_expect_tx(&c_full[s], NW * kCodeBox);
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    tc::tma_load_2d(st + mi * kCodeBox, mi == 0 ? &m_codes0 : &m_codes1, &c_full[s], j * (BKU / 2),
                                    (int)(tile * BM));
                j += 2;
                while (j >= a.C) {
                    j -= a.C;
                    ++tile;
                }
            }
        }
    } else if (warp == 6) {
        // ---- scale producer: one 2048-k box per matrix per scale stage ----
        if (lane == 0) {
            int64_t tile = tile_lo;
            int j = j_lo;
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < n_units; ++i) {
                if (i == 0 || j % kScaleUnits == 0) {
                    if (!tc::mbar_wait(&s_empty[s], ph ^ 1)) {
                        fail(a, 19);
                        break;
                    }
                    uint8_t *st = s_ring + (size_t)s * NW * kScaleBox;
                    tc::mbar_arrive_expect_tx(&s_full[s], NW * kScaleBox);
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi)
                        tc::tma_load_2d(st + mi * kScaleBox, mi == 0 ? &m_scales0 : &m_scales1, &s_full[s],
                                        (j / kScaleUnits) * (kScaleUnits * BKU / 16), (int)(tile * BM));
                    if (++s == C::kSStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (++j == a.C) {
                    j = 0;
                    ++tile;
                }
            }
        }
    } else if (warp == 7) {
        // ---- activation producer: per unit and 64-k sub-box, the N token rows
        // only - from the f16 image (one bulk copy; the rows are contiguous
        // there), or in bf16 mode straight from x through its tensor map (the
        // 128-byte swizzle lands the rows in MMA layout).  Rows >= N of the
        // MMA's B operand only feed accumulator columns the epilogue ignores,
        // so they are zeroed once and never loaded: for small N the
        // activations take almost no copy bandwidth from the weight stream.
        for (int o = lane * 16; o < C::kXStages * kXUnit; o += 32 * 16)
            *reinterpret_cast<uint4 *>(x_ring + o) = make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tc::prefetch_tensormap(&m_x);
            tc::griddep_wait();
            const bool bf16_mode = load_mode(a) != 0;
            const uint32_t row_bytes = (uint32_t)a.N * 128;
            int j = j_lo, s = 0;
            uint32_t ph = 0;
            for (int i = 0; i < n_units; ++i) {
                if (!tc::mbar_wait(&x_empty[s], ph ^ 1)) {
                    fail(a, 12);
                    break;
                }
                uint8_t *dst = x_ring + (size_t)s * kXUnit;
                tc::mbar_arrive_expect_tx(&x_full[s], 4 * row_bytes);
                if (bf16_mode) {
#pragma unroll
                    for (int sb = 0; sb < 4; ++sb)
                        tc::tma_load_2d(dst + sb * (NTOK * 128), &m_x, &x_full[s], j * BKU + sb * 64, 0);
                } else {
                    const uint8_t *src = a.x_img + (size_t)j * kXUnit;
#pragma unroll
                    for (int sb = 0; sb < 4; ++sb)
                        bulk_load(dst + sb * (NTOK * 128), src + sb * (NTOK * 128), row_bytes, &x_full[s]);
                }
                if (++s == C::kXStages) {
                    s = 0;
                    ph ^= 1;
                }
                if (++j == a.C)
                    j = 0;
            }
        }
    } else if (warp < kMmaWarps) {
        // ---- MMA issuers: issuer q owns matrix q / kChains, chain q % kChains ----
        if (lane == 0) {
            tc::griddep_wait();
            IssuerArgs ia{x_ring, x_full, x_empty, a_full, a_empty, d_full, d_empty, tmem_a, tmem_d, n_units, j_lo};
            mma_issuer<NW>(a, ia, warp);
        }
    } else {
        // ---- dequantisers (warps 8..23) and epilogue (warps 8..11) ----
        tc::griddep_wait();
        const int mode = load_mode(a);
        const int dq = threadIdx.x - kFirstDqWarp * 32;  // 0..511
        if (dq < NW * NTOK) {
            const int mi = dq / NTOK, n = dq % NTOK;
            const float t = __ldg(a.ts[mi]);
            fac_s[dq] = mode ? t * 256.0f : t * a.factor[n];
        }
        tc::named_bar_sync(1, kDqThreads);  // fac_s visible to the epilogue threads
        const int grp = dq >> 7;                          // 0..3
        const int quarter = warp & 3;                     // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;                // row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        // This group's share of a unit: 16-byte code chunks chunk0.. (32 k each)
        // of sub-stage my_sub of matrix my_mi, and the scale bytes of those
        // chunks (2 per chunk) at byte sc_off of the unit's 16 scale bytes.
        const int my_sub = (NW == 1) ? 0 : (grp & 1);
        const int my_mi = (NW == 1) ? 0 : (grp >> 1);
        const int chunk0 = (NW == 1) ? grp * 2 : (grp & 1) * 4;
        constexpr int kChunks = NW == 1 ? 2 : 4;
        const int sc_off = chunk0 * 2;
        const uint32_t col0 = (NW == 1) ? (uint32_t)grp * 32 : (uint32_t)my_mi * 64;
        const int swz = r & 7;
        int64_t tile = tile_lo;
        int j = j_lo;
        int seg = -1;
        int sc = 0, ss = 0, sa = 0;
        uint32_t phc = 0, phs = 0, pha = 0;
        // A sub-stage of unit i for this group: the ring advances by kSubs per
        // unit; this group's slot is my_sub sub-stages further.
        for (int t = 0; t < my_sub; ++t)
            if (++sa == C::kAStages) {
                sa = 0;
                pha ^= 1;
            }
        bool ok = true;
        for (int i = 0; i < n_units && ok; ++i) {
            const bool first = (i == 0) || j == 0;
            const bool last = (i == n_units - 1) || j == a.C - 1;
            const bool scale_first = (i == 0) || (j % kScaleUnits == 0);
            const bool scale_last = last || ((j + 1) % kScaleUnits == 0);
            if (first)
                ++seg;
            if (scale_first && i > 0 && ++ss == C::kSStages) {  // unit 0 uses scale stage 0
                ss = 0;
                phs ^= 1;
            }
            // the scale box of this unit was waited for at its first unit
            if (!tc::mbar_wait(&c_full[sc], phc) || (scale_first && !tc::mbar_wait(&s_full[ss], phs))) {
                fail(a, 16);
                ok = false;
                break;
            }
            // copy this thread's codes and scales to registers, release the slots
            const uint8_t *crow = c_ring + ((size_t)sc * NW + my_mi) * kCodeBox + r * 128;
            uint4 cw[kChunks];
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
                cw[c] = *reinterpret_cast<const uint4 *>(crow + (((chunk0 + c) ^ swz) << 4));
            // 64-byte rows, 64-byte swizzle: 16-byte chunk c of row r sits at c ^ ((r >> 1) & 3).
            const uint8_t *sp = s_ring + ((size_t)ss * NW + my_mi) * kScaleBox + r * 64 +
                                (((j % kScaleUnits) ^ ((r >> 1) & 3)) << 4) + sc_off;
            uint32_t scw[kChunks / 2];
            if (NW == 1) {
                scw[0] = *reinterpret_cast<const uint32_t *>(sp);
            } else {
                const uint2 v2 = *reinterpret_cast<const uint2 *>(sp);
                scw[0] = v2.x;
                scw[kChunks / 2 - 1] = v2.y;
            }
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&c_empty[sc]);
                if (scale_last)
                    tc::mbar_arrive(&s_empty[ss]);
            }
            if (++sc == C::kCStages) {
                sc = 0;
                phc ^= 1;
            }

            // dequantise and store into this group's columns of A sub-stage (unit i, my_sub)
            if (!tc::mbar_wait(&a_empty[sa], pha ^ 1)) {
                fail(a, 17);
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const uint32_t acol = tmem_a + sa * C::kACols + col0 + lane_off;
#pragma unroll
            for (int h = 0; h < kChunks / 2; ++h) {  // 64 k -> 32 TMEM columns per store
                uint32_t out[32];
                dequant_chunk(cw[2 * h], scw[h] & 0xFFFF, mode, out);
                dequant_chunk(cw[2 * h + 1], scw[h] >> 16, mode, out + 16);
                tc::tmem_st_32x32b_x32(acol + h * 32, out);
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(&a_full[sa]);
            for (int t = 0; t < C::kSubs; ++t)
                if (++sa == C::kAStages) {
                    sa = 0;
                    pha ^= 1;
                }

            if (last && grp == 0) {
                // ---- epilogue for this tile segment (first dequantiser group) ----
                const int db = seg & 1;
                if (!tc::mbar_wait(&d_full[db], ((uint32_t)seg >> 1) & 1)) {
                    fail(a, 18);
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                float sum[NW][16];
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        sum[mi][n] = 0.0f;
#pragma unroll
                for (int ch = 0; ch < C::kChains; ++ch) {
                    uint32_t v[NW][16];
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi)
                        tc::tmem_ld_32x32b_x16(tmem_d + db * C::kDCols + (ch * NW + mi) * 16 + lane_off, v[mi]);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi)
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            sum[mi][n] += __uint_as_float(v[mi][n]);  // chains added in a fixed order
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(&d_empty[db]);
                epilogue<NW>(a, fac_s, sum, (int)tile, j, (int)(lo + i), (int)tile_lo, b, r);
            }
            if (++j == a.C) {
                j = 0;
                ++tile;
            }
        }
    }

    // Lane 0 of the producer and MMA warps ran their loops alone: reconverge
    // each warp first, so the block-wide barrier below really waits for every
    // thread (a partially arrived warp would otherwise count as arrived).
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    auto enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NW>
cudaError_t launch_main(const CUtensorMap (&maps)[5], const Args &a, cudaStream_t stream)
{
    using C = Cfg<NW>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(skinny_tc_kernel<NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)C::kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, skinny_tc_kernel<NW>, maps[0], maps[1], maps[2], maps[3], maps[4], a);
}

}  // namespace sk

// Units (128 rows x 256 k) times CTAs must stay below 2^31: the kernel's
// stream-K arithmetic is 32-bit.
bool skinny_tc_supported(int64_t M, int64_t K)
{
    if (K < 256 || K % 256 != 0 || M < 1)
        return false;
    const int64_t units = ((M + 127) / 128) * (K / 256);
    return units * kSkinnyTcMaxCtas < (INT64_C(1) << 31);
}

size_t skinny_tc_workspace_bytes(int64_t M, int64_t K, int n_weights)
{
    return sk::ws_layout(M, K, n_weights).total;
}

cudaError_t launch_skinny_tc(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                             const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                             int out_bf16, void *workspace, int num_sms, cudaStream_t stream)
{
    using namespace sk;
    const WsLayout L = ws_layout(M, K, n_weights);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    float *factor = reinterpret_cast<float *>(ws);
    int *flags = reinterpret_cast<int *>(ws + 64);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + 128);

    Args a{};
    a.N = N;
    a.M = M;
    a.K = K;
    a.C = (int)((K + BKU - 1) / BKU);
    a.T = (M + BM - 1) / BM;
    a.total = a.T * a.C;
    a.P = (int)std::max<int64_t>(1, std::min<int64_t>(a.total, std::min<int64_t>(num_sms, kSkinnyTcMaxCtas)));
    for (int i = 0; i < 2; ++i)
        a.ts[i] = ts[i < n_weights ? i : 0];
    a.factor = factor;
    a.flags = flags;
    a.counters = reinterpret_cast<uint32_t *>(ws + L.counters);
    a.partial = reinterpret_cast<float *>(ws + L.partial);
    a.x_img = ws + L.ximg;
    a.err = err;
    a.y = y;
    a.out_bf16 = out_bf16;

    CUtensorMap maps[5];
    for (int i = 0; i < 2; ++i) {
        const int s = i < n_weights ? i : 0;
        // boxes: one unit of codes (BKU/2 bytes per row, 128-byte swizzle) and
        // of scales (BKU/16 bytes per row), 128 rows each
        static_assert(kCodeBox == BM * (BKU / 2) && kScaleBox == BM * (BKU * kScaleUnits / 16), "box sizes");
        static_assert(BKU * kScaleUnits / 16 == 64, "scale box rows are 64 bytes (64-byte swizzle)");
        if (!make_map(&maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, codes[s], (uint64_t)K / 2, (uint64_t)M,
                      (uint64_t)K / 2, BKU / 2, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&maps[2 + i], CU_TENSOR_MAP_DATA_TYPE_UINT8, scales[s], (uint64_t)K / 16, (uint64_t)M,
                      (uint64_t)K / 16, BKU * kScaleUnits / 16, BM, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    // x itself ([N][K] bf16), read by the main kernel in bf16 mode: boxes of
    // 64 k x N rows with the 128-byte swizzle of the MMA operand layout.
    if (!make_map(&maps[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64,
                  (uint32_t)N, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    // prep (programmatic dependent launch on the previous kernel in the stream)
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(N);
        cfg.blockDim = dim3(kPrepThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_prep_kernel, x, N, K, ws + L.ximg, factor, flags,
                                           a.counters, a.T, err);
        if (e != cudaSuccess)
            return e;
    }
    return n_weights == 1 ? launch_main<1>(maps, a, stream) : launch_main<2>(maps, a, stream);
}

}  // namespace nvfp4
