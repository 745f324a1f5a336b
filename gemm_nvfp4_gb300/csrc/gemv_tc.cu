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
//                the split-K tile counters.
//   main kernel  one CTA per SM, stream-K over units (tile of 128 rows,
//                256 k) so every SM streams the same bytes:
//     warps 4,5  TMA: the code box [128 rows][128 B] (128-byte swizzle) and
//                scale box [128 rows][16 B] of each unit (even / odd units)
//                into a 10-unit ring.  They do not depend on the prep kernel,
//                so weights stream while the previous kernel still runs.
//     warp 6     activation copies: the N token rows of each unit.
//     warps 12-27 dequantise in four independent groups: item t (half a unit,
//                or a quarter unit of both gate and up matrices) goes to group
//                t % 4; thread = weight row = TMEM lane; codes and scales from
//                shared memory -> f16x2 (or bf16x2) -> tcgen05.st into a
//                6-item TMEM ring.  Groups work on different items, so one
//                group's waits overlap another's arithmetic.
//     warps 0-3  one thread each issues tcgen05.mma kind::f16 (M=128, N=16,
//                K=16, A in TMEM) into its own fp32 accumulator chain in a
//                double-buffered TMEM accumulator.
//     warps 8-11 epilogue: chains added in a fixed order, whole tiles stored.
//   K is split across CTAs in one of two ways, chosen by the host from the
//   shapes: stream-K (each CTA a contiguous share of the tile-major unit
//   list; a tile split across CTAs is finished by the last CTA to arrive, one
//   counter per tile in the workspace, adding the partials in CTA order; the
//   CTA's last segment is added by the epilogue and dequantiser threads
//   together), or cluster-K for one matrix whose tiles fit one per cluster
//   (a cluster of 4 CTAs splits each tile's K; the leader adds the partials of
//   ranks 0..3 in order through distributed shared memory).  Both are
//   deterministic.
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
#include "skinny.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace sk {

constexpr int BM = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int BKU = 256;         // k per unit (one code box per matrix)
constexpr int NTOK = 16;         // MMA N (tokens, padded)
// Warp roles: 0..3 MMA issuers (one per SM sub-partition), 4 and 5 weight
// producers (even / odd units: codes and scales), 6 activation producer,
// 7 idle, 8..11 epilogue (one warp per TMEM lane quarter), 12..27
// dequantisers (four groups of four warps, one warp per lane quarter).
// Several producer threads are used because one thread issuing TMA copies
// back to back tops out well below HBM bandwidth on GB300, while two to four
// issuing threads reach it.  Several MMA issuers are used because a thread
// issuing tcgen05.mma competes for issue slots with the dequantiser warps of
// its sub-partition; N = 16 MMAs are short, so issue rate matters.
constexpr int kMmaWarps = 4;
constexpr int kEpiWarp0 = 8;
constexpr int kFirstDqWarp = 12;
constexpr int kDqWarps = 16;
constexpr int kGroups = 4;           // dequantiser groups
constexpr int kThreads = (kFirstDqWarp + kDqWarps) * 32;
constexpr int kEpiThreads = 128;
constexpr int kCodeBox = BM * 128;   // 16 KB: 128 rows x 128 code bytes (256 k), 128-byte swizzle
constexpr int kScaleBox = BM * 16;   // 2 KB: 128 rows x 16 scale bytes (256 k), no swizzle
constexpr int kXUnit = NTOK * BKU * 2;  // 8 KB: activation image of one unit
constexpr uint32_t kTmemCols = 512;

// FP6 E2M3 weights (FMT 1): a unit's 192 code bytes per row arrive as three
// [128 rows][64 B] boxes with the 64-byte swizzle; the scale bytes (one per
// 128 k) are read by the dequantisers from global memory ahead of use.
constexpr int kCodeBox6 = BM * 64;    // 8 KB

template <int NW, int FMT = 0>
struct Cfg {
    // The weight ring holds most of the shared memory: with ~4 us of loaded
    // DRAM latency, every SM needs well over 100 KB of weights in flight.
    // A stage holds one unit: NW code boxes, then NW scale boxes (NVFP4), or
    // NW x 3 FP6 code boxes.
    static constexpr int kStageBytes = FMT == 0 ? NW * (kCodeBox + kScaleBox) : NW * 3 * kCodeBox6;
    static constexpr int kCStages = FMT == 0 ? (NW == 1 ? 10 : 5) : (NW == 1 ? 7 : 3);  // weight ring (units)
    static constexpr int kXStages = NW == 1 ? 4 : 3;   // activation ring (units, from L2)
    // Work item of one dequantiser group = one TMEM A stage of 64 columns
    // (128 weights per row):
    //   NW = 1: half a unit (128 k); group g takes half g % 2 of the units
    //           i = g / 2 (mod 2) of the CTA's range;
    //   NW = 2: a quarter unit (64 k) of both matrices (matrix m in columns
    //           [32m, 32m+32)); group g takes quarter g of every unit.
    // Item t = i * kItems + h goes to group t % 4, so the groups run on
    // different items and one group's waits overlap another's arithmetic.
    static constexpr int kItems = NW == 1 ? 2 : 4;     // items per unit
    static constexpr int kUnitStep = kGroups / kItems;  // units between two items of a group
    static constexpr int kItemK = BKU / kItems;          // k per item (per matrix)
    static constexpr int kReaders = kItems * 4;          // warps that read one weight stage
    static constexpr int kAStages = 6;                   // TMEM A ring (items)
    static constexpr int kACols = 64;
    // Independent accumulation chains per matrix: issuer q accumulates matrix
    // q / kChains over the K steps kk = q % kChains (mod kChains) of each item
    // into its own chain; the epilogue adds the chains in a fixed order.
    static constexpr int kChains = kMmaWarps / NW;
    static constexpr int kPerItem = kItemK / 16 / kChains;  // MMAs per issuer and item
    static constexpr int kDCols = 16 * NW * kChains;   // one accumulator buffer
    static constexpr int kCkBytes = BM * NW * NTOK * 4;  // cluster-K partial staging
    static constexpr size_t kSmemBytes =
        (size_t)kCStages * kStageBytes + (size_t)kXStages * kXUnit + kCkBytes + 1024 + 1024;
    static_assert(kPerItem == 2, "two MMAs per issuer and item");
    static_assert(kAStages * kACols + 2 * kDCols <= (int)kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kStageBytes % 1024 == 0, "code boxes stay 1024-byte aligned (128-byte swizzle)");
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
    uint32_t *counters;    // [T] per-tile arrival counters
    float *partial;        // [P][2][NW][16][128]
    const uint8_t *x_img;  // [C][8 KB] f16 activation image (shared-memory layout)
    uint32_t *err;
    void *y;
    int out_bf16;
    int bf16_only;  // 1: no prep kernel; bf16 operands read from x itself
    int cs;         // > 1: cluster-K (clusters of cs CTAs split every tile's K); 1: stream-K
    int ncl;        // cluster-K: number of clusters
    const uint8_t *scales6[2];  // FP6: UE8M0 scales [M][K/128] (read by the dequantisers)
};

// Workspace layout (bytes): header 256 (factor[16], flags[16], err), per-tile
// split-K counters in a fixed region of kCounterRegion bytes, the f16
// activation image, split-K partials.  The counters must be zero when a call
// without the prep kernel starts; every call leaves them zero (the last CTA to
// arrive on a tile resets its counter), and the fixed region keeps any call's
// image or partials from landing on a later call's counters (the mma.sync
// path, whose partials do start at byte 256, zeroes every partial it reads).
constexpr size_t kCounterRegion = size_t(1) << 20;

struct WsLayout {
    size_t counters, ximg, partial, total;
};

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(int64_t M, int64_t K, int nw)
{
    WsLayout w;
    const int64_t T = (M + BM - 1) / BM;
    const int64_t C = (K + BKU - 1) / BKU;
    (void)T;
    w.counters = 256;
    w.ximg = w.counters + kCounterRegion;
    w.partial = w.ximg + (size_t)C * kXUnit;
    w.total = w.partial + (size_t)kSkinnyTcMaxCtas * 2 * nw * NTOK * BM * 4;
    return w;
}

// Stream-K partition in 32-bit arithmetic (the host keeps total * P < 2^31):
// CTA b owns units [b * total / P, (b + 1) * total / P).
NVFP4_DEVINL int cta_of(uint32_t q, uint32_t total, uint32_t P) { return (int)(((q + 1) * P - 1) / total); }
NVFP4_DEVINL uint32_t cta_lo(uint32_t b, uint32_t total, uint32_t P) { return b * total / P; }

// The units of one CTA: tiles tile0, tile0 + tstep, ...; unit j of a tile
// runs over [jb, je), except that the first tile starts at j_first.
struct Range {
    int64_t tile0, tstep;
    int j_first, jb, je, n_units;
};

// Stream-K: CTA b owns units [b * total / P, (b + 1) * total / P) of the
// tile-major unit list.
NVFP4_DEVINL Range cta_range(const Args &a, int b)
{
    if (a.cs > 1) {
        // Cluster-K: cluster q takes tiles q, q + ncl, ...; its CTA of rank r
        // takes units [r * C / cs, (r + 1) * C / cs) of each of them.
        const int q = b / a.cs, r = b % a.cs;
        Range g;
        g.tile0 = q;
        g.tstep = a.ncl;
        g.jb = r * a.C / a.cs;
        g.je = (r + 1) * a.C / a.cs;
        g.j_first = g.jb;
        const int64_t k = q < a.T ? (a.T - q + a.ncl - 1) / a.ncl : 0;
        g.n_units = (int)(k * (g.je - g.jb));
        return g;
    }
    const int64_t lo = (int64_t)b * a.total / a.P, hi = (int64_t)(b + 1) * a.total / a.P;
    Range g;
    g.tile0 = lo / a.C;
    g.tstep = 1;
    g.j_first = (int)(lo - g.tile0 * a.C);
    g.jb = 0;
    g.je = a.C;
    g.n_units = (int)(hi - lo);
    return g;
}


NVFP4_DEVINL void fail(const Args &a, uint32_t code) { atomicExch(a.err, code); }

NVFP4_DEVINL int load_mode(const Args &a)
{
    if (a.bf16_only)
        return 1;
    int f = 0;
    for (int n = 0; n < a.N; ++n)
        f |= a.flags[n];
    return f ? 1 : 0;
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
                                                                   int *flags, uint32_t *counters, int64_t T)
{
    tc::griddep_launch_dependents();
    tc::griddep_wait();  // x may come from the previous kernel; the workspace may be in use by it
    const int n = blockIdx.x;
    const int tid = threadIdx.x;
    for (int64_t i = (int64_t)n * kPrepThreads + tid; i < T; i += (int64_t)N * kPrepThreads)
        counters[i] = 0;
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

// Output value of row m, token n from the fp32 sums of the matrices.
template <int NW>
NVFP4_DEVINL void store_out(const Args &a, const float *fac, int n, int64_t m, float s0, float s1)
{
    const float val = NW == 1 ? s0 * fac[n] : silu_mul(s0 * fac[n], s1 * fac[NTOK + n]);
    const int64_t idx = (int64_t)n * a.M + m;
    if (a.out_bf16)
        reinterpret_cast<uint16_t *>(a.y)[idx] = f32_to_bf16(val);
    else
        reinterpret_cast<float *>(a.y)[idx] = val;
}

// Split-K bookkeeping of one tile segment, shared by the epilogue threads
// and (for the CTA's last segment) the dequantiser threads.
struct SegInfo {
    int tile, b_lo, b_hi, reduce;
};

// Epilogue of one tile segment, run by the 128 epilogue threads (thread r
// holds row r's sums v[mi][n]).  A tile done by this CTA alone is written
// directly.  Otherwise the CTA publishes its partial ([mi][n][row] floats) and
// counts its arrival on the tile's counter with one release-acquire atomic
// after a barrier of the epilogue threads (the barrier orders every thread's
// partial stores before the release).  Returns in `si` whether this CTA
// arrived last and must add the tile's partials (reduce_tile).
template <int NW>
__device__ __noinline__ void publish_segment(const Args &a, const float *fac, const float (&v)[NW][16], int tile,
                                             bool whole, int first_tile, int b, int r, SegInfo *si)
{
    const uint32_t total = (uint32_t)a.total, P = (uint32_t)a.P, C = (uint32_t)a.C;
    const int64_t m = (int64_t)tile * BM + r;
    if (whole) {  // uniform across the epilogue threads
        if (m < a.M)
#pragma unroll
            for (int n = 0; n < NTOK; ++n)
                if (n < a.N)
                    store_out<NW>(a, fac, n, m, v[0][n], v[NW - 1][n]);
        if (r == 0)
            si->reduce = 0;
        return;
    }
    const int slot = (tile == first_tile) ? 0 : 1;
    float *mine = a.partial + ((size_t)b * 2 + slot) * NW * NTOK * BM + r;
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
#pragma unroll
        for (int n = 0; n < NTOK; ++n)
            if (n < a.N)
                mine[(mi * NTOK + n) * BM] = v[mi][n];
    tc::named_bar_sync(1, kEpiThreads);
    if (r == 0) {
        const int b_lo = cta_of((uint32_t)tile * C, total, P);
        const int b_hi = cta_of(((uint32_t)tile + 1) * C - 1, total, P);
        // release: this CTA's partial (every thread's stores, ordered before
        // this atomic by the barrier); acquire: the other CTAs' partials.
        const uint32_t old = atom_add_acq_rel(&a.counters[tile], 1u);
        si->tile = tile;
        si->b_lo = b_lo;
        si->b_hi = b_hi;
        si->reduce = old == (uint32_t)(b_hi - b_lo);
        if (si->reduce)
            a.counters[tile] = 0;  // all of the tile's CTAs have arrived: zero for the next call
    }
    tc::named_bar_sync(1, kEpiThreads);
}

// Last arriver of a split tile: add the partials of CTAs b_lo..b_hi in CTA
// order (deterministic) and write the outputs.  Threads t = 0..nthr-1 share
// the work: pair p = (token n, rows 4q..4q+3) for p = t, t + nthr, ...; each
// pair's partials are read with 16-byte loads, kBatch CTAs in flight.
template <int NW>
__device__ __noinline__ void reduce_tile(const Args &a, const float *fac, const SegInfo si, int t, int nthr)
{
    constexpr int kBatch = 4;
    const uint32_t total = (uint32_t)a.total, P = (uint32_t)a.P, C = (uint32_t)a.C;
    const int np = a.N * (BM / 4);
    for (int p = t; p < np; p += nthr) {
        const int n = p / (BM / 4), r4 = (p % (BM / 4)) * 4;
        float4 acc[NW];
#pragma unroll
        for (int mi = 0; mi < NW; ++mi)
            acc[mi] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b0 = si.b_lo; b0 <= si.b_hi; b0 += kBatch) {
            float4 pv[kBatch][NW];
            float4 *src[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int bb = b0 + q <= si.b_hi ? b0 + q : si.b_hi;
                const int sl = ((int)(cta_lo((uint32_t)bb, total, P) / C) == si.tile) ? 0 : 1;
                src[q] = reinterpret_cast<float4 *>(a.partial + ((size_t)bb * 2 + sl) * NW * NTOK * BM + r4 + n * BM);
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    pv[q][mi] = __ldcg(src[q] + mi * (NTOK * BM / 4));
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
                if (b0 + q <= si.b_hi)
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi) {
                        acc[mi].x += pv[q][mi].x;
                        acc[mi].y += pv[q][mi].y;
                        acc[mi].z += pv[q][mi].z;
                        acc[mi].w += pv[q][mi].w;
                    }
        }
        const int64_t m0 = (int64_t)si.tile * BM + r4;
        const float g[4] = {acc[0].x, acc[0].y, acc[0].z, acc[0].w};
        const float h[4] = {acc[NW - 1].x, acc[NW - 1].y, acc[NW - 1].z, acc[NW - 1].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (m0 + e < a.M)
                store_out<NW>(a, fac, n, m0 + e, g[e], h[e]);
    }
}

// Cluster-K epilogue of one tile segment (epilogue threads; thread r holds row
// r's accumulator sums v[mi][n]).  Every CTA of the cluster stages its partial
// in its own shared memory ([row][matrix * 16 + token] floats) and arrives on
// the leader's barrier (release at cluster scope); the leader (rank 0) adds
// the partials of ranks 0, 1, ... in that order through distributed shared
// memory, writes the outputs and then frees every rank's buffer.  A rank
// waits for that before reusing the buffer (and before exiting).
template <int NW>
__device__ __noinline__ void ck_epilogue(const Args &a, const float *fac, const float (&v)[NW][16], int64_t tile,
                                         int r, int et, int seg, float *buf, uint64_t *ck_full, uint64_t *ck_free)
{
    constexpr int kRow = NW * NTOK;  // floats per row
    const uint32_t rank = tc::cluster_ctarank();
    if (seg > 0 && !tc::bar_and(1, kEpiThreads, tc::mbar_wait_cluster(ck_free, (uint32_t)(seg - 1) & 1))) {
        fail(a, 23);
        return;
    }
    float *row = buf + r * kRow;
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
#pragma unroll
        for (int n = 0; n < NTOK; n += 4)
            *reinterpret_cast<float4 *>(row + mi * NTOK + n) =
                make_float4(v[mi][n], v[mi][n + 1], v[mi][n + 2], v[mi][n + 3]);
    tc::fence_acq_rel_cluster();
    tc::named_bar_sync(1, kEpiThreads);
    if (et == 0)
        tc::mbar_arrive_remote(tc::mapa(ck_full, 0));
    if (rank != 0)
        return;
    if (!tc::bar_and(1, kEpiThreads, tc::mbar_wait_cluster(ck_full, (uint32_t)seg & 1))) {
        fail(a, 24);
        return;
    }
    float acc[NW][NTOK];
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
#pragma unroll
        for (int n = 0; n < NTOK; ++n)
            acc[mi][n] = 0.0f;
    for (int k = 0; k < a.cs; ++k) {  // ranks in order: deterministic
        const uint32_t src = tc::mapa(buf + r * kRow, (uint32_t)k);
#pragma unroll
        for (int mi = 0; mi < NW; ++mi)
#pragma unroll
            for (int n = 0; n < NTOK; n += 4) {
                const float4 p = tc::ld_shared_cluster_v4(src + (uint32_t)((mi * NTOK + n) * 4));
                acc[mi][n] += p.x;
                acc[mi][n + 1] += p.y;
                acc[mi][n + 2] += p.z;
                acc[mi][n + 3] += p.w;
            }
    }
    const int64_t m = tile * BM + r;
    if (m < a.M)
#pragma unroll
        for (int n = 0; n < NTOK; ++n)
            if (n < a.N) {
                const float val = NW == 1 ? acc[0][n] * fac[n]
                                          : silu_mul(acc[0][n] * fac[n], acc[NW - 1][n] * fac[NTOK + n]);
                const int64_t idx = (int64_t)n * a.M + m;
                if (a.out_bf16)
                    reinterpret_cast<uint16_t *>(a.y)[idx] = f32_to_bf16(val);
                else
                    reinterpret_cast<float *>(a.y)[idx] = val;
            }
    tc::named_bar_sync(1, kEpiThreads);  // every read of the ranks' buffers is done
    if (et < a.cs)
        tc::mbar_arrive_remote(tc::mapa(ck_free, (uint32_t)et));
}

struct IssuerArgs {
    const uint8_t *x_ring;
    uint64_t *x_full, *x_empty, *a_full, *a_empty, *d_full, *d_empty;
    uint32_t tmem_a, tmem_d;
    int n_units, j_lo, jb, je;
};

// One MMA issuer (warp q, lane 0): matrix q / kChains, accumulator chain
// q % kChains, K steps kk = chain (mod kChains) of every item - two MMAs per
// item in both configurations.  The descriptor and TMEM offsets of those MMAs
// are computed once, so each MMA costs a few issue slots (the issuing thread
// shares its sub-partition with ALU-bound dequantisers).  One copy of the loop
// serves all issuers: per-issuer specialisations multiply the kernel's code
// size and starve the dequantisers' instruction fetch.
template <int NW>
NVFP4_DEVINL void mma_issuer(const Args &a, const IssuerArgs &p, int q)
{
    using C = Cfg<NW>;
    constexpr int kI = C::kItems, kT = C::kPerItem;
    const int mi = q / C::kChains;
    const int chain = q % C::kChains;
    uint32_t boff[kI][kT], aoff[kT];
#pragma unroll
    for (int t = 0; t < kT; ++t) {
        const int kk = chain + C::kChains * t;  // K step within the item
        aoff[t] = (uint32_t)(mi * 32 + kk * 8);
#pragma unroll
        for (int h = 0; h < kI; ++h) {
            const int kl = h * C::kItemK + kk * 16;  // k within the unit
            // B: 64-k sub-box kl / 64 of the activation unit (16 rows x 128 B,
            // 128-byte swizzle), 32-byte step kl % 64 inside it; descriptor
            // addresses are in 16-byte units.
            boff[h][t] = (uint32_t)((kl >> 6) * (NTOK * 128 / 16) + 2 * ((kl >> 4) & 3));
        }
    }
    const uint32_t idesc = tc::idesc_f16kind(BM, NTOK, (uint32_t)load_mode(a));
    int j = p.j_lo;
    int seg = -1;
    int sx = 0, sa = 0;
    uint32_t phx = 0, pha = 0;
    for (int i = 0; i < p.n_units; ++i) {
        const bool first = (i == 0) || j == p.jb;
        const bool last = (i == p.n_units - 1) || j == p.je - 1;
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
        for (int h = 0; h < kI; ++h) {
            if (!tc::mbar_wait(&p.a_full[sa], pha)) {
                fail(a, 15);
                return;
            }
            tc::fence_after_sync();
            const uint32_t acol = p.tmem_a + (uint32_t)(sa * C::kACols);
#pragma unroll
            for (int t = 0; t < kT; ++t)
                tc::mma_f16_ts(dcol, acol + aoff[t], bdesc0 + boff[h][t], idesc,
                               (first && h == 0 && t == 0) ? 0u : 1u);
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
        if (++j == p.je)
            j = p.jb;
    }
}

template <int NW, int FMT = 0>
__global__ void __launch_bounds__(kThreads, 1)
skinny_tc_kernel(const __grid_constant__ CUtensorMap m_codes0, const __grid_constant__ CUtensorMap m_codes1,
                 const __grid_constant__ CUtensorMap m_scales0, const __grid_constant__ CUtensorMap m_scales1,
                 const __grid_constant__ CUtensorMap m_x, Args a)
{
    using C = Cfg<NW, FMT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *c_ring = smem;                                          // [kCStages][NW codes, NW scales]
    uint8_t *x_ring = c_ring + (size_t)C::kCStages * C::kStageBytes;  // [kXStages][8 KB]
    float *ck_buf = reinterpret_cast<float *>(x_ring + (size_t)C::kXStages * kXUnit);  // [128][NW * 16]
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(ck_buf) + C::kCkBytes);
    uint64_t *c_full = bars;
    uint64_t *c_empty = c_full + C::kCStages;
    uint64_t *x_full = c_empty + C::kCStages;
    uint64_t *x_empty = x_full + C::kXStages;
    uint64_t *a_full = x_empty + C::kXStages;
    uint64_t *a_empty = a_full + C::kAStages;
    uint64_t *d_full = a_empty + C::kAStages;
    uint64_t *d_empty = d_full + 2;
    uint64_t *ck_full = d_empty + 2;
    uint64_t *ck_free = ck_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ck_free + 1);
    float *fac_s = reinterpret_cast<float *>(tmem_slot + 4);  // [NW][16] epilogue factors
    SegInfo *seg_s = reinterpret_cast<SegInfo *>(fac_s + 2 * NTOK);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;

    if (threadIdx.x == 0) {
        // Let the next kernel in the stream be scheduled as soon as SMs free up;
        // it waits for this grid's completion before it reads anything we write.
        tc::griddep_launch_dependents();
        // Consumers arrive once per warp (lane 0 after __syncwarp): hundreds
        // of per-thread arrivals on one mbarrier serialise in shared memory.
        for (int s = 0; s < C::kCStages; ++s) {
            tc::mbar_init(&c_full[s], 1);
            tc::mbar_init(&c_empty[s], C::kReaders);
        }
        for (int s = 0; s < C::kXStages; ++s) {
            tc::mbar_init(&x_full[s], 1);
            tc::mbar_init(&x_empty[s], kMmaWarps);
        }
        for (int s = 0; s < C::kAStages; ++s) {
            tc::mbar_init(&a_full[s], 4);  // the four warps of one group
            tc::mbar_init(&a_empty[s], kMmaWarps);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&d_full[s], kMmaWarps);
            tc::mbar_init(&d_empty[s], kEpiThreads / 32);
        }
        tc::mbar_init(ck_full, a.cs > 1 ? a.cs : 1);
        tc::mbar_init(ck_free, 1);
        tc::fence_mbar_init();
        tc::prefetch_tensormap(&m_codes0);
        if (FMT == 0)
            tc::prefetch_tensormap(&m_scales0);
        if (NW == 2) {
            tc::prefetch_tensormap(&m_codes1);
            if (FMT == 0)
                tc::prefetch_tensormap(&m_scales1);
        }
    }
    if (warp == 0)
        tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (a.cs > 1)
        tc::cluster_sync();  // every CTA's barriers are initialised before remote arrivals
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_a = tmem;
    const uint32_t tmem_d = tmem + C::kAStages * C::kACols;

    // Every role walks the CTA's units lo..hi-1 with incremental (tile, j)
    // and ring (stage, phase) counters: no 64-bit division in the loops.
    const Range rg = cta_range(a, b);
    const int n_units = rg.n_units;
    const int64_t tile_lo = rg.tile0;
    const int j_lo = rg.j_first;

    if (warp == 4 || warp == 5) {
        // ---- weight producers: even units (warp 4) and odd units (warp 5);
        // a unit's code and scale boxes complete one barrier ----
        if (lane == 0) {
            const int par = warp - 4;
            int64_t tile = tile_lo;
            int j = j_lo + par;
            if (j >= rg.je) {
                j -= rg.je - rg.jb;
                tile += rg.tstep;
            }
            for (int i = par; i < n_units; i += 2) {
                const int s = i % C::kCStages;
                const uint32_t ph = (uint32_t)(i / C::kCStages) & 1;
                if (!tc::mbar_wait(&c_empty[s], ph ^ 1)) {
                    fail(a, 11);
                    break;
                }
                uint8_t *st = c_ring + (size_t)s * C::kStageBytes;
                tc::mbar_arrive_expect_tx(&c_full[s], C::kStageBytes);
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
                    if (FMT == 0) {
                        tc::tma_load_2d(st + mi * kCodeBox, mi == 0 ? &m_codes0 : &m_codes1, &c_full[s],
                                        j * (BKU / 2), (int)(tile * BM));
                        tc::tma_load_2d(st + NW * kCodeBox + mi * kScaleBox, mi == 0 ? &m_scales0 : &m_scales1,
                                        &c_full[s], j * (BKU / 16), (int)(tile * BM));
                    } else {
#pragma unroll
                        for (int bx = 0; bx < 3; ++bx)
                            tc::tma_load_2d(st + (mi * 3 + bx) * kCodeBox6, mi == 0 ? &m_codes0 : &m_codes1,
                                            &c_full[s], j * (BKU / 4 * 3) + bx * 64, (int)(tile * BM));
                    }
                }
                j += 2;
                while (j >= rg.je) {
                    j -= rg.je - rg.jb;
                    tile += rg.tstep;
                }
            }
        }
    } else if (warp == 6) {
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
                if (++j == rg.je)
                    j = rg.jb;
            }
        }
    } else if (warp < kMmaWarps) {
        // ---- MMA issuers: issuer q owns matrix q / kChains, chain q % kChains ----
        if (lane == 0) {
            tc::griddep_wait();
            IssuerArgs ia{x_ring, x_full, x_empty, a_full, a_empty, d_full, d_empty, tmem_a, tmem_d, n_units, j_lo,
                          rg.jb, rg.je};
            mma_issuer<NW>(a, ia, warp);
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ---- epilogue (warps 8..11, one per TMEM lane quarter) ----
        tc::griddep_wait();
        const int mode = load_mode(a);
        const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..127
        if (et < NW * NTOK) {
            const int mi = et / NTOK, n = et % NTOK;
            if (FMT == 1) {
                fac_s[et] = 1.0f;  // FP6: the dequantised weights carry their scale exactly
            } else {
                const float t = __ldg(a.ts[mi]);
                fac_s[et] = mode ? t * 256.0f : t * a.factor[n];
            }
        }
        if (et == 0)
            seg_s->reduce = 0;
        tc::named_bar_sync(1, kEpiThreads);  // fac_s visible to all epilogue threads
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        int64_t tile = tile_lo;
        int j = j_lo;
        int seg = -1, seg_j0 = 0;
        for (int i = 0; i < n_units; ++i) {
            const bool first = (i == 0) || j == rg.jb;
            const bool last = (i == n_units - 1) || j == rg.je - 1;
            if (first) {
                ++seg;
                seg_j0 = j;
            }
            if (last) {
                const int db = seg & 1;
                // every epilogue thread takes the same branch (named barriers follow)
                if (!tc::bar_and(1, kEpiThreads, tc::mbar_wait(&d_full[db], ((uint32_t)seg >> 1) & 1))) {
                    fail(a, 18);
                    if (et == 0)
                        seg_s->reduce = 0;
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
                if (a.cs > 1) {
                    ck_epilogue<NW>(a, fac_s, sum, tile, r, et, seg, ck_buf, ck_full, ck_free);
                    if (++j == rg.je) {
                        j = rg.jb;
                        tile += rg.tstep;
                    }
                    continue;
                }
                // this CTA did the whole tile: units 0 .. C-1
                const bool whole = seg_j0 == 0 && j == a.C - 1;
                publish_segment<NW>(a, fac_s, sum, (int)tile, whole, (int)tile_lo, b, r, seg_s);
                if (i == n_units - 1)
                    break;  // the CTA's last segment is reduced by all threads below
                if (seg_s->reduce)
                    reduce_tile<NW>(a, fac_s, *seg_s, r, kEpiThreads);
            }
            if (++j == rg.je) {
                j = rg.jb;
                tile += rg.tstep;
            }
        }
        // cluster-K: the leader has read this CTA's last partial before it exits
        if (a.cs > 1 && seg >= 0 && !tc::mbar_wait_cluster(ck_free, (uint32_t)seg & 1))
            fail(a, 25);
        // The dequantisers have finished: they help with the last segment.
        tc::named_bar_sync(2, kEpiThreads + kDqWarps * 32);
        if (seg_s->reduce)
            reduce_tile<NW>(a, fac_s, *seg_s, r, kEpiThreads + kDqWarps * 32);
    } else if (warp >= kFirstDqWarp) {
        // ---- dequantisers (warps 12..27): group g takes items t = g (mod 4) ----
        tc::griddep_wait();
        const int mode = load_mode(a);
        const int g = (warp - kFirstDqWarp) >> 2;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;  // row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int swz = r & 7;
        constexpr int kCh = BKU / C::kItems / 32;  // 16-byte code chunks per matrix and item
        const int h = (NW == 1) ? (g & 1) : g;     // item within the unit
        int i = (NW == 1) ? (g >> 1) : 0;          // first unit of this group
        // Ring positions: unit i in the weight ring, item i * kItems + h in the
        // A ring (both below the ring sizes here, so phase 0).
        int sc = i, sa = i * C::kItems + h;
        uint32_t phc = 0, pha = 0;
        // FP6: this thread's scale byte of each item (one per 128 k of its row)
        // comes from global memory, loaded kSPf items of the group ahead.
        constexpr int kSPf = 3;
        constexpr int kCh6 = BKU / C::kItems * 3 / 4 / 16;  // 16-byte FP6 code chunks per matrix and item
        auto scale6 = [&](int iu, int mi) -> uint32_t {
            if (FMT != 1 || iu >= n_units)
                return 127u;
            const uint32_t span = (uint32_t)(rg.je - rg.jb);
            const uint32_t L = (uint32_t)(rg.j_first - rg.jb) + (uint32_t)iu;
            const int64_t m = (rg.tile0 + (int64_t)(L / span) * rg.tstep) * BM + r;
            const int blk = 2 * (rg.jb + (int)(L % span)) + (NW == 1 ? h : (h >> 1));
            return m < a.M ? (uint32_t)__ldg(a.scales6[mi] + m * (a.K / 128) + blk) : 127u;
        };
        uint32_t s6ring[kSPf][NW], scl6[NW];
        if (FMT == 1) {
#pragma unroll
            for (int p = 0; p < kSPf; ++p)
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    s6ring[p][mi] = scale6(i + p * C::kUnitStep, mi);
        }
        for (int it = 0; i < n_units; i += C::kUnitStep, ++it) {
            if (!tc::mbar_wait(&c_full[sc], phc)) {
                fail(a, 16);
                break;
            }
            // copy this thread's codes and scale bytes to registers, release the stage
            const uint8_t *stage = c_ring + (size_t)sc * C::kStageBytes;
            uint4 cw[NW][FMT == 0 ? kCh : kCh6];
            uint32_t scw[NW][kCh / 2];
            if (FMT == 1) {
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
#pragma unroll
                    for (int c = 0; c < kCh6; ++c) {
                        // byte b of the unit row: box b / 64, 16-byte chunk (b / 16) % 4, 64-byte swizzle
                        const int b6 = h * kCh6 * 16 + 16 * c;
                        cw[mi][c] = *reinterpret_cast<const uint4 *>(
                            stage + (mi * 3 + (b6 >> 6)) * kCodeBox6 + r * 64 + ((((b6 >> 4) & 3) ^ ((r >> 1) & 3)) << 4));
                    }
#pragma unroll
                    for (int p = 0; p < kSPf; ++p)
                        if (it % kSPf == p) {
                            scl6[mi] = s6ring[p][mi];
                            s6ring[p][mi] = scale6(i + kSPf * C::kUnitStep, mi);
                        }
                }
            }
#pragma unroll
            for (int mi = 0; mi < NW && FMT == 0; ++mi) {
                const uint8_t *crow = stage + mi * kCodeBox + r * 128;
#pragma unroll
                for (int c = 0; c < kCh; ++c)
                    cw[mi][c] = *reinterpret_cast<const uint4 *>(crow + (((h * kCh + c) ^ swz) << 4));
                // scale bytes of the item: two per chunk, 16 per row and unit
                const uint8_t *srow = stage + NW * kCodeBox + mi * kScaleBox + r * 16 + h * kCh * 2;
                if (kCh == 4) {
                    const uint2 v2 = *reinterpret_cast<const uint2 *>(srow);
                    scw[mi][0] = v2.x;
                    scw[mi][kCh / 2 - 1] = v2.y;
                } else {
                    scw[mi][0] = *reinterpret_cast<const uint32_t *>(srow);
                }
            }
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(&c_empty[sc]);
            sc += C::kUnitStep;
            if (sc >= C::kCStages) {
                sc -= C::kCStages;
                phc ^= 1;
            }

            // dequantise into A stage sa: 64 columns = two stores of 32
            if (!tc::mbar_wait(&a_empty[sa], pha ^ 1)) {
                fail(a, 17);
                break;
            }
            tc::fence_after_sync();
            const uint32_t acol = tmem_a + sa * C::kACols + lane_off;
#pragma unroll
            for (int q = 0; q < 2; ++q) {  // NW = 1: chunks 2q, 2q+1; NW = 2: matrix q
                const int mi = NW == 1 ? 0 : q;
                if constexpr (FMT == 1) {
                    // 64 k = eight 8-code groups of 6 bytes, from this item's code words
                    const Fp6Mult mult = fp6_mult(scl6[mi]);
                    auto w = [&](int k) -> uint32_t {  // code word k of the item (constant after unrolling)
                        const uint4 &v = cw[mi][k >> 2];
                        return (k & 3) == 0 ? v.x : (k & 3) == 1 ? v.y : (k & 3) == 2 ? v.z : v.w;
                    };
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t out[16];
#pragma unroll
                        for (int gg = 0; gg < 4; ++gg) {
                            const int gi = (NW == 1 ? 8 * q : 0) + 4 * hh + gg;  // group within the item
                            const int wi = (6 * gi) >> 2;
                            const bool odd = ((6 * gi) & 3) != 0;             // group starts mid-word
                            const uint32_t lo = odd ? (w(wi) >> 16) | (w(wi + 1) << 16) : w(wi);
                            const uint32_t hi = odd ? (w(wi + 1) >> 16) : (w(wi + 1) & 0xFFFFu);
                            const uint4 pv = e2m3x8_to_bf16(lo, hi);
                            out[4 * gg + 0] = fp6_apply(pv.x, mult);
                            out[4 * gg + 1] = fp6_apply(pv.y, mult);
                            out[4 * gg + 2] = fp6_apply(pv.z, mult);
                            out[4 * gg + 3] = fp6_apply(pv.w, mult);
                        }
                        tc::tmem_st_32x32b_x16(acol + q * 32 + hh * 16, out);
                    }
                } else {
                    const int c0 = NW == 1 ? 2 * q : 0;
                    const uint32_t sw = scw[mi][NW == 1 ? q : 0];
                    uint32_t out[32];
                    dequant_chunk(cw[mi][c0], sw & 0xFFFF, mode, out);
                    dequant_chunk(cw[mi][c0 + 1], sw >> 16, mode, out + 16);
                    tc::tmem_st_32x32b_x32(acol + q * 32, out);
                }
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(&a_full[sa]);
            sa += kGroups;
            if (sa >= C::kAStages) {
                sa -= C::kAStages;
                pha ^= 1;
            }
        }
        // help the epilogue threads add the partials of the CTA's last segment
        tc::named_bar_sync(2, kEpiThreads + kDqWarps * 32);
        if (seg_s->reduce)
            reduce_tile<NW>(a, fac_s, *seg_s, kEpiThreads + (threadIdx.x - kFirstDqWarp * 32),
                            kEpiThreads + kDqWarps * 32);
    }

    // Lane 0 of the producer and MMA warps ran their loops alone: reconverge
    // each warp first, so the block-wide barrier below really waits for every
    // thread (a partially arrived warp would otherwise count as arrived).
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    // Cluster-K: no CTA leaves while a peer may still read its shared memory
    // or arrive on its barriers (even after a wait of either gave up).  Every
    // wait before this point is bounded, so every thread gets here.
    if (a.cs > 1)
        tc::cluster_sync();
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

template <int NW, int FMT = 0>
cudaError_t set_smem_attr()
{
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    return once_per_device(once, attr_err, [] {
        return cudaFuncSetAttribute(skinny_tc_kernel<NW, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)Cfg<NW, FMT>::kSmemBytes);
    });
}

template <int NW, int FMT = 0>
cudaLaunchConfig_t main_config(const Args &a, cudaStream_t stream, cudaLaunchAttribute (&attr)[2])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<NW, FMT>::kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)(a.cs > 1 ? a.cs : 1);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.cs > 1 ? 2 : 1;
    return cfg;
}

// Clusters of `cs` CTAs of the main kernel that fit on the current device at
// once (0 if none), cached per device.
template <int NW, int FMT = 0>
int max_active_clusters(int cs)
{
    static std::mutex mu;
    static int cache[64][3];
    static bool have[64][3];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || set_smem_attr<NW, FMT>() != cudaSuccess)
        return 0;
    const int ci = cs == 2 ? 0 : (cs == 4 ? 1 : 2);
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev][ci]) {
        Args probe{};
        probe.cs = cs;
        probe.P = cs;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = main_config<NW, FMT>(probe, nullptr, attr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, skinny_tc_kernel<NW, FMT>, &cfg) != cudaSuccess)
            n = 0;
        cudaGetLastError();  // a failed query leaves no sticky error
        cache[dev][ci] = n;
        have[dev][ci] = true;
    }
    return cache[dev][ci];
}

template <int NW, int FMT = 0>
cudaError_t launch_main(const CUtensorMap (&maps)[5], const Args &a, cudaStream_t stream)
{
    const cudaError_t attr_err = set_smem_attr<NW, FMT>();
    if (attr_err != cudaSuccess)
        return attr_err;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = main_config<NW, FMT>(a, stream, attr);
    return cudaLaunchKernelEx(&cfg, skinny_tc_kernel<NW, FMT>, maps[0], maps[1], maps[2], maps[3], maps[4], a);
}

// Split of the K dimension of every tile: stream-K over all SMs (any split,
// partials reduced through global memory by the last CTA to arrive), or
// cluster-K (clusters of 2 or 4 CTAs each splitting whole tiles, partials
// reduced through distributed shared memory: a shorter end of call, but the
// tiles must spread over fewer, fixed-size groups).  The choice depends on
// the shapes and the device only, never on N, so results do not depend on N.
// Unit times per SM and the end-of-call saving are measured on GB300.
template <int NW, int FMT = 0>
void choose_split(Args &a, int num_sms)
{
    a.cs = 1;
    a.ncl = 0;
    a.P = (int)std::max<int64_t>(1, std::min<int64_t>(a.total, std::min<int64_t>(num_sms, kSkinnyTcMaxCtas)));
    // us per 128 x 256 unit (per matrix pair) per SM; FP6 units carry 1.35x the bytes
    const double t_unit = (NW == 1 ? 0.55 : 1.1) * (FMT == 1 ? 1.35 : 1.0);
    const double tail_saving = 3.0;               // us: global split-K reduction vs cluster reduction
    // Enough tiles to fill nearly every SM one each: whole tiles, no split-K.
    // The split's partial stores and last-arriver reduction then cost more
    // than the few idle SMs (27B gate/up, 136 tiles on 152 SMs: decode streams
    // at N = 4 / 9 / 16 +3 / +11 / +22 %, N = 1 -2 %).  With 60 % of the SMs
    // (9B gate/up, 96 tiles) the N = 1 decode stream lost 8 %, so the bar is
    // 85 %.  FP6 units carry 1.35x the bytes, so the split's overhead weighs
    // less: its 27B gate/up stream went 2.11 -> 2.00 TB/s at N = 1 without the
    // split (1.87 -> 1.95 at N = 16), and FP6 keeps stream-K.
    if (FMT == 0 && a.T <= num_sms && a.T <= kSkinnyTcMaxCtas && a.T * 100 >= (int64_t)num_sms * 85) {
        a.P = (int)a.T;
        return;
    }
    double best = (double)((a.total + a.P - 1) / a.P) * t_unit + tail_saving;
    // Measured: cluster-K wins only for one matrix whose tiles fit one per
    // cluster (e.g. 4096 x 4096: 11.6 -> 10.6 us at N = 1); with several tiles
    // per cluster, or for the fused gate/up pair, it was slower (whole
    // clusters must free up before they start).
    if constexpr (NW == 1) {
        for (int cs : {4, 2}) {
            if (a.C < cs)
                continue;
            const int64_t ncl = std::min<int64_t>(a.T, max_active_clusters<NW, FMT>(cs));
            if (ncl < 1 || ncl < a.T || ncl * cs > kSkinnyTcMaxCtas)
                continue;
            const int64_t tiles = (a.T + ncl - 1) / ncl, units = (a.C + cs - 1) / cs;
            const double est = (double)(tiles * units) * t_unit;
            if (est < best) {
                best = est;
                a.cs = cs;
                a.ncl = (int)ncl;
                a.P = (int)(ncl * cs);
            }
        }
    }
}

}  // namespace sk

// Units (128 rows x 256 k) times CTAs must stay below 2^31: the kernel's
// stream-K arithmetic is 32-bit.
bool skinny_tc_supported(int64_t M, int64_t K)
{
    if (K < 256 || K % 256 != 0 || M < 1)
        return false;
    const int64_t tiles = (M + 127) / 128;
    const int64_t units = tiles * (K / 256);
    return units * kSkinnyTcMaxCtas < (INT64_C(1) << 31) && tiles * 4 <= (int64_t)sk::kCounterRegion;
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
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + kStatusWordOffset);

    Args a{};
    a.N = N;
    a.M = M;
    a.K = K;
    a.C = (int)((K + BKU - 1) / BKU);
    a.T = (M + BM - 1) / BM;
    a.total = a.T * a.C;
    if (n_weights == 1)
        choose_split<1>(a, num_sms);
    else
        choose_split<2>(a, num_sms);
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
        static_assert(kCodeBox == BM * (BKU / 2) && kScaleBox == BM * (BKU / 16), "box sizes");
        if (!make_map(&maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, codes[s], (uint64_t)K / 2, (uint64_t)M,
                      (uint64_t)K / 2, BKU / 2, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&maps[2 + i], CU_TENSOR_MAP_DATA_TYPE_UINT8, scales[s], (uint64_t)K / 16, (uint64_t)M,
                      (uint64_t)K / 16, BKU / 16, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    // x itself ([N][K] bf16), read by the main kernel in bf16 mode: boxes of
    // 64 k x N rows with the 128-byte swizzle of the MMA operand layout.
    if (!make_map(&maps[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64,
                  (uint32_t)N, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    // One matrix with N >= 2: no prep kernel; the main kernel reads x itself as
    // bf16 operands (products exact either way, and fp32 sums of exactly
    // scaled products scale exactly, so the results are the same bits).  The
    // prep's latency outweighs the cheaper f16 dequantisation here, while the
    // fused gate/up pair (twice the dequantisation per unit) and N = 1 keep
    // it.  The split-K counters are then zero from the previous call (every
    // call leaves the workspace zero) instead of being zeroed by the prep.
    a.bf16_only = (n_weights == 1 && N >= 2) ? 1 : 0;
    if (!a.bf16_only) {
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
                                           a.counters, a.T);
        if (e != cudaSuccess)
            return e;
    }
    return n_weights == 1 ? launch_main<1>(maps, a, stream) : launch_main<2>(maps, a, stream);
}

cudaError_t launch_skinny_tc_fp6(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                                 const uint8_t *const *scales, int n_weights, void *y, int out_bf16,
                                 void *workspace, int num_sms, cudaStream_t stream)
{
    using namespace sk;
    const WsLayout L = ws_layout(M, K, n_weights);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    Args a{};
    a.N = N;
    a.M = M;
    a.K = K;
    a.C = (int)(K / BKU);
    a.T = (M + BM - 1) / BM;
    a.total = a.T * a.C;
    if (n_weights == 1)
        choose_split<1, 1>(a, num_sms);
    else
        choose_split<2, 1>(a, num_sms);
    for (int i = 0; i < 2; ++i) {
        a.ts[i] = nullptr;
        a.scales6[i] = scales[i < n_weights ? i : 0];
    }
    a.factor = reinterpret_cast<float *>(ws);
    a.flags = reinterpret_cast<int *>(ws + 64);
    a.counters = reinterpret_cast<uint32_t *>(ws + L.counters);
    a.partial = reinterpret_cast<float *>(ws + L.partial);
    a.x_img = ws + L.ximg;
    a.err = reinterpret_cast<uint32_t *>(ws + kStatusWordOffset);
    a.y = y;
    a.out_bf16 = out_bf16;
    a.bf16_only = 1;  // FP6 weights take bf16 operands: no prep kernel

    CUtensorMap maps[5];
    for (int i = 0; i < 2; ++i) {
        const int s = i < n_weights ? i : 0;
        // a unit's 192 code bytes per row as three [128 rows][64 B] boxes, 64-byte swizzle
        if (!make_map(&maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, codes[s], (uint64_t)K / 4 * 3, (uint64_t)M,
                      (uint64_t)K / 4 * 3, 64, BM, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
        maps[2 + i] = maps[i];  // no scale maps
    }
    if (!make_map(&maps[4], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64,
                  (uint32_t)N, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    return n_weights == 1 ? launch_main<1, 1>(maps, a, stream) : launch_main<2, 1>(maps, a, stream);
}

}  // namespace nvfp4
