// prefill.cu -- NVFP4 x bf16 products for N > 16 tokens on the 5th-generation
// tensor cores (tcgen05), with an optional SwiGLU epilogue for the gate/up pair.
//
// The prefill of both engines on the pages multiplies each weight by many
// tokens at once: qwentin README, "How it works" (a wide GEMM reading every
// weight once for N tokens); bw24 README, NVFP4 decode path (a tensor-core GEMM
// for prefill).  Their kernels target consumer Blackwell (mma.sync, int8 or FP6
// block-scale); this one is written for sm_103a:
//
//   CTA tile: 128 weight rows (MMA M) x 256 tokens (MMA N), K in stages of 64.
//   warp 0      TMA producer: x tile [256 tokens][64 k] bf16, 128-byte swizzle.
//   warp 1      allocates TMEM.  Warps 1 and 2: one thread each issues
//               tcgen05.mma (bf16 x bf16 -> fp32, A and B from shared
//               memory) and commits to mbarriers: for the gate/up pair each
//               owns one matrix's accumulator, for one matrix each takes half
//               of every stage's K steps into its own accumulator (a thread
//               needs longer to issue an M=128, N=256 MMA than the tensor core
//               needs to run it).
//   warps 3..10 dequantise: each thread turns 32 k of one weight row (16 code
//               bytes, 2 scale bytes) into exact bf16 values e2m1 * scale * 2^-8
//               and stores them in the 128-byte-swizzled K-major layout the
//               MMA reads; then, after the K loop, they read the fp32
//               accumulators out of TMEM (tcgen05.ld) and store
//               y = acc * 2^8 * ts, or h = silu(g) * u for the gate/up pair.
//   warp 11     (K % 256 == 0) streams the weight codes ([128 rows][32 B] per
//               stage) and scales ([128 rows][16 B] per four stages) into
//               shared-memory rings by TMA, so the dequantisers read shared
//               memory.  Per-thread global loads of 16 bytes from 128
//               different rows kept the load/store unit busy with one
//               wavefront per row; that, not the tensor pipe, bounded the
//               kernel.  Other K (and the FP6 format) load codes and scales per
//               thread from global memory through a 4-stage register ring.
//               FP6 weights (K % 128 == 0) take their codes ([128 rows][48 B]
//               per stage) by TMA as well and their scale bytes (one per 128 k)
//               through a small register ring.
//   One matrix with TMA-fed weights: the dequantisers write the A operand to
//   tensor memory (tcgen05.st, a 4-stage ring beside the accumulator) and
//   warp 1 alone issues every MMA (kind::f16, A from tensor memory) into one
//   accumulator; the shared-memory A path's proxy fence per stage cost that
//   kernel ~12 %.  The gate/up pair keeps A in shared memory: its two
//   256-column accumulators fill the tensor memory.
//
// Exactness: every product e2m1 * scale * x is exact in the fp32 accumulator
// (bf16 operands with at most 6 and 8 significant bits).  The accumulation
// order is fixed by the shapes, so results are deterministic.
//
// Every mbarrier wait is bounded (2 s of wall time): on a timeout the kernel
// sets word 0 of the workspace to a nonzero code and every role leaves its
// loop, so the kernel ends instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace pf {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int kDqWarps = 8;
constexpr int kIssuers = 2;  // MMA-issuing warps (1 and 2)
constexpr int kFirstDqWarp = 1 + kIssuers;
constexpr int kThreads = kFirstDqWarp * 32 + kDqWarps * 32;
constexpr int kCodeWarp = kFirstDqWarp + kDqWarps;  // code / scale TMA producer (TMA-code mode)
constexpr int kThreadsTma = kThreads + 32;
constexpr int kSBytes = BM * 16;         // NVFP4 scales of four stages: 128 rows x 16 bytes
// codes of one stage: 128 rows x 32 bytes (NVFP4) or 48 bytes (FP6)
template <int FMT> constexpr int code_row_bytes() { return FMT == 0 ? BK / 2 : BK / 4 * 3; }
constexpr int kABytes = BM * BK * 2;  // 16 KB per weight matrix per stage

// TMAC: the weight codes and scales reach shared memory by TMA (a code ring
// of kSc stages and a scale ring of two 4-stage groups) instead of per-thread
// global loads; needs K % 256 == 0 (16-byte row pitch of the scale rows).
// TA (TMA-fed, one matrix): the dequantised A operand goes to tensor memory
// (tcgen05.st) instead of shared memory, and one thread issues every MMA into
// a single accumulator: no generic-to-async proxy fence per stage, no A tile
// in shared memory.  Tensor memory: accumulator in columns [0, TN), A ring of
// kStages x 32 columns from column kAcol0.
template <int NW, bool TMAC = false, int FMT = 0, int TN = BN>
struct Cfg {
    static constexpr bool kTA = TMAC && NW == 1;
    static constexpr int kBBytes = TN * BK * 2;           // activation tile of one stage
    static constexpr int kStages = NW == 1 ? 4 : 3;
    static constexpr int kPf = 4;                         // dequant register prefetch depth (K steps in flight)
    static constexpr int kCBytes = BM * code_row_bytes<FMT>();
    static constexpr int kSc =
        kTA ? (FMT == 0 ? 12 : 8) : (FMT == 0 ? (NW == 1 ? 6 : 3) : (NW == 1 ? 5 : 2));  // code ring (TMAC)
    static constexpr int kAcol0 = 256;
    static constexpr uint32_t kTmemCols = 512;  // two accumulators of 256 columns, or one + the A ring
    static constexpr int kIssue = kTA ? 1 : kIssuers;     // threads issuing MMAs
    static constexpr size_t kRingBytes =
        TMAC ? (size_t)kSc * NW * kCBytes + (FMT == 0 ? 2 * NW * kSBytes : 0) : 0;
    static constexpr size_t kSmemBytes = (size_t)kStages * ((kTA ? 0 : NW * kABytes) + kBBytes) + kRingBytes +
                                         1024 /* barriers */ + 1024 /* alignment */;
    static_assert(kSmemBytes <= 232448, "shared memory per block");
};

struct Args {
    const uint8_t *codes[2];
    const uint8_t *scales[2];
    const float *ts[2];
    void *y;
    int out_bf16;
    int64_t N, M, K;
    int num_kb;
    uint32_t *err;
    int row_tiles, token_tiles, group;  // raster: groups of `group` row tiles
    // Split mode (one matrix, A in tensor memory, fewer tiles than SMs): the
    // grid's CTAs take equal contiguous ranges of the (tile, 256-k group)
    // units, so a CTA has at most two tile segments; a tile shared by several
    // CTAs is finished by the last to arrive, adding every CTA's fp32 partial
    // in CTA order.
    int split;
    int grid;             // CTAs: one per tile, or (split mode) one per SM
    int kq;               // 256-k groups per tile (num_kb / 4)
    int64_t units;        // tiles * kq
    float *partial;       // [2 * gridDim][TN][BM] raw fp32 accumulators
    uint32_t *counters;   // [tiles] arrivals (zeroed by the host before the launch)
};

// Tile index -> (row tile, token tile) in the raster order: groups of `group`
// weight row tiles; inside a group row tiles vary fastest, then token tiles.
NVFP4_DEVINL void tile_coords(const Args &a, int64_t tile, int64_t &row_tile, int64_t &token_tile)
{
    const int64_t per_group = (int64_t)a.group * a.token_tiles;
    const int64_t gidx = tile / per_group;
    const int64_t first = gidx * a.group;
    const int64_t rows = (a.row_tiles - first) < a.group ? (a.row_tiles - first) : a.group;
    const int64_t in = tile - gidx * per_group;
    row_tile = first + in % rows;
    token_tile = in / rows;
}

// The k blocks a CTA computes: one segment (a whole tile) without split mode,
// else one or two segments of its unit range.  Scalars, not arrays: the
// segment of a stage is picked with selects, so nothing goes to local memory.
struct Segs {
    int n;
    int64_t tile_a, tile_b;
    int kb0_a, kb0_b, nkb_a, nkb_b;  // first 64-k block and number of blocks of each segment
    int64_t m0_a, m0_b;
    int n0_a, n0_b;
    bool whole_a, whole_b;
};

// CTA whose unit range holds unit u (ranges [b * units / G, (b + 1) * units / G)).
NVFP4_DEVINL int64_t split_cta_of(int64_t u, int64_t units, int64_t G) { return ((u + 1) * G - 1) / units; }

template <int TN, bool SPLIT>
NVFP4_DEVINL Segs cta_segments(const Args &a, int64_t b, int64_t G)
{
    Segs sg{};
    if (!SPLIT) {
        sg.n = 1;
        sg.tile_a = b;
        sg.kb0_a = 0;
        sg.nkb_a = a.num_kb;
        sg.whole_a = true;
    } else {
        const int64_t lo = b * a.units / G, hi = (b + 1) * a.units / G;
        sg.n = 0;
        if (lo < hi) {
            const int64_t t = lo / a.kq;
            const int64_t e = (t + 1) * a.kq < hi ? (t + 1) * a.kq : hi;
            sg.n = 1;
            sg.tile_a = t;
            sg.kb0_a = (int)(lo - t * a.kq) * 4;
            sg.nkb_a = (int)(e - lo) * 4;
            sg.whole_a = (lo == t * a.kq) && (e == (t + 1) * a.kq);
            if (e < hi) {  // the range reaches into the next tile (at most one more: units / G <= kq)
                sg.n = 2;
                sg.tile_b = t + 1;
                sg.kb0_b = 0;
                sg.nkb_b = (int)(hi - e) * 4;
                sg.whole_b = hi == (t + 2) * a.kq;
            }
        }
    }
    int64_t rt, tt;
    tile_coords(a, sg.tile_a, rt, tt);
    sg.m0_a = rt * BM;
    sg.n0_a = (int)(tt * TN);
    if (sg.n > 1) {
        tile_coords(a, sg.tile_b, rt, tt);
        sg.m0_b = rt * BM;
        sg.n0_b = (int)(tt * TN);
    }
    return sg;
}

// Exact bf16 dequantisation of one 32-bit code word (k = 8q .. 8q+7) into
// four bf16x2 words in natural k order, each value e2m1 * scale * 2^-8.
NVFP4_DEVINL uint4 dequant_word_natural(uint32_t w, uint32_t mult)
{
    constexpr uint32_t kMag = 0x01C001C0u;
    const uint32_t te = w & 0x08080808u;
    const uint32_t to = w & 0x80808080u;
    const uint32_t p0 = bf16x2_mul(((w << 6) & kMag) | ((te << 12) & ~kMag), mult);  // k0, k4
    const uint32_t p1 = bf16x2_mul(((w << 2) & kMag) | ((to << 8) & ~kMag), mult);   // k1, k5
    const uint32_t p2 = bf16x2_mul(((w >> 2) & kMag) | ((te << 4) & ~kMag), mult);   // k2, k6
    const uint32_t p3 = bf16x2_mul(((w >> 6) & kMag) | (to & ~kMag), mult);          // k3, k7
    return make_uint4(prmt(p0, p1, 0x5410),   // k0, k1
                      prmt(p2, p3, 0x5410),   // k2, k3
                      prmt(p0, p1, 0x7632),   // k4, k5
                      prmt(p2, p3, 0x7632));  // k6, k7
}

NVFP4_DEVINL uint32_t scale_mult_bf16(uint32_t byte)
{
    return f32_to_bf16x2_bcast(__fmul_rn(e4m3_to_f32(byte & 0xFF), 0x1p118f));
}

struct DqItem {
    uint4 code;   // 16 code bytes = 32 k of one row
    uint32_t scl; // 2 scale bytes
};

template <bool ALIGNED>
NVFP4_DEVINL DqItem dq_load(const Args &a, int mi, int64_t m, int kb, int half)
{
    DqItem it{make_uint4(0, 0, 0, 0), 0};
    const int64_t k0 = (int64_t)kb * BK + half * 32;
    const int64_t rem = a.K - k0;
    if (m >= a.M || rem <= 0)
        return it;
    const uint8_t *cp = a.codes[mi] + m * (a.K >> 1) + (k0 >> 1);
    const uint8_t *sp = a.scales[mi] + m * (a.K >> 4) + (k0 >> 4);
    if (rem >= 32) {
        if (ALIGNED) {
            it.code = ldg_stream_v4(cp);
            it.scl = __ldg(reinterpret_cast<const uint16_t *>(sp));
        } else {
            const uint2 lo = ldg_stream_v2(cp), hi = ldg_stream_v2(cp + 8);
            it.code = make_uint4(lo.x, lo.y, hi.x, hi.y);
            it.scl = (uint32_t)__ldg(sp) | ((uint32_t)__ldg(sp + 1) << 8);
        }
    } else {  // 16 valid k
        const uint2 lo = ldg_stream_v2(cp);
        it.code = make_uint4(lo.x, lo.y, 0, 0);
        it.scl = __ldg(sp);
    }
    return it;
}

// FP6 E2M3 weights: 32 k of one row = 24 code bytes and the scale byte of the
// row's 128-k block (K % 128 == 0, so every stage is complete).
struct DqItem6 {
    uint2 code[3];
    uint32_t scl;
};

NVFP4_DEVINL DqItem6 dq_load6(const Args &a, int mi, int64_t m, int kb, int half)
{
    DqItem6 it{{make_uint2(0, 0), make_uint2(0, 0), make_uint2(0, 0)}, 127u};
    const int64_t k0 = (int64_t)kb * BK + half * 32;
    if (m >= a.M || k0 >= a.K)
        return it;
    const uint8_t *cp = a.codes[mi] + m * (a.K / 8 * 6) + k0 / 4 * 3;
#pragma unroll
    for (int i = 0; i < 3; ++i)
        it.code[i] = ldg_stream_v2(cp + 8 * i);
    it.scl = __ldg(a.scales[mi] + m * (a.K / 128) + k0 / 128);
    return it;
}

NVFP4_DEVINL void fail(const Args &a, uint32_t code)
{
    atomicExch(a.err, code);
}

// FMT 0: NVFP4 weights; FMT 1: FP6 E2M3 weights (dequantised exactly to
// e2m3 * 2^(s-127), no tensor scale).
// Weight tiles by TMA (TMAC) need the code and scale tensor maps; without it
// they are unused.
struct WeightMaps {
    CUtensorMap codes[2];
    CUtensorMap scales[2];
};

// TN: tokens per tile (MMA N), 256 or 192; the host picks it per call so that
// the grid fills the SMs' waves (the accumulation order does not depend on it).
template <int NW, bool ALIGNED, int FMT = 0, bool TMAC = false, int TN = BN, bool SPLIT = false>
__global__ void __launch_bounds__(TMAC ? kThreadsTma : kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ WeightMaps wmaps, Args a)
{
    using C = Cfg<NW, TMAC, FMT, TN>;
    constexpr int kBBytes = C::kBBytes;
    using Item = typename std::conditional<FMT == 0, DqItem, DqItem6>::type;
    constexpr int S = C::kStages;
    constexpr int SC = C::kSc;
    constexpr int kCBytes = C::kCBytes;
    constexpr int kCRow = code_row_bytes<FMT>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool TA = C::kTA;
    uint8_t *sa = smem;                                  // [S][NW][kABytes] (not TA)
    uint8_t *sb = smem + (TA ? 0 : (size_t)S * NW * kABytes);  // [S][kBBytes]
    uint8_t *sc_ring = sb + (size_t)S * kBBytes;         // [SC][NW][kCBytes]      (TMAC)
    uint8_t *ss_ring = sc_ring + (size_t)SC * NW * kCBytes;  // [2][NW][kSBytes] (TMAC)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sb + (size_t)S * kBBytes + C::kRingBytes);
    uint64_t *full_a = bars, *full_b = bars + S, *empty = bars + 2 * S, *tmem_full = bars + 3 * S;
    uint64_t *cfull = bars + 3 * S + 1, *cempty = cfull + SC, *sfull = cempty + SC, *sempty = sfull + 2;
    uint64_t *tmem_empty = sempty + 2;  // split mode: segment 0's accumulator has been read
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmem_empty + 1);
    int *last_s = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The CTA's k blocks: one whole tile (raster order: the host picks the
    // raster so that the operand re-read across the grid stays resident in
    // L2), or in split mode one or two segments of its unit range.  Stage i of
    // the CTA runs k block kb_of(i) of segment seg_of(i); ring positions follow i.
    static_assert(!SPLIT || (NW == 1 && TMAC && FMT == 0), "split mode: one NVFP4 matrix, A in tensor memory");
    const Segs sgs = cta_segments<TN, SPLIT>(a, blockIdx.x, gridDim.x);
    const int64_t m0 = sgs.m0_a;
    const int num_kb = SPLIT ? sgs.nkb_a + (sgs.n > 1 ? sgs.nkb_b : 0) : a.num_kb;
    auto in_b = [&](int i) -> bool { return SPLIT && sgs.n > 1 && i >= sgs.nkb_a; };
    auto kb_of = [&](int i) -> int { return in_b(i) ? sgs.kb0_b + (i - sgs.nkb_a) : sgs.kb0_a + i; };
    auto m0_of = [&](int i) -> int64_t { return in_b(i) ? sgs.m0_b : sgs.m0_a; };
    auto n0_of = [&](int i) -> int { return in_b(i) ? sgs.n0_b : sgs.n0_a; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(&full_a[s], kDqWarps);
            tc::mbar_init(&full_b[s], 1);
            tc::mbar_init(&empty[s], C::kIssue);
        }
        tc::mbar_init(tmem_full, C::kIssue);
        tc::mbar_init(tmem_empty, kDqWarps);
        if (TMAC) {
            for (int c = 0; c < SC; ++c) {
                tc::mbar_init(&cfull[c], 1);
                tc::mbar_init(&cempty[c], kDqWarps);
            }
            for (int c = 0; c < 2; ++c) {
                tc::mbar_init(&sfull[c], 1);
                tc::mbar_init(&sempty[c], kDqWarps);
            }
        }
        tc::fence_mbar_init();
        tc::prefetch_tensormap(&tmap_x);
    }
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, C::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer (x tiles) ----------------
        if (lane == 0) {
            for (int kb = 0; kb < num_kb; ++kb) {
                const int s = kb % S;
                const uint32_t ph = (kb / S) & 1;
                if (!tc::mbar_wait(&empty[s], ph ^ 1)) {
                    fail(a, 1);
                    break;
                }
                tc::mbar_arrive_expect_tx(&full_b[s], kBBytes);
                tc::tma_load_2d(sb + (size_t)s * kBBytes, &tmap_x, &full_b[s], kb_of(kb) * BK, n0_of(kb));
            }
        }
    } else if (warp < kFirstDqWarp) {
        // ---------------- MMA issuers (warps 1, 2) ----------------
        // A thread spends longer issuing one M=128, N=256 MMA than the tensor
        // core takes to run it, so two threads issue: for the gate/up pair
        // issuer q owns matrix q; for one matrix issuer q takes the K steps
        // 2q, 2q+1 of every stage into accumulator q (added in the epilogue).
        if (TA && lane == 0 && warp == 1) {
            // one issuer, one accumulator, A from tensor memory
            constexpr uint32_t idesc = tc::idesc_bf16(BM, TN);
            for (int kb = 0; kb < num_kb; ++kb) {
                const bool seg_start = kb == 0 || (SPLIT && sgs.n > 1 && kb == sgs.nkb_a);
                if (SPLIT && kb > 0 && seg_start) {
                    // split mode: segment 0 is complete; its accumulator must be
                    // read by the epilogue before segment 1 overwrites it
                    tc::mma_commit(tmem_full);
                    if (!tc::mbar_wait(tmem_empty, 0)) {
                        fail(a, 8);
                        break;
                    }
                    tc::fence_after_sync();
                }
                const int s = kb % S;
                const uint32_t ph = (kb / S) & 1;
                if (!tc::mbar_wait(&full_a[s], ph) || !tc::mbar_wait(&full_b[s], ph)) {
                    fail(a, 2);
                    break;
                }
                tc::fence_after_sync();
                const uint64_t bdesc = tc::smem_desc_sw128(sb + (size_t)s * kBBytes);
                const uint32_t acol = tmem_base + C::kAcol0 + s * (BK / 2);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    tc::mma_f16_ts(tmem_base, acol + 8 * k, bdesc + 2 * k, idesc, (!seg_start || k > 0) ? 1u : 0u);
                tc::mma_commit(&empty[s]);
            }
            tc::mma_commit(tmem_full);
        } else if (!TA && lane == 0) {
            const int q = warp - 1;
            constexpr uint32_t idesc = tc::idesc_bf16(BM, TN);
            bool ok = true;
            for (int kb = 0; kb < num_kb && ok; ++kb) {
                const int s = kb % S;
                const uint32_t ph = (kb / S) & 1;
                if (!tc::mbar_wait(&full_a[s], ph) || !tc::mbar_wait(&full_b[s], ph)) {
                    fail(a, 2);
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint64_t bdesc = tc::smem_desc_sw128(sb + (size_t)s * kBBytes);
                if (NW == 2) {
                    const uint64_t adesc = tc::smem_desc_sw128(sa + ((size_t)s * NW + q) * kABytes);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc::mma_bf16_ss(tmem_base + q * TN, adesc + 2 * k, bdesc + 2 * k, idesc,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                } else {
                    const uint64_t adesc = tc::smem_desc_sw128(sa + (size_t)s * kABytes);
#pragma unroll
                    for (int k = 2 * q; k < 2 * q + 2; ++k)
                        tc::mma_bf16_ss(tmem_base + q * TN, adesc + 2 * k, bdesc + 2 * k, idesc,
                                        (kb > 0 || k > 2 * q) ? 1u : 0u);
                }
                tc::mma_commit(&empty[s]);
            }
            tc::mma_commit(tmem_full);
        }
    } else if (TMAC && warp == kCodeWarp) {
        // ---------------- weight code / scale TMA producer ----------------
        // Codes: one [128 rows][32 B] box per matrix and stage into a ring of
        // SC stages.  Scales: one [128 rows][16 B] box per matrix and group of
        // four stages into a ring of two groups.  Rows past M read as zeros.
        if (lane == 0) {
            for (int mi = 0; mi < NW; ++mi) {
                tc::prefetch_tensormap(&wmaps.codes[mi]);
                if (FMT == 0)
                    tc::prefetch_tensormap(&wmaps.scales[mi]);
            }
            for (int kb = 0; kb < num_kb; ++kb) {
                if (FMT == 0 && (kb & 3) == 0) {
                    const int sg = kb >> 2, ss = sg & 1;
                    if (!tc::mbar_wait(&sempty[ss], ((uint32_t)(sg >> 1) & 1) ^ 1)) {
                        fail(a, 6);
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&sfull[ss], NW * kSBytes);
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi)
                        tc::tma_load_2d(ss_ring + ((size_t)ss * NW + mi) * kSBytes, &wmaps.scales[mi], &sfull[ss],
                                        (kb_of(kb) >> 2) * 16, (int)m0_of(kb));
                }
                const int c = kb % SC;
                if (!tc::mbar_wait(&cempty[c], ((uint32_t)(kb / SC) & 1) ^ 1)) {
                    fail(a, 7);
                    break;
                }
                tc::mbar_arrive_expect_tx(&cfull[c], NW * kCBytes);
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    tc::tma_load_2d(sc_ring + ((size_t)c * NW + mi) * kCBytes, &wmaps.codes[mi], &cfull[c],
                                    kb_of(kb) * kCRow, (int)m0_of(kb));
            }
        }
    } else {
        // ---------------- dequantise producers ----------------
        const int dq = threadIdx.x - kFirstDqWarp * 32;  // 0..255
        // TA: a warp may write only its own quarter of the tensor-memory lanes
        const int row = TA ? 32 * (warp & 3) + lane : (dq & (BM - 1));  // 0..127
        const int half = dq >> 7;                  // which 32 k of the 64-k stage
        const int64_t m = m0 + row;
        bool ok = true;
        // TA: the dequantised 32 k of this row (four 8-k chunks, 16 columns)
        // for stage s go to tensor memory.
        auto put_a_tmem = [&](int s, const uint4 (&v)[4]) {
            const uint32_t w[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                                    v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
            tc::tmem_st_32x32b_x16(tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + C::kAcol0 + s * (BK / 2) +
                                       half * 16,
                                   w);
        };
        // Hand stage s to the MMA: proxy fence for shared memory, or the
        // tensor-memory store wait.
        auto publish_a = [&](int s) {
            if constexpr (TA) {
                tc::tmem_st_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(&full_a[s]);
            } else {
                // every thread orders its own shared-memory writes before the
                // async proxy; the warp then arrives once
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(&full_a[s]);
            }
        };
        // Epilogue of segment seg: TMEM -> registers -> global.  A whole tile
        // is stored directly; a split segment stores its raw fp32 accumulators
        // ([token][row] in the CTA's slot) and the last CTA of the tile adds
        // every contributor's slot in CTA order.
        auto finish_split = [&](int seg) {
            const int dq = threadIdx.x - kFirstDqWarp * 32;  // 0..255
            tc::named_bar_sync(1, kDqWarps * 32);             // every partial store of this CTA is done
            const int64_t G = gridDim.x;
            const int64_t t = seg ? sgs.tile_b : sgs.tile_a;
            const int64_t b_lo = split_cta_of(t * a.kq, a.units, G);
            const int64_t b_hi = split_cta_of((t + 1) * a.kq - 1, a.units, G);
            if (dq == 0) {
                // release: this CTA's partial (ordered by the barrier); acquire: the others'
                uint32_t old;
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.counters + t) : "memory");
                *last_s = old == (uint32_t)(b_hi - b_lo);
                if (*last_s)
                    a.counters[t] = 0;
            }
            tc::named_bar_sync(1, kDqWarps * 32);
            if (!*last_s)
                return;
            // thread: rows 4 rq .. 4 rq + 3 (one 16-byte load per contributor and
            // token), token columns cg, cg + 8, ...; contributors added in CTA order
            const int rq = dq & 31, cg = dq >> 5;
            const int64_t mq = (seg ? sgs.m0_b : sgs.m0_a) + 4 * rq;
            const int64_t sn0 = seg ? sgs.n0_b : sgs.n0_a;
            const float tsv = FMT == 0 ? __ldg(a.ts[0]) * 256.0f : 1.0f;
            const int nc = (int)(b_hi - b_lo) + 1;
            const float *src[4];
            for (int c = 0; c < 4; ++c) {
                const int64_t bb = b_lo + (c < nc ? c : nc - 1);
                src[c] = a.partial + (size_t)(2 * bb + (t - (bb * a.units / G) / a.kq)) * TN * BM + 4 * rq;
            }
#pragma unroll 2
            for (int col = cg; col < TN; col += 8) {
                const int64_t n = sn0 + col;
                if (n >= a.N)
                    break;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c0 = 0; c0 < nc; c0 += 4) {
                    float4 v[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float *p = c0 == 0 ? src[c] : a.partial + (size_t)(2 * (b_lo + c0 + c) +
                                            (t - ((b_lo + c0 + c) * a.units / G) / a.kq)) * TN * BM + 4 * rq;
                        v[c] = (c0 + c < nc) ? __ldcg(reinterpret_cast<const float4 *>(p + (size_t)col * BM))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (c0 + c < nc) {
                            acc.x += v[c].x;
                            acc.y += v[c].y;
                            acc.z += v[c].z;
                            acc.w += v[c].w;
                        }
                }
                const float r4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int64_t m = mq + e;
                    if (m < a.M) {
                        const float vv = r4[e] * tsv;
                        const int64_t idx = n * a.M + m;
                        if (a.out_bf16)
                            reinterpret_cast<uint16_t *>(a.y)[idx] = f32_to_bf16(vv);
                        else
                            reinterpret_cast<float *>(a.y)[idx] = vv;
                    }
                }
            }
        };
        auto epilogue = [&](int seg) {
            bool have = tc::mbar_wait(tmem_full, (uint32_t)seg & 1);
            const bool split_seg = SPLIT && !(seg ? sgs.whole_b : sgs.whole_a);
            if (SPLIT)
                have = tc::bar_and(1, kDqWarps * 32, have);  // uniform: named barriers follow
            if (!have)
                fail(a, 4);
            tc::fence_after_sync();
            const int64_t sm0 = seg ? sgs.m0_b : sgs.m0_a;
            const int sn0 = seg ? sgs.n0_b : sgs.n0_a;
            if (have) {
                const int quarter = warp & 3;          // TMEM lanes this warp may access
                const int chalf = (warp - kFirstDqWarp) >> 2;  // which half of the TN token columns
                const int64_t mrow = sm0 + quarter * 32 + lane;
                float ts[NW];
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    ts[mi] = FMT == 0 ? __ldg(a.ts[mi]) * 256.0f : 1.0f;
                float *slot = a.partial + (size_t)(2 * blockIdx.x + seg) * TN * BM + quarter * 32 + lane;
                // TA: only column chunks holding at least one real token
                // (warp-uniform; a runtime bound also keeps this loop rolled)
#pragma unroll 1
                for (int cc = 0; cc < TN / 64 && (!TA || sn0 + chalf * (TN / 2) + cc * 32 < a.N); ++cc) {
                    const int col = chalf * (TN / 2) + cc * 32;
                    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + col;
                    // two accumulators: gate and up, or (one matrix) K steps 0-1 and 2-3
                    uint32_t r[2][32];
                    tc::tmem_ld_32x32b_x32(taddr, r[0]);
                    if (!TA)
                        tc::tmem_ld_32x32b_x32(taddr + TN, r[1]);
                    tc::tmem_ld_wait();
                    if (SPLIT && split_seg) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            slot[(size_t)(col + j) * BM] = __uint_as_float(r[0][j]);
                    } else if (mrow < a.M) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int64_t n = (int64_t)sn0 + col + j;
                            if (n < a.N) {
                                float v;
                                if (TA) {
                                    v = __uint_as_float(r[0][j]) * ts[0];
                                } else if (NW == 1) {
                                    v = (__uint_as_float(r[0][j]) + __uint_as_float(r[1][j])) * ts[0];
                                } else {
                                    const float gg = __uint_as_float(r[0][j]) * ts[0];
                                    const float uu = __uint_as_float(r[NW - 1][j]) * ts[NW - 1];
                                    v = __fdiv_rn(gg, 1.0f + expf(-gg)) * uu;
                                }
                                const int64_t idx = n * a.M + mrow;
                                if (a.out_bf16)
                                    reinterpret_cast<uint16_t *>(a.y)[idx] = f32_to_bf16(v);
                                else
                                    reinterpret_cast<float *>(a.y)[idx] = v;
                            }
                        }
                    }
                }
            }
            if (SPLIT && seg + 1 < sgs.n) {
                // segment 1 follows: hand the accumulator back to the MMA issuer
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(tmem_empty);
            }
            if constexpr (SPLIT) {
                if (split_seg && have)
                    finish_split(seg);
            }
        };
        bool epi0_done = false;
        if constexpr (TMAC && FMT == 1) {
            // FP6 codes from the TMA ring; the scale byte of a row (one per
            // 128 k = two stages) through a small register prefetch ring.
            const int64_t nblk = a.K / 128;
            auto scale_at = [&](int mi, int64_t blk) -> uint32_t {
                return (m < a.M && blk < nblk) ? (uint32_t)__ldg(a.scales[mi] + m * nblk + blk) : 127u;
            };
            uint32_t sring[4][NW];
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    sring[p][mi] = scale_at(mi, p);
            uint32_t scl[NW];
            for (int kb = 0; kb < num_kb; ++kb) {
                if ((kb & 1) == 0) {
                    const int blk = kb >> 1;
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        if ((blk & 3) == p) {
#pragma unroll
                            for (int mi = 0; mi < NW; ++mi) {
                                scl[mi] = sring[p][mi];
                                sring[p][mi] = scale_at(mi, blk + 4);
                            }
                        }
                }
                const int c = kb % SC;
                if (!tc::mbar_wait(&cfull[c], (uint32_t)(kb / SC) & 1)) {
                    fail(a, 5);
                    ok = false;
                    break;
                }
                uint2 cw[NW][3];
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
#pragma unroll
                    for (int i = 0; i < 3; ++i)
                        cw[mi][i] = *reinterpret_cast<const uint2 *>(sc_ring + ((size_t)c * NW + mi) * kCBytes +
                                                                     row * kCRow + half * 24 + 8 * i);
                const int s = kb % S;
                if (!tc::mbar_wait(&empty[s], ((uint32_t)(kb / S) & 1) ^ 1)) {
                    fail(a, 3);
                    ok = false;
                    break;
                }
                if (TA)
                    tc::fence_after_sync();  // the MMAs that read this A stage are complete
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
                    const Fp6Mult mult = fp6_mult(scl[mi]);
                    if constexpr (TA) {
                        uint4 v[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            v[q] = fp6_group(cw[mi], q, mult);
                        put_a_tmem(s, v);
                    } else {
                        uint8_t *arow = sa + ((size_t)s * NW + mi) * kABytes + row * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 v = fp6_group(cw[mi], q, mult);
                            const int chunk = half * 4 + q;
                            *reinterpret_cast<uint4 *>(arow + ((chunk ^ (row & 7)) << 4)) = v;
                        }
                    }
                }
                publish_a(s);
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(&cempty[c]);
            }
        }
        if constexpr (TMAC && FMT == 0) {
            // Codes and scales from the TMA rings; a warp releases a ring slot
            // once its lanes have turned the slot's bytes into bf16 tiles.
            for (int kb = 0; kb < num_kb; ++kb) {
                if (SPLIT && sgs.n > 1 && kb == sgs.nkb_a) {  // split mode: segment 0 is done
                    epilogue(0);
                    epi0_done = true;
                }
                const int c = kb % SC;
                const int ss = (kb >> 2) & 1;
                if (!tc::mbar_wait(&cfull[c], (uint32_t)(kb / SC) & 1) ||
                    ((kb & 3) == 0 && !tc::mbar_wait(&sfull[ss], (uint32_t)(kb >> 3) & 1))) {
                    fail(a, 5);
                    ok = false;
                    break;
                }
                DqItem cur[NW];
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
                    cur[mi].code = *reinterpret_cast<const uint4 *>(sc_ring + ((size_t)c * NW + mi) * kCBytes +
                                                                    row * kCRow + half * 16);
                    cur[mi].scl = *reinterpret_cast<const uint16_t *>(ss_ring + ((size_t)ss * NW + mi) * kSBytes +
                                                                      row * 16 + (kb & 3) * 4 + half * 2);
                }
                const int s = kb % S;
                if (!tc::mbar_wait(&empty[s], ((uint32_t)(kb / S) & 1) ^ 1)) {
                    fail(a, 3);
                    ok = false;
                    break;
                }
                if (TA)
                    tc::fence_after_sync();  // the MMAs that read this A stage are complete
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
                    const uint32_t mlo = scale_mult_bf16(cur[mi].scl);
                    const uint32_t mhi = scale_mult_bf16(cur[mi].scl >> 8);
                    const uint32_t words[4] = {cur[mi].code.x, cur[mi].code.y, cur[mi].code.z, cur[mi].code.w};
                    if constexpr (TA) {
                        uint4 v[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            v[q] = dequant_word_natural(words[q], q < 2 ? mlo : mhi);
                        put_a_tmem(s, v);
                    } else {
                        uint8_t *arow = sa + ((size_t)s * NW + mi) * kABytes + row * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 v = dequant_word_natural(words[q], q < 2 ? mlo : mhi);
                            const int chunk = half * 4 + q;
                            *reinterpret_cast<uint4 *>(arow + ((chunk ^ (row & 7)) << 4)) = v;
                        }
                    }
                }
                publish_a(s);
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&cempty[c]);
                    if ((kb & 3) == 3)
                        tc::mbar_arrive(&sempty[ss]);
                }
            }
        }
        auto load = [&](int mi, int kb) -> Item {
            if constexpr (FMT == 0)
                return dq_load<ALIGNED>(a, mi, m, kb, half);
            else
                return dq_load6(a, mi, m, kb, half);
        };
        Item ring[C::kPf][NW];
        if (!TMAC) {
#pragma unroll
            for (int p = 0; p < C::kPf; ++p)
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    ring[p][mi] = load(mi, p < num_kb ? p : num_kb);
        }
        for (int kb0 = 0; !TMAC && kb0 < num_kb && ok; kb0 += C::kPf) {
#pragma unroll
            for (int p = 0; p < C::kPf; ++p) {
                const int kb = kb0 + p;
                if (kb >= num_kb || !ok)
                    break;
                Item cur[NW];
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
                    cur[mi] = ring[p][mi];
                    if (kb + C::kPf < num_kb)
                        ring[p][mi] = load(mi, kb + C::kPf);
                }
                const int s = kb % S;
                const uint32_t ph = (kb / S) & 1;
                if (!tc::mbar_wait(&empty[s], ph ^ 1)) {
                    fail(a, 3);
                    ok = false;
                    break;
                }
#pragma unroll
                for (int mi = 0; mi < NW; ++mi) {
                    uint8_t *arow = sa + ((size_t)s * NW + mi) * kABytes + row * 128;
                    if constexpr (FMT == 0) {
                        const uint32_t mlo = scale_mult_bf16(cur[mi].scl);
                        const uint32_t mhi = scale_mult_bf16(cur[mi].scl >> 8);
                        const uint32_t words[4] = {cur[mi].code.x, cur[mi].code.y, cur[mi].code.z,
                                                   cur[mi].code.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 v = dequant_word_natural(words[q], q < 2 ? mlo : mhi);
                            const int chunk = half * 4 + q;
                            *reinterpret_cast<uint4 *>(arow + ((chunk ^ (row & 7)) << 4)) = v;
                        }
                    } else {
                        const Fp6Mult mult = fp6_mult(cur[mi].scl);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 v = fp6_group(cur[mi].code, q, mult);
                            const int chunk = half * 4 + q;
                            *reinterpret_cast<uint4 *>(arow + ((chunk ^ (row & 7)) << 4)) = v;
                        }
                    }
                }
                publish_a(s);
            }
        }

        if (SPLIT && sgs.n > 1 && !epi0_done)
            epilogue(0);
        if (!SPLIT || sgs.n > 0)
            epilogue(SPLIT ? sgs.n - 1 : 0);
    }

    // Lane 0 of warps 0 and 1 ran the producer / MMA loops alone: reconverge
    // each warp first, so the block-wide barrier below really waits for every
    // thread (a partially arrived warp would otherwise count as arrived).
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, C::kTmemCols);
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

template <int NW, bool ALIGNED, int FMT = 0, bool TMAC = false, int TN = BN, bool SPLIT = false>
cudaError_t launch_t(const CUtensorMap &map, const WeightMaps &wm, const Args &a, cudaStream_t stream)
{
    using C = Cfg<NW, TMAC, FMT, TN>;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_errs[kMaxDevices];
    const cudaError_t attr_err = once_per_device(once, attr_errs, [] {
        return cudaFuncSetAttribute(prefill_kernel<NW, ALIGNED, FMT, TMAC, TN, SPLIT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    dim3 grid((unsigned)a.grid);
    prefill_kernel<NW, ALIGNED, FMT, TMAC, TN, SPLIT>
        <<<grid, TMAC ? kThreadsTma : kThreads, C::kSmemBytes, stream>>>(map, wm, a);
    return cudaGetLastError();
}

// Token tile for a TMA-fed launch: 192 instead of 256 when that fills the
// SMs' waves better.  A CTA's time is modelled as a part that does not scale
// with the tile (dequantisation, prologue, epilogue: ~1/4) plus the MMA part
// proportional to TN.
inline int pick_token_tile(int64_t N, int64_t row_tiles, int num_sms)
{
    auto cost = [&](int tn) {
        const int64_t ctas = row_tiles * ((N + tn - 1) / tn);
        const int64_t waves = (ctas + num_sms - 1) / num_sms;
        return (double)waves * (0.25 + tn / 256.0);
    };
    return cost(192) < cost(256) ? 192 : 256;
}

// 2-D uint8 tensor map over rows of `pitch` bytes (box: 128 rows x box_bytes).
static bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *m, const uint8_t *base,
                        int64_t pitch, int64_t rows, uint32_t box_bytes)
{
    const cuuint64_t dims[2] = {(cuuint64_t)pitch, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch};
    const cuuint32_t box[2] = {box_bytes, (cuuint32_t)BM};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pf

// Split mode (see Args): one NVFP4 matrix with K % 256 == 0 whose 256-token
// tiles would fill less than three quarters of the SMs.  Its workspace holds
// the tile counters and two partial slots per CTA; the size bound holds for
// any device with up to kMaxSplitCtas SMs, so it depends on the shape alone.
constexpr int kMaxSplitCtas = 256;
constexpr size_t kSplitCounterBytes = 1024;  // one u32 per tile (< kMaxSplitCtas tiles)

static bool split_possible(int64_t N, int64_t M, int64_t K, int n_weights)
{
    const int64_t tiles = ((M + pf::BM - 1) / pf::BM) * ((N + pf::BN - 1) / pf::BN);
    return n_weights == 1 && K % 256 == 0 && tiles * 4 < (int64_t)kMaxSplitCtas * 3;
}

static bool use_split(int64_t N, int64_t M, int64_t K, int n_weights, int num_sms)
{
    const int64_t tiles = ((M + pf::BM - 1) / pf::BM) * ((N + pf::BN - 1) / pf::BN);
    return split_possible(N, M, K, n_weights) && num_sms <= kMaxSplitCtas && tiles * 4 < (int64_t)num_sms * 3;
}

size_t prefill_workspace_bytes(int64_t N, int64_t M, int64_t K, int n_weights)
{
    // the device status word at kStatusWordOffset; split mode adds its counters and partials
    if (!split_possible(N, M, K, n_weights))
        return 256;
    return 256 + kSplitCounterBytes + (size_t)2 * kMaxSplitCtas * pf::BN * pf::BM * sizeof(float);
}

static cudaError_t prefill_impl(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                                const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                                int out_bf16, void *workspace, int fmt, int num_sms, cudaStream_t stream)
{
    auto encode = pf::encode_fn();
    if (!encode)
        return cudaErrorNotSupported;
    const bool tma_weights = fmt == 1 || K % 256 == 0;
    const int64_t row_tiles = (M + pf::BM - 1) / pf::BM;
    const bool split = fmt == 0 && use_split(N, M, K, n_weights, num_sms);
    const int tn = split ? pf::BN : tma_weights ? pf::pick_token_tile(N, row_tiles, num_sms) : pf::BN;
    const int64_t token_tiles = (N + tn - 1) / tn;
    if (row_tiles * token_tiles > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {pf::BK, (cuuint32_t)tn};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    pf::Args a{};
    for (int i = 0; i < 2; ++i) {
        const int s = i < n_weights ? i : 0;
        a.codes[i] = codes[s];
        a.scales[i] = scales[s];
        a.ts[i] = ts ? ts[s] : nullptr;
    }
    a.y = y;
    a.out_bf16 = out_bf16;
    a.N = N;
    a.M = M;
    a.K = K;
    a.num_kb = (int)((K + pf::BK - 1) / pf::BK);
    a.err = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(workspace) + kStatusWordOffset);
    a.row_tiles = (int)row_tiles;
    a.token_tiles = (int)token_tiles;
    a.split = split ? 1 : 0;
    if (split) {
        uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
        a.kq = a.num_kb / 4;
        a.units = row_tiles * token_tiles * a.kq;
        a.counters = reinterpret_cast<uint32_t *>(ws + 256);
        a.partial = reinterpret_cast<float *>(ws + 256 + kSplitCounterBytes);
        // at most one CTA per unit: every CTA's range is non-empty, so a
        // tile's contributors are the contiguous CTAs b_lo .. b_hi
        a.grid = (int)std::min<int64_t>(num_sms, a.units);
        const cudaError_t me = cudaMemsetAsync(a.counters, 0, (size_t)row_tiles * token_tiles * 4, stream);
        if (me != cudaSuccess)
            return me;
    } else {
        a.grid = (int)(row_tiles * token_tiles);
    }
    {
        // Which operand stays in L2 for the whole grid: if the activations fit,
        // token tiles vary fastest (group of 1 row tile: x is read from HBM
        // once, each weight row tile once per wave); else if the weights fit,
        // row tiles vary fastest (one group of all rows); else groups whose
        // weights fit.  (Keeping the 50 MB of weights resident instead of the
        // 71 MB of activations for the 27B down projection at N = 2048 was
        // measured slower: 0.50 against 0.54 of the bf16 peak.)
        constexpr double kL2Budget = 110e6;  // of the 129 MB L2
        const double x_bytes = (double)N * (double)K * 2.0;
        const double w_tile = (double)pf::BM * (double)K * (fmt == 1 ? 0.7578125 : 0.5625) * n_weights;
        int g;
        if (x_bytes <= kL2Budget)
            g = 1;
        else if (w_tile * (double)row_tiles <= kL2Budget)
            g = (int)row_tiles;
        else
            g = (int)(kL2Budget / w_tile);
        a.group = g < 1 ? 1 : (g > (int)row_tiles ? (int)row_tiles : g);
    }
    pf::WeightMaps wm;
    memset(&wm, 0, sizeof(wm));
    if (fmt == 1) {
        // FP6 codes by TMA: row pitch 3K/4 is a multiple of 16 bytes (K % 128 == 0)
        for (int i = 0; i < n_weights; ++i)
            if (!pf::encode_rows(encode, &wm.codes[i], codes[i], K / 4 * 3, M, pf::code_row_bytes<1>()))
                return cudaErrorInvalidValue;
        if (tn == 192)
            return n_weights == 1 ? pf::launch_t<1, true, 1, true, 192>(map, wm, a, stream)
                                  : pf::launch_t<2, true, 1, true, 192>(map, wm, a, stream);
        return n_weights == 1 ? pf::launch_t<1, true, 1, true>(map, wm, a, stream)
                              : pf::launch_t<2, true, 1, true>(map, wm, a, stream);
    }
    if (K % 256 == 0) {
        // Codes and scales by TMA: row pitches K/2 and K/16 are multiples of 16 bytes.
        for (int i = 0; i < n_weights; ++i)
            if (!pf::encode_rows(encode, &wm.codes[i], codes[i], K / 2, M, pf::BK / 2) ||
                !pf::encode_rows(encode, &wm.scales[i], scales[i], K / 16, M, 16))
                return cudaErrorInvalidValue;
        if (split)
            return pf::launch_t<1, true, 0, true, 256, true>(map, wm, a, stream);
        if (tn == 192)
            return n_weights == 1 ? pf::launch_t<1, true, 0, true, 192>(map, wm, a, stream)
                                  : pf::launch_t<2, true, 0, true, 192>(map, wm, a, stream);
        return n_weights == 1 ? pf::launch_t<1, true, 0, true>(map, wm, a, stream)
                              : pf::launch_t<2, true, 0, true>(map, wm, a, stream);
    }
    const bool aligned = K % 32 == 0;
    if (n_weights == 1)
        return aligned ? pf::launch_t<1, true>(map, wm, a, stream) : pf::launch_t<1, false>(map, wm, a, stream);
    return aligned ? pf::launch_t<2, true>(map, wm, a, stream) : pf::launch_t<2, false>(map, wm, a, stream);
}

cudaError_t launch_prefill(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                           const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                           int out_bf16, void *workspace, int num_sms, cudaStream_t stream)
{
    return prefill_impl(x, N, M, K, codes, scales, ts, n_weights, y, out_bf16, workspace, 0, num_sms, stream);
}

cudaError_t launch_prefill_fp6(const uint16_t *x, int64_t N, int64_t M, int64_t K, const uint8_t *const *codes,
                               const uint8_t *const *scales, int n_weights, void *y, int out_bf16,
                               void *workspace, int num_sms, cudaStream_t stream)
{
    return prefill_impl(x, N, M, K, codes, scales, nullptr, n_weights, y, out_bf16, workspace, 1, num_sms, stream);
}

// Failure-path self-test: one thread waits, with the same bounded wait as the
// pipelines above, on a barrier that nothing arrives at.  When the wait gives
// up (tc::kWaitLimitNs of wall time) the kernel records kStatusSelftest in the
// status word, as a compute kernel records its own code, and returns; nothing
// faults and the context stays usable.
__global__ void wait_timeout_selftest_kernel(uint32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0)
        return;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    if (!tc::mbar_wait(&bar, 0))  // phase 0 never completes
        atomicExch(status, kStatusSelftest);
}

cudaError_t launch_wait_timeout_selftest(void *workspace, cudaStream_t stream)
{
    uint32_t *status = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(workspace) + kStatusWordOffset);
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace nvfp4
