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
constexpr int kMaxContrib = 64;       // split mode: CTAs sharing one tile, at most
constexpr int kRedCols = 16;          // split-mode reduction: token columns per work item
constexpr int kRedThreads = 256;      // its threads: rows 4 rq .. 4 rq + 3 of two columns each

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
    // Split mode (stream-K; one matrix, A in tensor memory): the tiles from
    // sk_base / kq on are cut into (tile, 256-k group) units, and CTA b takes
    // the b-th of sk_grid equal contiguous unit ranges: a partial tile at
    // each end of the range, whole tiles between.  A CTA stores the fp32
    // accumulators of a tile it shares as a partial; the reduction launch
    // that follows adds every shared tile's partials in CTA order.  The tiles
    // before sk_base / kq belong to a whole-tile launch that precedes this one
    // on the stream.
    int split;
    int grid;             // CTAs: one per tile, or (split mode) sk_grid
    int kq;               // 256-k groups per tile (num_kb / 4)
    int after_whole;      // split mode: a whole-tile launch precedes this one
    int64_t sk_base;      // first stream-K unit: (tiles of the whole-tile launch) * kq
    int64_t units;        // stream-K units
    int sk_grid;          // CTAs sharing them (<= units)
    float *partial;       // [2 * gridDim][TN][BM] raw fp32 accumulators: a CTA's first and last segment
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

// A CTA's walk over its k blocks.  Without split mode: one whole tile.  In
// split mode: its unit range [lo, hi), which crosses tiles (a partial tile at
// each end, whole tiles between).  Every role walks the same sequence of
// (segment, 64-k block) stages with its own cursor: an outer loop over
// segments, whose inner loop over the segment's k blocks is the whole-tile
// loop (the divisions of tile_coords run once per segment, not per stage).
struct SegCursor {
    int64_t tile;   // tile of the current segment
    int64_t hi;     // end of the CTA's unit range (absolute units)
    int kb;         // first 64-k block of the segment (within its tile)
    int kb_end;     // end of the segment (64-k blocks)
    int seg;        // segment number within the CTA
    int64_t m0;     // first weight row of the tile
    int n0;         // first token of the tile
    bool whole;     // the segment covers the whole K range of its tile
};

// First tile of stream-K CTA b's range.
NVFP4_DEVINL int64_t sk_first_tile(const Args &a, int64_t b)
{
    return (a.sk_base + b * a.units / a.sk_grid) / a.kq;
}

template <int TN>
NVFP4_DEVINL void seg_coords(const Args &a, SegCursor &c)
{
    int64_t rt, tt;
    tile_coords(a, c.tile, rt, tt);
    c.m0 = rt * BM;
    c.n0 = (int)(tt * TN);
}

template <int TN>
NVFP4_DEVINL void seg_enter(const Args &a, SegCursor &c, int64_t lo)
{
    c.tile = lo / a.kq;
    const int64_t base = c.tile * a.kq;
    const int64_t e = base + a.kq < c.hi ? base + a.kq : c.hi;
    c.kb = (int)(lo - base) * 4;
    c.kb_end = (int)(e - base) * 4;
    c.whole = lo == base && e == base + a.kq;
    seg_coords<TN>(a, c);
}

template <int TN, bool SPLIT>
NVFP4_DEVINL SegCursor cta_cursor(const Args &a, int64_t b, int &num_kb)
{
    SegCursor c{};
    if (!SPLIT) {
        c.tile = b;
        c.kb_end = a.num_kb;
        c.whole = true;
        num_kb = a.num_kb;
        seg_coords<TN>(a, c);
    } else {
        const int64_t lo = a.sk_base + b * a.units / a.sk_grid;
        c.hi = a.sk_base + (b + 1) * a.units / a.sk_grid;
        num_kb = (int)(c.hi - lo) * 4;
        seg_enter<TN>(a, c, lo);
    }
    return c;
}

// More segments follow the cursor's one.
NVFP4_DEVINL bool seg_more(const Args &a, const SegCursor &c) { return (c.tile + 1) * a.kq < c.hi; }

// Move to the start of the next segment (false if there is none).
template <int TN>
NVFP4_DEVINL bool seg_skip(const Args &a, SegCursor &c)
{
    if (!seg_more(a, c))
        return false;
    ++c.seg;
    seg_enter<TN>(a, c, (c.tile + 1) * a.kq);
    return true;
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
    static_assert(3 * S + 1 + 2 * SC + 4 + 1 <= 128, "barriers and TMEM slot in the 1024-byte barrier area");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The CTA's k blocks: one whole tile (raster order: the host picks the
    // raster so that the operand re-read across the grid stays resident in
    // L2), or in split mode the segments of its unit range.  Stage i of the
    // CTA runs the cursor's k block; ring positions follow i.
    static_assert(!SPLIT || (NW == 1 && TMAC && FMT == 0), "split mode: one NVFP4 matrix, A in tensor memory");
    int num_kb;
    const SegCursor c0 = cta_cursor<TN, SPLIT>(a, blockIdx.x, num_kb);
    const int64_t m0 = c0.m0;

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
    // A stream-K launch is a programmatic dependent launch, so the set-up
    // above overlaps the end of the kernel before it on the stream.  As the
    // call's first launch it reads and writes nothing global before that
    // kernel has completed; after whole tiles it reads nothing they write and
    // waits for them before it exits.  (Whole-tile launches are ordinary
    // ones: a wait in each of their CTAs cost 1-2 % over several waves.)
    // Only then may the launch after this one start: after whole tiles the
    // stream-K launch (it computes other tiles), after the stream-K launch
    // its reduction (which waits for this launch's completion before reading
    // anything).
    if (SPLIT && !a.after_whole)
        tc::griddep_wait();
    tc::griddep_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer (x tiles) ----------------
        if (lane == 0) {
            SegCursor cur = c0;
            int kb = 0;  // the CTA's stage: ring position
            bool ok = true;
            do {
                // the segment's k blocks kt (within its tile)
                const int k1 = SPLIT ? cur.kb_end : num_kb;
                for (int kt = SPLIT ? cur.kb : 0; kt < k1; ++kt, ++kb) {
                    const int s = kb % S;
                    const uint32_t ph = (kb / S) & 1;
                    if (!tc::mbar_wait(&empty[s], ph ^ 1)) {
                        fail(a, 1);
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&full_b[s], kBBytes);
                    tc::tma_load_2d(sb + (size_t)s * kBBytes, &tmap_x, &full_b[s], kt * BK, cur.n0);
                }
            } while (SPLIT && ok && seg_skip<TN>(a, cur));
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
            SegCursor cur = c0;
            int kb = 0;  // the CTA's stage: ring position
            bool ok = true;
            for (;;) {
                const int k0 = SPLIT ? cur.kb : 0, k1 = SPLIT ? cur.kb_end : num_kb;
                for (int kt = k0; kt < k1; ++kt, ++kb) {
                    const int s = kb % S;
                    const uint32_t ph = (kb / S) & 1;
                    if (!tc::mbar_wait(&full_a[s], ph) || !tc::mbar_wait(&full_b[s], ph)) {
                        fail(a, 2);
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint64_t bdesc = tc::smem_desc_sw128(sb + (size_t)s * kBBytes);
                    const uint32_t acol = tmem_base + C::kAcol0 + s * (BK / 2);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc::mma_f16_ts(tmem_base, acol + 8 * k, bdesc + 2 * k, idesc, (kt > k0 || k > 0) ? 1u : 0u);
                    tc::mma_commit(&empty[s]);
                }
                if (!SPLIT || !ok || !seg_skip<TN>(a, cur))
                    break;
                // split mode: the segment is complete; its accumulator must be
                // read by the epilogue before the next segment overwrites it
                tc::mma_commit(tmem_full);
                if (!tc::mbar_wait(tmem_empty, (uint32_t)(cur.seg - 1) & 1)) {
                    fail(a, 8);
                    break;
                }
                tc::fence_after_sync();
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
            SegCursor cur = c0;
            int kb = 0;  // the CTA's stage: ring position (segments are whole 4-stage groups)
            bool ok = true;
            do {
                const int m0c = (int)cur.m0;
                const int k1 = SPLIT ? cur.kb_end : num_kb;
                for (int kt = SPLIT ? cur.kb : 0; kt < k1; ++kt, ++kb) {
                    if (FMT == 0 && (kb & 3) == 0) {
                        const int sg = kb >> 2, ss = sg & 1;
                        if (!tc::mbar_wait(&sempty[ss], ((uint32_t)(sg >> 1) & 1) ^ 1)) {
                            fail(a, 6);
                            ok = false;
                            break;
                        }
                        tc::mbar_arrive_expect_tx(&sfull[ss], NW * kSBytes);
#pragma unroll
                        for (int mi = 0; mi < NW; ++mi)
                            tc::tma_load_2d(ss_ring + ((size_t)ss * NW + mi) * kSBytes, &wmaps.scales[mi],
                                            &sfull[ss], (kt >> 2) * 16, m0c);
                    }
                    const int c = kb % SC;
                    if (!tc::mbar_wait(&cempty[c], ((uint32_t)(kb / SC) & 1) ^ 1)) {
                        fail(a, 7);
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&cfull[c], NW * kCBytes);
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi)
                        tc::tma_load_2d(sc_ring + ((size_t)c * NW + mi) * kCBytes, &wmaps.codes[mi], &cfull[c],
                                        kt * kCRow, m0c);
                }
            } while (SPLIT && ok && seg_skip<TN>(a, cur));
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
        // ([token][row] in the CTA's slot) for the reduction launch.
        auto epilogue = [&](const SegCursor &sg) {
            const bool have = tc::mbar_wait(tmem_full, (uint32_t)sg.seg & 1);
            const bool split_seg = SPLIT && !sg.whole;
            if (!have)
                fail(a, 4);
            tc::fence_after_sync();
            const int64_t sm0 = sg.m0;
            const int sn0 = sg.n0;
            if (have) {
                const int quarter = warp & 3;          // TMEM lanes this warp may access
                const int chalf = (warp - kFirstDqWarp) >> 2;  // which half of the TN token columns
                const int64_t mrow = sm0 + quarter * 32 + lane;
                float ts[NW];
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    ts[mi] = FMT == 0 ? __ldg(a.ts[mi]) * 256.0f : 1.0f;
                // a partial segment is the first (slot 0) or last (slot 1) of the
                // CTA's stream-K range
                float *slot = a.partial +
                              (size_t)(2 * blockIdx.x + (SPLIT && sg.tile != sk_first_tile(a, blockIdx.x) ? 1 : 0)) *
                                  TN * BM +
                              quarter * 32 + lane;
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
            if (SPLIT && seg_more(a, sg)) {
                // another segment follows: hand the accumulator back to the MMA issuer
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(tmem_empty);
            }
        };
        SegCursor dcur = c0;  // the dequantisers' stage cursor
        if constexpr (TMAC && FMT == 1) {
            // FP6 codes from the TMA ring; the scale byte of a row (one per
            // 128 k = two stages) through a small register prefetch ring.
            const uint32_t fp6_ring_a = tc::smem_addr(sc_ring) + (uint32_t)(row * kCRow + half * 24);
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
                    for (int i = 0; i < 3; ++i)  // ld.shared from 32-bit shared addresses
                        cw[mi][i] = tc::lds64(fp6_ring_a + (uint32_t)((c * NW + mi) * kCBytes + 8 * i));
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
            // Stage kb is a ring position; in split mode the segments follow
            // one another, each ending with its epilogue.
            const uint32_t sc_ring_a = tc::smem_addr(sc_ring) + (uint32_t)(row * kCRow + half * 16);
            const uint32_t ss_ring_a = tc::smem_addr(ss_ring) + (uint32_t)(row * 16 + half * 2);
            int kb = 0;
            for (;;) {
                const int kend = kb + (SPLIT ? dcur.kb_end - dcur.kb : num_kb);
                for (; kb < kend; ++kb) {
                    const int c = kb % SC;
                    const int ss = (kb >> 2) & 1;
                    if (!tc::mbar_wait(&cfull[c], (uint32_t)(kb / SC) & 1) ||
                        ((kb & 3) == 0 && !tc::mbar_wait(&sfull[ss], (uint32_t)(kb >> 3) & 1))) {
                        fail(a, 5);
                        ok = false;
                        break;
                    }
                    // ld.shared from 32-bit shared addresses (a generic load
                    // waits on the long scoreboard)
                    DqItem cur[NW];
#pragma unroll
                    for (int mi = 0; mi < NW; ++mi) {
                        cur[mi].code = tc::lds128(sc_ring_a + (uint32_t)((c * NW + mi) * kCBytes));
                        cur[mi].scl = tc::lds16(ss_ring_a + (uint32_t)((ss * NW + mi) * kSBytes + (kb & 3) * 4));
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
                if (!SPLIT || !ok || !seg_more(a, dcur))
                    break;
                epilogue(dcur);
                seg_skip<TN>(a, dcur);
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

        // The last segment's epilogue.  After a failed wait the loop ends
        // early: the epilogues of the segments it did not reach still run
        // (their waits give up too), so that every dequantiser warp meets the
        // epilogues' named barriers the same number of times.
        do {
            epilogue(dcur);
        } while (SPLIT && seg_skip<TN>(a, dcur));
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
    // A stream-K launch after whole tiles overlaps them (it reads nothing
    // they write) and completes only after them, so that work ordered after
    // this call sees every tile.
    if (SPLIT && threadIdx.x == 0)
        tc::griddep_wait();
}

// Rows mq .. mq + 3 of token n of the output, from fp32 values.
NVFP4_DEVINL void store_rows4(const Args &a, int64_t n, int64_t mq, float4 v)
{
    const int64_t idx = n * a.M + mq;
    if ((a.M & 3) == 0 && mq + 3 < a.M) {  // 16- / 8-byte aligned, all in range
        if (a.out_bf16)
            *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(a.y) + idx) =
                make_uint2(f32_to_bf16(v.x) | ((uint32_t)f32_to_bf16(v.y) << 16),
                           f32_to_bf16(v.z) | ((uint32_t)f32_to_bf16(v.w) << 16));
        else
            *reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.y) + idx) = v;
    } else {
        const float r4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (mq + e < a.M) {
                if (a.out_bf16)
                    reinterpret_cast<uint16_t *>(a.y)[idx + e] = f32_to_bf16(r4[e]);
                else
                    reinterpret_cast<float *>(a.y)[idx + e] = r4[e];
            }
    }
}

// Split mode, second launch (programmatic dependent launch after the
// stream-K one): every tile that several CTAs shared is the sum of their
// fp32 partials, added in CTA order (fixed by the shape, so deterministic),
// times the tensor scale.  The work spreads over every SM: item (tile,
// kRedCols token columns); thread (rq, cs) adds rows 4 rq .. 4 rq + 3 of
// columns cs and cs + 8, four contributors per batch, so eight 16-byte loads
// are in flight per thread.  A tile that one CTA covered whole was stored by
// that CTA.
// Contributors of tile t: CTAs b_lo .. b_hi.  Every one after b_lo starts its
// range inside t, so t is its first tile and its partial is in slot 2 b;
// b_lo's is in slot 2 b_lo, or 2 b_lo + 1 (its last segment) if its range
// starts before t.  NARROW: the index arithmetic in 32 bits, which the host
// picks when every intermediate fits (a fraction of the cost of 64-bit
// divisions).  A contributor or tile outside the plan's ranges (impossible
// with the host's plan) records status 10 and skips the item.
template <bool NARROW>
__global__ void __launch_bounds__(kRedThreads, 4) split_reduce_kernel(Args a)
{
    using I = typename std::conditional<NARROW, uint32_t, int64_t>::type;
    // The next call's first launch may take the SMs as they free up: it waits
    // for this one's completion before any global access.
    tc::griddep_launch_dependents();
    tc::griddep_wait();  // the stream-K launch has completed: its partials are visible
    constexpr int kItemsPerTile = BN / kRedCols;
    const I units = (I)a.units, G = (I)a.sk_grid, kq = (I)a.kq, sk_base = (I)a.sk_base;
    const I group = (I)a.group, token_tiles = (I)a.token_tiles, row_tiles = (I)a.row_tiles;
    const I t0 = sk_base / kq;
    const int64_t items = a.units / a.kq * kItemsPerTile;
    const int rq = threadIdx.x & 31, cs = threadIdx.x >> 5;
    const float tsv = __ldg(a.ts[0]) * 256.0f;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const I t = t0 + (I)(it / kItemsPerTile);
        const int q = (int)(it % kItemsPerTile);
        // CTA b's range is [b units / G, (b + 1) units / G) (relative to
        // sk_base; G <= units, so none is empty): unit u lies in the range of
        // CTA ((u + 1) G - 1) / units
        const I b_lo = ((t * kq - sk_base + 1) * G - 1) / units;         // CTA of the tile's first unit
        const I b_hi = (((t + 1) * kq - sk_base) * G - 1) / units;       // and of its last
        const int nc = (int)(b_hi - b_lo) + 1;
        if (nc < 2)
            continue;
        const uint32_t f0 = (sk_base + b_lo * units / G) / kq != t ? 1u : 0u;
        // raster: groups of `group` row tiles, row tiles fastest inside a group
        const I per_group = group * token_tiles;
        const I gidx = t / per_group;
        const I first = gidx * group;
        const I rows = row_tiles - first < group ? row_tiles - first : group;
        const I in = t - gidx * per_group;
        const I rt = first + in % rows, tt = in / rows;
        if (nc > kMaxContrib || b_hi >= G || rt >= row_tiles || tt >= token_tiles) {
            if (threadIdx.x == 0)
                fail(a, 10);
            continue;
        }
        const int64_t mq = (int64_t)rt * BM + 4 * rq;
        const int64_t n0 = (int64_t)tt * BN;
        const int ncols = (int)(a.N - n0 < BN ? a.N - n0 : BN);
        const int col0 = q * kRedCols + cs;
        if (col0 >= ncols)
            continue;
        const float *base = a.partial + (size_t)(2 * (size_t)b_lo) * BN * BM + 4 * rq;
        float4 acc[2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
            acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < nc; c0 += 4) {
            float4 v[4][2];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int cc = c0 + c;
                const float *p = base + (size_t)(2 * cc + (cc == 0 ? f0 : 0u)) * BN * BM;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = col0 + 8 * j;
                    v[c][j] = (cc < nc && col < ncols)
                                  ? __ldcg(reinterpret_cast<const float4 *>(p + (size_t)col * BM))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (c0 + c < nc) {
                        acc[j].x += v[c][j].x;
                        acc[j].y += v[c][j].y;
                        acc[j].z += v[c][j].z;
                        acc[j].w += v[c][j].w;
                    }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = col0 + 8 * j;
            if (col < ncols)
                store_rows4(a, n0 + col, mq,
                            make_float4(acc[j].x * tsv, acc[j].y * tsv, acc[j].z * tsv, acc[j].w * tsv));
        }
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
    if (SPLIT) {
        // programmatic dependent launch: the CTAs start on SMs as the kernel
        // before them frees them (see the kernel for what waits for it)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(TMAC ? kThreadsTma : kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, prefill_kernel<NW, ALIGNED, FMT, TMAC, TN, SPLIT>, map, wm, a);
    }
    prefill_kernel<NW, ALIGNED, FMT, TMAC, TN, SPLIT>
        <<<grid, TMAC ? kThreadsTma : kThreads, C::kSmemBytes, stream>>>(map, wm, a);
    return cudaGetLastError();
}

// The split-mode reduction, programmatically dependent on the stream-K
// launch: its CTAs take SMs as the stream-K CTAs leave them and wait for that
// launch's completion before reading a partial.  Four CTAs fit on an SM;
// the grid stops at eight CTAs per SM and takes any further items in its
// grid-stride loop.
inline cudaError_t launch_split_reduce(const Args &a, int num_sms, cudaStream_t stream)
{
    const int64_t items = a.units / a.kq * (BN / kRedCols);
    const int64_t cap = (int64_t)num_sms * 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(items < cap ? items : cap));
    cfg.blockDim = dim3(kRedThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // 32-bit index arithmetic when every intermediate fits: (u + 1) * G for
    // a unit u, b * units for a CTA b < G, and the unit numbers themselves
    const uint64_t lim = uint64_t(1) << 32;
    const bool narrow = (uint64_t)(a.units + 1) * (uint64_t)a.sk_grid < lim &&
                        (uint64_t)(a.sk_base + a.units) < lim;
    if (narrow)
        return cudaLaunchKernelEx(&cfg, split_reduce_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, split_reduce_kernel<false>, a);
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

// Split mode (see Args): one NVFP4 matrix with K % 256 == 0.  Its workspace
// holds two partial slots per CTA; the grid has at most
// min(kMaxSplitCtas, units) CTAs, so the size depends on the shape alone.
constexpr int kMaxSplitCtas = 256;

static bool split_possible(int64_t K, int n_weights, int fmt) { return fmt == 0 && n_weights == 1 && K % 256 == 0; }

static int64_t split_units(int64_t N, int64_t M, int64_t K)
{
    return ((M + pf::BM - 1) / pf::BM) * ((N + pf::BN - 1) / pf::BN) * (K / 256);
}

// How a split call shares its work (see Args).
struct SplitPlan {
    int64_t dp_waves;  // waves of whole tiles in a launch of their own, before the stream-K launch
    int64_t units;     // stream-K units after them
    int64_t sk_grid;   // CTAs sharing the stream-K units
};

// Of the 129 MB L2, what a launch's operands may take and still be read from
// HBM about once.
constexpr double kL2Budget = 110e6;

// The split for a single NVFP4 matrix, and whether it beats whole tiles
// alone.  Two forms:
//   - operands resident in L2 (x and the weights fit): every unit is shared
//     out, each CTA an equal contiguous range (up to two partial tiles);
//     CTAs at different k of a tile cost nothing extra when nothing is
//     evicted;
//   - otherwise the full waves run as whole tiles (a launch of their own)
//     and the R = tiles mod SMs tiles left split into f equal k slices, one
//     CTA each: slice j of every tile starts at the same k, so the CTAs
//     sharing a token tile still read the same activations at the same
//     time, as in a wave.
// Time in 64-k stages of a 256-token tile: a tile of TN tokens takes
// num_kb * (0.25 + TN / 256) / 1.25 stages plus kFixed (prologue, pipeline
// fill, epilogue); whole tiles run in waves of num_sms CTAs.  A split CTA
// pays kFixed for each of up to three segments, and the reduction launch
// reads every 128 KB partial once, spread over the SMs: kRedFixed stages
// plus 0.05 * 152 / SMs stages per partial.  A tile has at most
// kMaxContrib contributors.
static bool split_plan(int64_t N, int64_t M, int64_t K, int n_weights, int fmt, int num_sms, SplitPlan *sp)
{
    if (!split_possible(K, n_weights, fmt) || num_sms > kMaxSplitCtas)
        return false;
    constexpr double kFixed = 10.0, kRedFixed = 6.0;
    const double red_per_partial = 0.05 * 152.0 / (double)num_sms;
    const int64_t row_tiles = (M + pf::BM - 1) / pf::BM;
    const int64_t kq = K / 256;
    const double num_kb = (double)(K / pf::BK);
    auto whole = [&](int tn) {
        const int64_t ctas = row_tiles * ((N + tn - 1) / tn);
        const int64_t waves = (ctas + num_sms - 1) / num_sms;
        return (double)waves * (num_kb * (0.25 + tn / 256.0) / 1.25 + kFixed);
    };
    const double best_whole = whole(192) < whole(256) ? whole(192) : whole(256);
    const int64_t tiles = row_tiles * ((N + pf::BN - 1) / pf::BN);
    const double operand_bytes = (double)N * (double)K * 2.0 + (double)M * (double)K * 0.5625;
    double t_split;
    if (operand_bytes <= kL2Budget) {
        sp->dp_waves = 0;
        sp->units = tiles * kq;
        int64_t G = sp->units < num_sms ? sp->units : num_sms;
        // ranges of at least units / G units: a tile meets at most
        // ceil(kq / (units / G)) + 1 of them
        auto contributors = [&](int64_t g) {
            const int64_t u = sp->units / g;
            return (kq + u - 1) / u + 1;
        };
        while (G > 1 && contributors(G) > pf::kMaxContrib)
            --G;
        sp->sk_grid = G;
        // partials: every range meets at most two shared tiles
        t_split = (double)sp->units * 4.0 / G + 3.0 * kFixed + kRedFixed + red_per_partial * 2.0 * (double)G;
    } else {
        const int64_t rem = tiles % num_sms;
        if (rem == 0)
            return false;
        int64_t fmax = num_sms / rem;
        fmax = fmax < kq ? fmax : kq;
        fmax = fmax < pf::kMaxContrib ? fmax : pf::kMaxContrib;
        int64_t f = 1;
        double best = num_kb;
        for (int64_t ff = 2; ff <= fmax; ++ff) {
            const double tf = num_kb / (double)ff + red_per_partial * (double)(rem * ff);
            if (tf < best) {
                best = tf;
                f = ff;
            }
        }
        if (f < 2)
            return false;
        sp->dp_waves = tiles / num_sms;
        sp->units = rem * kq;
        sp->sk_grid = rem * f;
        t_split = (double)sp->dp_waves * (num_kb + kFixed) + best + 3.0 * kFixed + kRedFixed;
    }
    if (sp->units / sp->sk_grid > (int64_t(1) << 24))
        return false;  // a CTA's stage count must fit an int
    return t_split < best_whole;
}

size_t prefill_workspace_bytes(int64_t N, int64_t M, int64_t K, int n_weights, int fmt)
{
    // the device status word at kStatusWordOffset; split mode adds its partials
    if (!split_possible(K, n_weights, fmt))
        return 256;
    const int64_t units = split_units(N, M, K);
    const int64_t ctas = units < kMaxSplitCtas ? units : kMaxSplitCtas;
    return 256 + (size_t)2 * ctas * pf::BN * pf::BM * sizeof(float);
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
    SplitPlan sp{};
    const bool split = split_plan(N, M, K, n_weights, fmt, num_sms, &sp);
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
        a.after_whole = sp.dp_waves > 0;
        a.sk_base = sp.dp_waves * num_sms * a.kq;
        a.units = sp.units;
        a.partial = reinterpret_cast<float *>(ws + 256);
        // at most one stream-K CTA per unit: every range is non-empty, so a
        // tile's contributors are the contiguous CTAs b_lo .. b_hi
        a.sk_grid = (int)sp.sk_grid;
        a.grid = a.sk_grid;
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
        if (split) {
            if (sp.dp_waves > 0) {
                // the full waves: whole tiles 0 .. dp_waves * SMs - 1
                pf::Args w = a;
                w.split = 0;
                w.after_whole = 0;
                w.grid = (int)(sp.dp_waves * num_sms);
                const cudaError_t e = pf::launch_t<1, true, 0, true, 256>(map, wm, w, stream);
                if (e != cudaSuccess)
                    return e;
            }
            const cudaError_t e = pf::launch_t<1, true, 0, true, 256, true>(map, wm, a, stream);
            if (e != cudaSuccess)
                return e;
            return pf::launch_split_reduce(a, num_sms, stream);
        }
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
