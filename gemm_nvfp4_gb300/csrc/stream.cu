// stream.cu -- a list of skinny NVFP4 products (N = 1..16 tokens) in one
// persistent launch: the decode step of a whole stack of layers, or any other
// sequence of matvecs and fused gate/up + SwiGLU products, each weight
// streamed from HBM once.
//
// What it computes is the decode / batched-verify matvec of the pages, job by
// job (bw24 README, NVFP4 decode path and speculative decoding sections;
// qwentin README, "Highlights", verify reading each weight once for the whole
// draft tree):
//   y_j[n][m] = ts_j * sum_k e2m1(code_j[m][k]) * e4m3(scale_j[m][k/16]) * x_j[n][k]
// or h_j = silu(g) * u for a gate/up pair.  A job's x is either a caller buffer
// or the bf16 output of an earlier job of the list, so a chain such as
// O -> gate/up + SwiGLU -> down -> next layer's QKV runs inside one launch:
// the persistent-MLP chain of qwentin README ("How it works", one kernel for
// the MLP chain) and the one-replay-per-token decode of bw24 README
// (CUDA-graph decode).
//
// Why one launch: a single product at N = 1 streams its weights in 1.4 to
// 8 us at HBM speed, while a launch pays several microseconds to fill its
// pipeline and to drain and reduce split-K partials.  Here the TMA weight
// producers of every SM walk the units of all jobs back to back, so HBM keeps
// streaming across job boundaries while the epilogue of one job overlaps the
// main loop of the next.
//
// Work decomposition (built on the host, stored in the plan buffer): jobs are
// grouped into phases; a job that reads an earlier job's output starts a new
// phase, and a phase's products start only once every tile of the previous
// phase is final.  Within a phase the units (128 weight rows x 256 k of one
// matrix; a gate/up tile interleaves its gate and up units) of all its jobs
// form one list that is cut into equal contiguous ranges, one per CTA
// (stream-K), so a CTA holds whole tiles except at the ends of its range.  A
// tile split between CTAs is finished by the last CTA to arrive, adding the
// partials in CTA order (deterministic).
//
// Activations enter the MMA as f16 (x * 2^s per token) when every element is
// exact in f16 after that scaling, else as bf16 (the dequantised weights in
// the matching format); either way every product is exact in the fp32
// accumulator.  The per-token decision needs max |x| and the smallest nonzero
// |x|: for a caller buffer they are measured at the start of the launch, for
// an earlier job's output they are accumulated by that job's epilogue.
//
// Every wait is bounded (2 s of wall time), then a code goes to the plan's
// status word and the CTA winds down.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "skinny.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace st {

using sk::dequant_chunk;

constexpr int BM = 128;    // weight rows per tile (MMA M, TMEM lanes)
constexpr int BKU = 256;   // k per unit
constexpr int NTOK = 16;   // MMA N (tokens, padded)
// Warp roles (32 warps): 0..7 MMA issuers, 8 and 9 weight producers, 10 the
// activation producer, 11 the activation converter, 12..15 epilogue, 16..31
// dequantisers (four groups of four warps, one warp per TMEM lane quarter).
// A thread issuing tcgen05.mma spends on the order of a hundred cycles per
// instruction, and a unit needs 16 of them (M = 128, N = 16, K = 16 each), so
// eight issuing threads share them, two per unit each.
constexpr int kMmaWarps = 8;
constexpr int kWProdWarp0 = 8;
constexpr int kXProdWarp = 10;
constexpr int kConvWarp = 11;
constexpr int kEpiWarp0 = 12;
constexpr int kFirstDqWarp = 16;
constexpr int kDqWarps = 16;
constexpr int kThreads = (kFirstDqWarp + kDqWarps) * 32;
constexpr int kEpiThreads = 128;
constexpr int kCodeBox = BM * 128;              // 16 KB: 128 rows x 128 code bytes (256 k), 128-byte swizzle
constexpr int kScaleBox = BM * 16;              // 2 KB: 128 rows x 16 scale bytes
constexpr int kStageBytes = kCodeBox + kScaleBox;
constexpr int kCStages = 10;                    // weight ring (units)
// Activation ring: 32 KB of units of four 64-k sub-boxes.  A sub-box holds 16
// token rows of 128 bytes, or 8 for N <= 8 (the MMA's B operand has 16 rows;
// rows >= N only feed accumulator columns nobody reads, so for N <= 8 rows
// 8..15 may overlap the next sub-box), so small N gets 8 slots of 4 KB.
constexpr int kXRingBytes = 32768;
constexpr int kXMaxStages = 8;
constexpr int kUnitSlots = 8;                   // unit-completion barriers (>= the activation and A rings, in units)
NVFP4_DEVINL int xrows_of(int N) { return N <= 8 ? 8 : 16; }
constexpr int kAStages = 4;                     // TMEM A ring (half units)
constexpr int kACols = 64;
constexpr int kDCols = 128;                     // one accumulator buffer: 8 chains x 16 columns
constexpr uint32_t kTmemCols = 512;
constexpr int kJobSlots = 8;                    // per-job info ring (mode, factors)
constexpr int kReaders = 8;                     // warps reading one weight stage (2 halves x 4 warps)
constexpr int kMaxN = 16;
constexpr int kPartialFloats = 2 * NTOK * BM;   // one split segment: [matrix][token][row]
static_assert(kAStages * kACols + 2 * kDCols <= (int)kTmemCols, "TMEM budget");
static_assert(kUnitSlots >= kXMaxStages && kUnitSlots >= kAStages / 2, "unit barriers cover both rings");
static_assert((kUnitSlots & (kUnitSlots - 1)) == 0, "unit barrier index by mask");
static_assert(kAStages == 4 && kCStages % 2 == 0,
              "dequantiser group g owns A slot g and walks every other unit's weight stage");

// ---------------------------------------------------------------------------
// Plan layout (device memory, built by stream_plan; every offset from the
// start of the plan buffer)
// ---------------------------------------------------------------------------

// One product of the list.  Tensor maps live in global memory (CUtensorMap
// carries its own alignment, at least the 64 bytes the TMA needs): the TMA
// reads them from there.
struct JobDesc {
    CUtensorMap codes[2];   // [M][K/2] uint8, box 128 B x 128 rows, 128-byte swizzle
    CUtensorMap scales[2];  // [M][K/16] uint8, box 16 B x 128 rows
    CUtensorMap x;          // [N][K] bf16 (row stride x_ld), box 64 k x N rows, 128-byte swizzle
    const float *ts[2];
    const uint16_t *x_ptr;  // the activations (a caller buffer, or the producing job's y)
    void *y;
    int64_t x_ld;           // elements between token rows of x
    int64_t M, K;
    int32_t nw;             // 1 matrix, or 2 (gate, up) with SwiGLU
    int32_t out_bf16;
    int32_t C;              // k units: K / 256
    int32_t input;          // -1: caller buffer; else the job whose output is x
    int32_t phase;
    int32_t wait_phase;     // -1, or the phase that must be complete before this job's products
    int32_t feeds;          // 1: another job reads this job's output (keep its statistics)
    int32_t pad;
    int64_t img_off;        // caller-buffer input: byte offset of its f16 image in the plan (else -1)
    int64_t pad2;
};

// A run of consecutive units of one tile done by one CTA.
struct Seg {
    int32_t job;
    int32_t tile;
    int16_t qb, qe;         // units [qb, qe) of the tile; unit q = k unit q / nw of matrix q % nw
    int32_t split;          // -1: the CTA does the whole tile; else the split tile's index
    int32_t slot;           // split: this segment's partial slot
    int32_t pad;
};

// A tile split across CTAs: its contributors' partial slots, in CTA order.
struct Split {
    int32_t first;          // index into the slot list
    int32_t count;
};

// Header at the start of the plan buffer.  Bytes 128..131 hold the device
// status word (as in every product workspace).
struct PlanHeader {
    uint64_t epoch;         // runs completed (advanced by the last CTA of a run)
    uint32_t finished;      // CTAs finished in the current run
    uint32_t magic;
    int32_t P, N, n_jobs, n_phases;
    int32_t n_items, n_splits, pad0, pad1;
    uint32_t off_jobs, off_phase_tiles, off_seg_start, off_segs;
    uint32_t off_splits, off_slot_list, off_items, off_prep_cnt;
    uint32_t off_phase_done, off_stats_in, off_stats_out, off_split_cnt;
    uint64_t off_partials;
};
static_assert(sizeof(PlanHeader) <= 128, "header below the status word");
constexpr uint32_t kPlanMagic = 0x4E565354u;  // "NVST"
constexpr size_t kHeaderBytes = 256;

// Per-job information the activation producer publishes to the other roles.
struct JobInfo {
    int32_t mode;           // 0: f16 operands, 1: bf16 operands
    int32_t convert;        // 1: the converter makes the f16 operand (an earlier job's output, f16 mode)
    int32_t pad[2];
    float xscale[NTOK];     // 2^s_n (f16 mode)
    float fac[2][NTOK];     // epilogue factor per matrix and token
};

// Per-token activation statistics: max |bf16 bits| and 0x7FFF - min nonzero
// |bf16 bits| (both combined with an integer max, so zero is the empty value).
struct TokStat {
    uint32_t mx, inv_mn;
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

NVFP4_DEVINL void fail(uint8_t *plan, uint32_t code)
{
    atomicExch(reinterpret_cast<uint32_t *>(plan + kStatusWordOffset), code);
}

NVFP4_DEVINL uint64_t ld_acquire_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

NVFP4_DEVINL void red_release_add_u64(uint64_t *p, uint64_t v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Generic-proxy global writes (made visible by an acquire) -> the TMA.
NVFP4_DEVINL void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bounded wait for a monotone counter to reach `target`.
NVFP4_DEVINL bool wait_counter(const uint64_t *p, uint64_t target)
{
    if (ld_acquire_u64(p) >= target)
        return true;
    const uint64_t t0 = tc::globaltimer();
    for (;;) {
        __nanosleep(128);
        if (ld_acquire_u64(p) >= target)
            return true;
        if (tc::globaltimer() - t0 > tc::kWaitLimitNs)
            return false;
    }
}

// f16 operands are exact for a token when, after scaling by 2^s with
// s = 142 - E(max) (so max |x| * 2^s lies in [2^15, 2^16)), every nonzero
// element keeps its lowest significant bit at or above 2^-24: the exponent
// fields of max and min nonzero |x| differ by at most 32, no subnormal bf16
// input, everything finite.  Returns s, or INT_MIN when bf16 is needed.
NVFP4_DEVINL int token_shift(uint32_t mx, uint32_t inv_mn)
{
    if (mx == 0)
        return 0;
    const uint32_t mn = 0x7FFFu - inv_mn;
    const int emax = (int)(mx >> 7), emin = (int)(mn >> 7);
    const int s = 142 - emax;
    if (mx >= 0x7F80u || emin < 1 || emax - emin > 32 || s > 120 || s < -120)
        return -0x7FFFFFFF - 1;
    return s;
}

NVFP4_DEVINL float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Max and (0x7FFF - min nonzero) of |bf16 bits| of four packed words of x.
NVFP4_DEVINL void absbits_minmax(uint4 v, uint32_t &mx, uint32_t &inv_mn)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[i] & 0x7FFFu, b = (w[i] >> 16) & 0x7FFFu;
        mx = max(mx, max(a, b));
        if (a)
            inv_mn = max(inv_mn, 0x7FFFu - a);
        if (b)
            inv_mn = max(inv_mn, 0x7FFFu - b);
    }
}

// 16-byte chunk of 8 bf16 activations -> 8 f16 values times 2^s (exact when
// the token passed token_shift).
NVFP4_DEVINL uint4 bf16x8_to_f16x8(uint4 v, float scale)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16) * scale;
        const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * scale;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(hi), "f"(lo));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace st
}  // namespace nvfp4

namespace nvfp4 {
namespace st {

// Shared-memory layout of the kernel.
constexpr size_t kSmemBytes = 1024                                   // alignment slack
                              + (size_t)kCStages * kStageBytes        // weight ring
                              + (size_t)kXRingBytes                   // activation ring
                              + (size_t)kJobSlots * sizeof(JobInfo)   // job information ring
                              + 96 * 8                                // mbarriers
                              + 256;                                  // TMEM address, flags, reductions
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Views of the plan buffer.
struct PlanView {
    const JobDesc *jobs;
    const int64_t *phase_tiles;
    const int32_t *seg_start;
    const Seg *segs;
    const Split *splits;
    const int32_t *slot_list;
    const int32_t *items;
    uint64_t *prep_cnt;
    uint64_t *phase_done;
    TokStat *stats_in;     // [n_jobs][16]
    TokStat *stats_out;    // [2][n_jobs][16]
    uint32_t *split_cnt;
    float *partials;       // [slots][kPartialFloats]
};

NVFP4_DEVINL PlanView view(uint8_t *plan, const PlanHeader &h)
{
    PlanView v;
    v.jobs = reinterpret_cast<const JobDesc *>(plan + h.off_jobs);
    v.phase_tiles = reinterpret_cast<const int64_t *>(plan + h.off_phase_tiles);
    v.seg_start = reinterpret_cast<const int32_t *>(plan + h.off_seg_start);
    v.segs = reinterpret_cast<const Seg *>(plan + h.off_segs);
    v.splits = reinterpret_cast<const Split *>(plan + h.off_splits);
    v.slot_list = reinterpret_cast<const int32_t *>(plan + h.off_slot_list);
    v.items = reinterpret_cast<const int32_t *>(plan + h.off_items);
    v.prep_cnt = reinterpret_cast<uint64_t *>(plan + h.off_prep_cnt);
    v.phase_done = reinterpret_cast<uint64_t *>(plan + h.off_phase_done);
    v.stats_in = reinterpret_cast<TokStat *>(plan + h.off_stats_in);
    v.stats_out = reinterpret_cast<TokStat *>(plan + h.off_stats_out);
    v.split_cnt = reinterpret_cast<uint32_t *>(plan + h.off_split_cnt);
    v.partials = reinterpret_cast<float *>(plan + h.off_partials);
    return v;
}

// Output value of row m, token n (stored as fp32 or bf16); returns the |bf16
// bits| of the stored value for the activation statistics (0 for fp32 output).
NVFP4_DEVINL uint32_t store_y(const JobDesc *J, int n, int64_t m, float val)
{
    const int64_t idx = (int64_t)n * J->M + m;
    if (J->out_bf16) {
        const uint16_t bits = f32_to_bf16(val);
        reinterpret_cast<uint16_t *>(J->y)[idx] = bits;
        return bits & 0x7FFFu;
    }
    reinterpret_cast<float *>(J->y)[idx] = val;
    return 0;
}

NVFP4_DEVINL float combine(int nw, const JobInfo *ji, int n, float s0, float s1)
{
    return nw == 1 ? s0 * ji->fac[0][n] : sk::silu_mul(s0 * ji->fac[0][n], s1 * ji->fac[1][n]);
}

NVFP4_DEVINL void stat_add(TokStat *st, uint32_t mx, uint32_t inv_mn)
{
    if (mx)
        atomicMax(&st->mx, mx);
    if (inv_mn)
        atomicMax(&st->inv_mn, inv_mn);
}

// Activation producer: wait until the job's activations and their statistics
// are final, derive the operand format and the per-token scales, and publish
// them in job-information slot lj % kJobSlots.  False after a timeout.
__device__ __noinline__ bool publish_job(uint8_t *plan, const PlanView &v, int N, int n_jobs, uint64_t e, int job,
                                         int lj, JobInfo *jinfo, uint64_t *j_full, uint64_t *j_empty)
{
    const JobDesc *J = v.jobs + job;
    const int wp = J->wait_phase;
    if (wp >= 0 && !wait_counter(v.phase_done + wp, (uint64_t)v.phase_tiles[wp] * (e + 1))) {
        fail(plan, 34);
        return false;
    }
    const TokStat *stt;
    if (J->input < 0) {
        if (!wait_counter(v.prep_cnt + job, (uint64_t)N * (e + 1))) {
            fail(plan, 35);
            return false;
        }
        stt = v.stats_in + (size_t)job * NTOK;
    } else {
        stt = v.stats_out + ((size_t)(e & 1) * n_jobs + J->input) * NTOK;
    }
    int sh[NTOK];
    int mode = 0;
    for (int n = 0; n < N; ++n) {
        const uint32_t mx = __ldcg(&stt[n].mx), inv = __ldcg(&stt[n].inv_mn);
        sh[n] = token_shift(mx, inv);
        if (sh[n] == -0x7FFFFFFF - 1)
            mode = 1;
    }
    fence_proxy_async_global();  // the activations are read by the TMA next
    const int slot = lj % kJobSlots;
    if (!tc::mbar_wait(&j_empty[slot], (((uint32_t)lj / kJobSlots) & 1) ^ 1)) {
        fail(plan, 36);
        return false;
    }
    JobInfo *ji = jinfo + slot;
    ji->mode = mode;
    ji->convert = (mode == 0 && J->input >= 0) ? 1 : 0;
    const float ts0 = __ldg(J->ts[0]), ts1 = J->nw == 2 ? __ldg(J->ts[1]) : 0.0f;
    for (int n = 0; n < NTOK; ++n) {
        const bool live = n < N;
        ji->xscale[n] = (live && mode == 0) ? pow2f(sh[n]) : 1.0f;
        const float f = !live ? 0.0f : mode ? 256.0f : pow2f(-sh[n]);
        ji->fac[0][n] = ts0 * f;
        ji->fac[1][n] = ts1 * f;
    }
    tc::mbar_arrive(&j_full[slot]);
    return true;
}

}  // namespace st
}  // namespace nvfp4

namespace nvfp4 {
namespace st {


// Everything the roles of stream_kernel share, set up once per CTA.  Each role
// runs in its own non-inlined function, so the registers one role needs (the
// epilogue holds 32 partial sums per thread) do not crowd another's loop.
struct Ctx {
    uint8_t *plan;
    const PlanHeader *H;
    const PlanHeader *hs;
    uint8_t *c_ring, *x_ring;
    JobInfo *jinfo;
    uint64_t *c_full, *c_empty, *x_raw, *x_full, *u_done, *a_full, *d_full, *d_empty, *j_full, *j_empty;
    int *last_s;
    uint32_t *red_s;
    const Seg *segs;
    const JobDesc *jobs;
    uint32_t tmem_a, tmem_d;
    int n_seg, N, P, n_jobs, xrows, x_sub, x_unit, x_stages, b;
    bool ok;
};

// A thread's handle on its CTA's context: the shared copy, and its warp and
// lane.  The roles read warp and lane from this handle in memory: computing
// them from threadIdx inside the roles, or passing them as arguments, ran
// about 5% slower (measured on the 9B and 27B decode streams).
struct CtxRef {
    const Ctx *shared;
    int warp, lane;
};

#define NVFP4_STREAM_UNPACK(cr)                                                                             \
    const Ctx &c = *(cr).shared;                                                                            \
    uint8_t *plan = (c).plan;                                                                               \
    const PlanHeader *H = (c).H;                                                                            \
    const PlanHeader &hd = *(c).hs;                                                                         \
    uint8_t *c_ring = (c).c_ring, *x_ring = (c).x_ring;                                                     \
    JobInfo *jinfo = (c).jinfo;                                                                             \
    uint64_t *c_full = (c).c_full, *c_empty = (c).c_empty, *x_raw = (c).x_raw, *x_full = (c).x_full;      \
    uint64_t *u_done = (c).u_done, *a_full = (c).a_full, *d_full = (c).d_full, *d_empty = (c).d_empty;   \
    uint64_t *j_full = (c).j_full, *j_empty = (c).j_empty;                                                 \
    int *last_s = (c).last_s;                                                                               \
    uint32_t *red_s = (c).red_s;                                                                            \
    const Seg *segs = (c).segs;                                                                             \
    const JobDesc *jobs = (c).jobs;                                                                         \
    const uint32_t tmem_a = (c).tmem_a, tmem_d = (c).tmem_d;                                              \
    const int n_seg = (c).n_seg, N = (c).N, P = (c).P, n_jobs = (c).n_jobs;                               \
    const int xrows = (c).xrows, x_sub = (c).x_sub, x_unit = (c).x_unit, x_stages = (c).x_stages;         \
    const int warp = (cr).warp, lane = (cr).lane, b = (c).b;                                                \
    const bool ok = (c).ok;                                                                                 \
    (void)plan; (void)H; (void)hd; (void)c_ring; (void)x_ring; (void)jinfo; (void)c_full; (void)c_empty;    \
    (void)x_raw; (void)x_full; (void)u_done; (void)a_full; (void)d_full; (void)d_empty; (void)j_full;      \
    (void)j_empty; (void)last_s; (void)red_s; (void)segs; (void)jobs; (void)tmem_a; (void)tmem_d;          \
    (void)n_seg; (void)N; (void)P; (void)n_jobs; (void)xrows; (void)x_sub; (void)x_unit; (void)x_stages;   \
    (void)warp; (void)lane; (void)b; (void)ok

// Role: weight producers.
__device__ __noinline__ void role_wprod(const CtxRef &cr)
{
    NVFP4_STREAM_UNPACK(cr);

        // ---- weight producers: even / odd units of the CTA's sequence ----
        if (lane == 0) {
            const int par = warp - kWProdWarp0;
            const uint32_t c_empty_a = tc::smem_addr(c_empty), c_full_a = tc::smem_addr(c_full);
            const uint32_t ring_a = tc::smem_addr(c_ring);
            int u = 0;
            int ws = par;
            uint32_t wph = 0;
            bool stop = false;
            int prev = -1;
            for (int si = 0; si < n_seg && !stop; ++si) {
                const Seg sg = segs[si];
                const JobDesc *J = jobs + sg.job;
                const int nw = J->nw;
                if (sg.job != prev) {
                    prev = sg.job;
                    for (int m = 0; m < nw; ++m) {
                        tc::prefetch_tensormap(&J->codes[m]);
                        tc::prefetch_tensormap(&J->scales[m]);
                    }
                }
                for (int q = sg.qb; q < sg.qe; ++q, ++u) {
                    if ((u & 1) != par)
                        continue;
                    const int s = ws;          // stage of unit u (u % kCStages), advanced two units at a time
                    const uint32_t ph = wph;
                    ws += 2;
                    if (ws >= kCStages) {
                        ws -= kCStages;
                        wph ^= 1;
                    }
                    if (!tc::mbar_wait_a(c_empty_a + 8u * (uint32_t)s, ph ^ 1)) {
                        fail(plan, 32);
                        stop = true;
                        break;
                    }
                    const uint32_t stg = ring_a + (uint32_t)s * (uint32_t)kStageBytes;
                    const uint32_t full = c_full_a + 8u * (uint32_t)s;
                    tc::mbar_arrive_expect_tx_a(full, kStageBytes);
                    const int m = q % nw, j = q / nw;
                    tc::tma_load_2d_a(stg, &J->codes[m], full, j * (BKU / 2), sg.tile * BM);
                    tc::tma_load_2d_a(stg + kCodeBox, &J->scales[m], full, j * (BKU / 16), sg.tile * BM);
                }
            }
        }
}

// Role: activation producer.
__device__ __noinline__ void role_xprod(const CtxRef &cr)
{
    NVFP4_STREAM_UNPACK(cr);

        // ---- activation producer: per job, wait for its inputs and publish its
        // operand format and scales; per unit, the N token rows of the unit's
        // four 64-k sub-boxes as bf16 through the job's tensor map (rows >= N of
        // the MMA's B operand feed accumulator columns nobody reads: zeroed once) ----
        for (int o = lane * 16; o < kXRingBytes; o += 32 * 16)
            *reinterpret_cast<uint4 *>(x_ring + o) = make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && ok) {
            const PlanView v = view(plan, hd);
            tc::griddep_wait();
            const uint64_t e = *reinterpret_cast<volatile const uint64_t *>(&H->epoch);
            const uint32_t row_bytes = (uint32_t)N * 128;
            const uint32_t u_done_a = tc::smem_addr(u_done), xring_a = tc::smem_addr(x_ring);
            const uint32_t x_raw_a = tc::smem_addr(x_raw), x_full_a = tc::smem_addr(x_full);
            int u = 0, lj = -1, prev = -1, xs = 0;
            bool stop = false;
            for (int si = 0; si < n_seg && !stop; ++si) {
                const Seg sg = segs[si];
                const JobDesc *J = jobs + sg.job;
                if (sg.job != prev) {
                    prev = sg.job;
                    ++lj;
                    if (!publish_job(plan, v, N, n_jobs, e, sg.job, lj, jinfo, j_full, j_empty))
                        break;
                    tc::prefetch_tensormap(&J->x);
                }
                const int nw = J->nw;
                // operands: the f16 image of a caller buffer (bulk copies), x
                // itself (bf16 mode), or x for the converter (an earlier job's
                // output in f16 mode)
                const JobInfo *ji = jinfo + lj % kJobSlots;
                const bool from_img = ji->mode == 0 && J->input < 0;
                const bool conv = ji->convert != 0;
                const uint8_t *img = plan + (J->img_off > 0 ? J->img_off : 0);
                for (int q = sg.qb; q < sg.qe; ++q, ++u) {
                    const int s = xs;
                    if (++xs == x_stages)
                        xs = 0;
                    // the slot's previous unit (u - x_stages) has been consumed
                    const int pu = u - x_stages;
                    if (pu >= 0 &&
                        !tc::mbar_wait_a(u_done_a + 8u * (uint32_t)(pu & (kUnitSlots - 1)), (uint32_t)(pu / kUnitSlots) & 1)) {
                        fail(plan, 33);
                        stop = true;
                        break;
                    }
                    const uint32_t dst = xring_a + (uint32_t)(s * x_unit);
                    const uint32_t bar = (conv ? x_raw_a : x_full_a) + 8u * (uint32_t)s;
                    const int j = q / nw;
                    if (from_img) {
                        // the image has the slot's layout: one copy per unit
                        // (rows >= N are never read)
                        tc::mbar_arrive_expect_tx_a(bar, (uint32_t)x_unit);
                        tc::bulk_load_a(dst, img + (size_t)j * x_unit, (uint32_t)x_unit, bar);
                    } else {
                        tc::mbar_arrive_expect_tx_a(bar, 4 * row_bytes);
#pragma unroll
                        for (int sb = 0; sb < 4; ++sb)
                            tc::tma_load_2d_a(dst + (uint32_t)(sb * x_sub), &J->x, bar, j * BKU + sb * 64, 0);
                    }
                }
            }
        }
}

// Role: activation converter.
__device__ __noinline__ void role_conv(const CtxRef &cr)
{
    NVFP4_STREAM_UNPACK(cr);

        // ---- activation converter, for an earlier job's output in f16 mode:
        // bf16 -> f16 * 2^s_n in place (the 128-byte swizzle moves whole
        // 16-byte chunks, so each chunk converts where it lies), then the unit
        // is ready for the MMA.  Other units never pass through here, so the
        // phase of each slot's barrier is tracked per slot.  The converter also
        // releases each job's information slot (with the epilogue), so it can
        // never fall a whole ring behind the activation producer. ----
        int u = 0, lj = -1, prev = -1;
        uint32_t rawph = 0;
        bool conv = false, stop = false;
        const int chunks = 4 * N * 8;
        for (int si = 0; si < n_seg && !stop; ++si) {
            const Seg sg = segs[si];
            if (sg.job != prev) {
                prev = sg.job;
                ++lj;
                if (!tc::mbar_wait(&j_full[lj % kJobSlots], ((uint32_t)lj / kJobSlots) & 1)) {
                    fail(plan, 37);
                    break;
                }
                conv = jinfo[lj % kJobSlots].convert != 0;
            }
            const JobInfo *ji = jinfo + lj % kJobSlots;
            for (int q = sg.qb; q < sg.qe && conv; ++q, ++u) {
                const int s = (int)((uint32_t)u % (uint32_t)x_stages);
                if (!tc::mbar_wait(&x_raw[s], (rawph >> s) & 1)) {
                    fail(plan, 38);
                    stop = true;
                    break;
                }
                rawph ^= 1u << s;
                uint8_t *base = x_ring + (size_t)s * x_unit;
                for (int i = lane; i < chunks; i += 32) {
                    const int sb = i / (N * 8), rem = i - sb * N * 8;
                    const int r = rem >> 3, c = rem & 7;
                    uint4 *p = reinterpret_cast<uint4 *>(base + sb * x_sub + r * 128 + c * 16);
                    *p = bf16x8_to_f16x8(*p, ji->xscale[r]);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(&x_full[s]);
            }
            if (!conv)
                u += sg.qe - sg.qb;
            __syncwarp();
            if (lane == 0 && (si + 1 == n_seg || segs[si + 1].job != sg.job))
                tc::mbar_arrive(&j_empty[lj % kJobSlots]);
        }
}

// Role: MMA issuers.
__device__ __noinline__ void role_mma(const CtxRef &cr)
{
    NVFP4_STREAM_UNPACK(cr);
    // ---- MMA issuers: issuer w owns accumulator slot w.  One matrix: chain
    // w takes K steps 2(w % 4) and 2(w % 4) + 1 of half unit w / 4 of every
    // unit, so an issuer waits for one half only (measured: +3 to +6 % on the
    // 9B and 27B streams at N <= 9 against every issuer taking one K step of
    // both halves; -1 % at N = 16).  A gate/up pair: slot w is matrix w / 4,
    // chain w % 4, K steps kk = w (mod 4) of that matrix's half units (the
    // gate and up units of a k range run on the two halves of the issuers at
    // the same time).  Ring positions are advanced incrementally: no
    // divisions in the loop. ----
    if (lane != 0)
        return;
    // barriers by 32-bit shared address (one register each, no conversion per use)
    const uint32_t x_full_a = tc::smem_addr(x_full), a_full_a = tc::smem_addr(a_full);
    const uint32_t u_done_a = tc::smem_addr(u_done), d_full_a = tc::smem_addr(d_full);
    const uint32_t d_empty_a = tc::smem_addr(d_empty), j_full_a = tc::smem_addr(j_full);
    int lj = -1, prev = -1;
    uint32_t idesc = 0;
    int xs = 0, sa = 0;            // activation and A ring slots
    uint32_t xph = 0, aph = 0;     // their phases
    uint32_t ud = 0;               // unit counter (completion barrier u % kUnitSlots)
    for (int si = 0; si < n_seg; ++si) {
        const Seg sg = segs[si];
        const int nw = jobs[sg.job].nw;
        if (sg.job != prev) {
            prev = sg.job;
            ++lj;
            if (!tc::mbar_wait_a(j_full_a + 8u * (uint32_t)(lj % kJobSlots), ((uint32_t)lj / kJobSlots) & 1)) {
                fail(plan, 39);
                return;
            }
            idesc = tc::idesc_f16kind(BM, NTOK, (uint32_t)jinfo[lj % kJobSlots].mode);
        }
        const int buf = si & 1;
        if (!tc::mbar_wait_a(d_empty_a + 8u * (uint32_t)buf, (((uint32_t)si >> 1) & 1) ^ 1)) {
            fail(plan, 40);
            return;
        }
        tc::fence_after_sync();
        const uint32_t dcol = tmem_d + (uint32_t)(buf * kDCols + warp * 16);
        // this issuer's K steps of a half unit, as A column and B descriptor offsets
        const int nk = nw == 1 ? 1 : 2, kk0 = nw == 1 ? warp : (warp & 3);
        uint32_t aoff[2], boff[2][2];
        for (int i = 0; i < 2; ++i) {
            const int kk = kk0 + 4 * i;
            aoff[i] = (uint32_t)(kk * 8);
            for (int h = 0; h < 2; ++h) {
                const int kl = h * 128 + kk * 16;  // k within the unit
                // B: sub-box kl / 64 of the unit, 32-byte step kl % 64 in it (16-byte units)
                boff[h][i] = (uint32_t)((kl >> 6) * (x_sub / 16) + 2 * ((kl >> 4) & 3));
            }
        }
        // one matrix: this issuer's two K steps of its half unit (constant offsets)
        uint32_t aoff1[2], boff1[2];
        for (int i = 0; i < 2; ++i) {
            const int kk = 2 * (warp & 3) + i;
            const int kl = (warp >> 2) * 128 + kk * 16;
            aoff1[i] = (uint32_t)(kk * 8);
            boff1[i] = (uint32_t)((kl >> 6) * (x_sub / 16) + 2 * ((kl >> 4) & 3));
        }
        const uint64_t xdesc = tc::smem_desc_sw128(x_ring);
        bool fresh = true;
        for (int q = sg.qb; q < sg.qe; ++q) {
            const bool mine = nw == 1 || (q & 1) == (warp >> 2);
            if (nw == 1) {
                // one matrix: this issuer's half unit only (slot sa + half; sa advances by two)
                if (!tc::mbar_wait_a(x_full_a + 8u * (uint32_t)xs, xph) ||
                    !tc::mbar_wait_a(a_full_a + 8u * (uint32_t)(sa + (warp >> 2)), aph)) {
                    fail(plan, 41);
                    return;
                }
                tc::fence_after_sync();
                const uint64_t bdesc0 = xdesc + (uint64_t)((xs * x_unit) >> 4);
                const uint32_t acol = tmem_a + (uint32_t)((sa + (warp >> 2)) * kACols);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    tc::mma_f16_ts(dcol, acol + aoff1[i], bdesc0 + boff1[i], idesc, fresh ? 0u : 1u);
                    fresh = false;
                }
                sa += 2;
                if (sa == kAStages) {
                    sa = 0;
                    aph ^= 1;
                }
            } else if (mine) {
                if (!tc::mbar_wait_a(x_full_a + 8u * (uint32_t)xs, xph)) {
                    fail(plan, 41);
                    return;
                }
                const uint64_t bdesc0 = xdesc + (uint64_t)((xs * x_unit) >> 4);
                for (int h = 0; h < 2; ++h) {
                    // one matrix: issuer w takes K steps 2(w % 4), 2(w % 4) + 1 of half w / 4 only
                    if (nw == 1 && h != (warp >> 2)) {
                        if (++sa == kAStages) {
                            sa = 0;
                            aph ^= 1;
                        }
                        continue;
                    }
                    if (!tc::mbar_wait_a(a_full_a + 8u * (uint32_t)sa, aph)) {
                        fail(plan, 42);
                        return;
                    }
                    tc::fence_after_sync();
                    const uint32_t acol = tmem_a + (uint32_t)(sa * kACols);
                    if (nw == 1) {
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            tc::mma_f16_ts(dcol, acol + aoff1[i], bdesc0 + boff1[i], idesc, fresh ? 0u : 1u);
                            fresh = false;
                        }
                    } else {
                        for (int i = 0; i < nk; ++i) {
                            tc::mma_f16_ts(dcol, acol + aoff[i], bdesc0 + boff[h][i], idesc, fresh ? 0u : 1u);
                            fresh = false;
                        }
                    }
                    if (++sa == kAStages) {
                        sa = 0;
                        aph ^= 1;
                    }
                }
            } else if (++sa, ++sa >= kAStages) {  // skip the unit's two half units
                sa -= kAStages;
                aph ^= 1;
            }
            // the unit's MMAs of this thread (if any) are done -> its share of u_done
            tc::mma_commit_a(u_done_a + 8u * (ud & (kUnitSlots - 1)));
            ++ud;
            if (++xs == x_stages) {
                xs = 0;
                xph ^= 1;
            }
        }
        tc::mma_commit_a(d_full_a + 8u * (uint32_t)buf);
    }
}

// Role: epilogue.
__device__ __noinline__ void role_epi(const CtxRef &cr)
{
    NVFP4_STREAM_UNPACK(cr);

        // ---- epilogue (one warp per TMEM lane quarter) ----
        const PlanView v = view(plan, hd);
        const int et = threadIdx.x - kEpiWarp0 * 32;  // 0..127
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint64_t e = 0;
        if (ok) {
            tc::griddep_wait();
            e = *reinterpret_cast<volatile const uint64_t *>(&H->epoch);
            // 1. statistics of the caller-provided activations: item i = (job,
            //    token) for i = b, b + P, ...; one writer per item.
            for (int i = b; i < hd.n_items; i += P) {
                const int item = v.items[i];
                const int job = item >> 5, n = item & 31;
                const JobDesc *J = v.jobs + job;
                const uint16_t *xr = J->x_ptr + (int64_t)n * J->x_ld;
                uint32_t mx = 0, inv = 0;
                for (int64_t c = et; c < J->K / 8; c += kEpiThreads)
                    absbits_minmax(ldg_v4(xr + c * 8), mx, inv);
                for (int o = 16; o > 0; o >>= 1) {
                    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
                    inv = max(inv, __shfl_xor_sync(0xFFFFFFFFu, inv, o));
                }
                if (lane == 0) {
                    red_s[2 * quarter] = mx;
                    red_s[2 * quarter + 1] = inv;
                }
                tc::named_bar_sync(1, kEpiThreads);
                if (et == 0) {
                    for (int w = 1; w < 4; ++w) {
                        mx = max(mx, red_s[2 * w]);
                        inv = max(inv, red_s[2 * w + 1]);
                    }
                    v.stats_in[(size_t)job * NTOK + n] = TokStat{mx, inv};
                    red_s[0] = mx;
                    red_s[1] = inv;
                }
                tc::named_bar_sync(1, kEpiThreads);
                // the token's f16 image (x * 2^s, in the activation ring's
                // layout), when f16 is exact for it; the job's activation
                // producer copies it unit by unit
                const int sh = token_shift(red_s[0], red_s[1]);
                if (sh != -0x7FFFFFFF - 1) {
                    const float scale = pow2f(sh);
                    uint8_t *img = plan + J->img_off + (size_t)n * 128;
                    for (int64_t c = et; c < J->K / 8; c += kEpiThreads) {
                        const int64_t k = c * 8;
                        const int kl = (int)(k & (BKU - 1)), ch = (kl >> 3) & 7;
                        uint8_t *dst = img + (size_t)(k / BKU) * x_unit + (kl >> 6) * x_sub + ((ch ^ (n & 7)) << 4);
                        *reinterpret_cast<uint4 *>(dst) = bf16x8_to_f16x8(ldg_v4(xr + k), scale);
                    }
                }
                tc::named_bar_sync(1, kEpiThreads);
                if (et == 0) {
                    fence_proxy_async_global();  // the image is read by bulk copies
                    red_release_add_u64(v.prep_cnt + job, 1);
                }
            }
            // 2. the next run accumulates output statistics in the other half:
            //    clear it now (this run does not touch it).
            for (int jj = b; jj < n_jobs; jj += P)
                if (v.jobs[jj].feeds && et < NTOK)
                    v.stats_out[((size_t)((e + 1) & 1) * n_jobs + jj) * NTOK + et] = TokStat{0, 0};
        }
        // 3. the CTA's segments
        const uint32_t j_full_a = tc::smem_addr(j_full), d_full_a = tc::smem_addr(d_full);
        const uint32_t d_empty_a = tc::smem_addr(d_empty);
        int lj = -1, prev = -1;
        for (int si = 0; si < n_seg; ++si) {
            const Seg sg = segs[si];
            const JobDesc *J = jobs + sg.job;
            const int nw = J->nw;
            if (sg.job != prev) {
                prev = sg.job;
                ++lj;
                if (!tc::bar_and(1, kEpiThreads,
                                 tc::mbar_wait_a(j_full_a + 8u * (uint32_t)(lj % kJobSlots),
                                                 ((uint32_t)lj / kJobSlots) & 1))) {
                    fail(plan, 43);
                    break;
                }
            }
            const JobInfo *ji = jinfo + lj % kJobSlots;
            const int buf = si & 1;
            if (!tc::bar_and(1, kEpiThreads, tc::mbar_wait_a(d_full_a + 8u * (uint32_t)buf, ((uint32_t)si >> 1) & 1))) {
                fail(plan, 44);
                break;
            }
            tc::fence_after_sync();
            // accumulator slots 0..7 (16 columns each), added in a fixed order:
            // one matrix: slots 0..7; a gate/up pair: gate 0..3, up 4..7
            float sum[2][NTOK];
#pragma unroll
            for (int n = 0; n < NTOK; ++n)
                sum[0][n] = sum[1][n] = 0.0f;
#pragma unroll 1
            for (int sl = 0; sl < 8; ++sl) {
                uint32_t a[NTOK];
                tc::tmem_ld_32x32b_x16(tmem_d + buf * kDCols + sl * 16 + lane_off, a);
                tc::tmem_ld_wait();
                if (nw == 2 && sl >= 4) {
#pragma unroll
                    for (int n = 0; n < NTOK; ++n)
                        sum[1][n] += __uint_as_float(a[n]);
                } else {
#pragma unroll
                    for (int n = 0; n < NTOK; ++n)
                        sum[0][n] += __uint_as_float(a[n]);
                }
            }
            if (nw == 2) {
                // a matrix with no unit in the segment got no MMA: its slots hold stale values
                const bool g_ok = (sg.qe - sg.qb >= 2) || (sg.qb % 2 == 0);
                const bool u_ok = (sg.qe - sg.qb >= 2) || (sg.qb % 2 == 1);
#pragma unroll
                for (int n = 0; n < NTOK; ++n) {
                    if (!g_ok)
                        sum[0][n] = 0.0f;
                    if (!u_ok)
                        sum[1][n] = 0.0f;
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive_a(d_empty_a + 8u * (uint32_t)buf);

            bool final_tile = false;
            TokStat *ost = v.stats_out + ((size_t)(e & 1) * n_jobs + sg.job) * NTOK;
            if (sg.split < 0) {
                // the CTA did the whole tile: outputs (and their statistics)
                const int64_t m = (int64_t)sg.tile * BM + r;
                const bool live = m < J->M;
#pragma unroll
                for (int n = 0; n < NTOK; ++n) {
                    if (n >= N)
                        break;
                    uint32_t ab = 0;
                    if (live)
                        ab = store_y(J, n, m, combine(nw, ji, n, sum[0][n], sum[1][n]));
                    if (J->feeds) {
                        uint32_t mx = ab, inv = ab ? 0x7FFFu - ab : 0u;
                        for (int o = 16; o > 0; o >>= 1) {
                            mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
                            inv = max(inv, __shfl_xor_sync(0xFFFFFFFFu, inv, o));
                        }
                        if (lane == 0)
                            stat_add(ost + n, mx, inv);
                    }
                }
                final_tile = true;
            } else {
                // publish this CTA's partial; the last contributor to arrive adds them all
                float *mine = v.partials + (size_t)sg.slot * kPartialFloats + r;
#pragma unroll
                for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                    for (int n = 0; n < NTOK; ++n)
                        if (mi < nw && n < N)
                            mine[(mi * NTOK + n) * BM] = sum[mi][n];
                tc::named_bar_sync(1, kEpiThreads);
                const Split spl = v.splits[sg.split];
                if (et == 0) {
                    // release: every thread's partial stores (ordered by the barrier);
                    // acquire: the other contributors' partials
                    const uint32_t old = sk::atom_add_acq_rel(v.split_cnt + sg.split, 1u);
                    *last_s = old == (uint32_t)(spl.count - 1);
                    if (*last_s)
                        v.split_cnt[sg.split] = 0;  // for the next run
                }
                tc::named_bar_sync(1, kEpiThreads);
                if (*last_s) {
                    for (int p = et; p < N * (BM / 4); p += kEpiThreads) {
                        const int n = p / (BM / 4), r4 = (p % (BM / 4)) * 4;
                        float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
                        for (int c0 = 0; c0 < spl.count; c0 += 4) {
                            float4 pv[4][2];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const int cc = min(c0 + c, spl.count - 1);
                                const float *src = v.partials + (size_t)v.slot_list[spl.first + cc] * kPartialFloats +
                                                   n * BM + r4;
#pragma unroll
                                for (int mi = 0; mi < 2; ++mi)
                                    pv[c][mi] = mi < nw ? __ldcg(reinterpret_cast<const float4 *>(src + mi * NTOK * BM))
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (c0 + c < spl.count)
#pragma unroll
                                    for (int mi = 0; mi < 2; ++mi) {
                                        acc[mi].x += pv[c][mi].x;
                                        acc[mi].y += pv[c][mi].y;
                                        acc[mi].z += pv[c][mi].z;
                                        acc[mi].w += pv[c][mi].w;
                                    }
                        }
                        const float g4[4] = {acc[0].x, acc[0].y, acc[0].z, acc[0].w};
                        const float u4[4] = {acc[1].x, acc[1].y, acc[1].z, acc[1].w};
                        uint32_t mx = 0, inv = 0;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int64_t m = (int64_t)sg.tile * BM + r4 + q;
                            if (m < J->M) {
                                const uint32_t ab = store_y(J, n, m, combine(nw, ji, n, g4[q], u4[q]));
                                mx = max(mx, ab);
                                if (ab)
                                    inv = max(inv, 0x7FFFu - ab);
                            }
                        }
                        if (J->feeds)
                            stat_add(ost + n, mx, inv);
                    }
                    final_tile = true;
                }
            }
            // every output, statistic and read of the job information is done
            tc::named_bar_sync(1, kEpiThreads);
            if (et == 0) {
                if (final_tile) {
                    fence_proxy_async_global();  // the outputs may be read by a later job's TMA
                    red_release_add_u64(v.phase_done + J->phase, 1);
                }
                if (si + 1 == n_seg || segs[si + 1].job != sg.job)
                    tc::mbar_arrive(&j_empty[lj % kJobSlots]);
            }
        }
}

// Role: dequantisers.
__device__ __noinline__ void role_dq(const CtxRef &cr)
{
    NVFP4_STREAM_UNPACK(cr);
    // ---- dequantisers: half unit t = 2u + h goes to group t % 4, so group g
    // takes half h = g % 2 of the units u = g / 2 (mod 2), always into A slot
    // g; it walks its units two at a time with incremental ring positions.
    // Shared memory is reached through 32-bit shared addresses (ld.shared,
    // one register per address), which keeps the loop within its registers. ----
    const int g = (warp - kFirstDqWarp) >> 2;
    const int h = g & 1;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int swz = r & 7;
    if (n_seg == 0)
        return;
    const uint32_t c_full_a = tc::smem_addr(c_full), c_empty_a = tc::smem_addr(c_empty);
    const uint32_t u_done_a = tc::smem_addr(u_done), a_full_a = tc::smem_addr(a_full) + 8u * (uint32_t)g;
    const uint32_t j_full_a = tc::smem_addr(j_full), jinfo_a = tc::smem_addr(jinfo);
    // this thread's row of the weight ring's code box, and of its scale box
    const uint32_t ring_row = tc::smem_addr(c_ring) + (uint32_t)(r * 128);
    const uint32_t ring_scl = tc::smem_addr(c_ring) + (uint32_t)(kCodeBox + r * 16 + h * 8);
    // cursor over the CTA's units: segment si, unit q of its tile, local job lj
    int si = 0, lj = 0;
    int job = segs[0].job, qe = segs[0].qe;
    int q = segs[0].qb;
    auto step = [&](int k) -> bool {  // advance k units; false past the last one
        q += k;
        while (q >= qe) {
            const int over = q - qe;
            if (++si >= n_seg)
                return false;
            const int nj = segs[si].job;
            if (nj != job)
                ++lj;
            job = nj;
            qe = segs[si].qe;
            q = segs[si].qb + over;
        }
        return true;
    };
    if (!step(g >> 1))
        return;
    uint32_t u = (uint32_t)(g >> 1);
    int sc = g >> 1;               // weight stage of unit u (u % kCStages) and its phase
    uint32_t phc = 0;
    int have = -1, mode = 0;
    const uint32_t acol = tmem_a + (uint32_t)(g * kACols) + lane_off;
    for (;;) {
        if (have != lj) {
            const uint32_t js = (uint32_t)(lj % kJobSlots);
            if (!tc::mbar_wait_a(j_full_a + 8u * js, ((uint32_t)lj / kJobSlots) & 1)) {
                fail(plan, 45);
                return;
            }
            mode = (int)tc::lds32(jinfo_a + js * (uint32_t)sizeof(JobInfo) + (uint32_t)offsetof(JobInfo, mode));
            have = lj;
        }
        if (!tc::mbar_wait_a(c_full_a + 8u * (uint32_t)sc, phc)) {
            fail(plan, 46);
            return;
        }
        const uint32_t stage_off = (uint32_t)sc * (uint32_t)kStageBytes;
        uint4 cw[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
            cw[cc] = tc::lds128(ring_row + stage_off + (uint32_t)(((h * 4 + cc) ^ swz) << 4));
        const uint2 sc8 = tc::lds64(ring_scl + stage_off);
        __syncwarp();
        if (lane == 0)
            tc::mbar_arrive_a(c_empty_a + 8u * (uint32_t)sc);
        // A slot g was last filled for unit u - 2: its MMAs must have completed
        if (u >= 2) {
            const uint32_t pu = u - 2;
            if (!tc::mbar_wait_a(u_done_a + 8u * (pu & (kUnitSlots - 1)), (pu / kUnitSlots) & 1)) {
                fail(plan, 47);
                return;
            }
        }
        tc::fence_after_sync();
        // one 16-byte chunk (32 k) at a time: 16 columns per store; the
        // operand format is fixed per job, so each format has its own loop
        auto put = [&](auto fmt) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t out[16];
                const uint32_t sw = cc < 2 ? sc8.x : sc8.y;
                dequant_chunk(cw[cc], (cc & 1) ? sw >> 16 : sw & 0xFFFF, decltype(fmt)::value, out);
                tc::tmem_st_32x32b_x16(acol + 16 * cc, out);
            }
        };
        if (mode == 0)
            put(std::integral_constant<int, 0>{});
        else
            put(std::integral_constant<int, 1>{});
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0)
            tc::mbar_arrive_a(a_full_a);
        u += 2;
        sc += 2;
        if (sc >= kCStages) {
            sc -= kCStages;
            phc ^= 1;
        }
        if (!step(2))
            return;
    }
}

__global__ void __launch_bounds__(kThreads, 1) stream_kernel(uint8_t *plan)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *c_ring = smem;                                        // [kCStages][codes 16 KB, scales 2 KB]
    uint8_t *x_ring = c_ring + (size_t)kCStages * kStageBytes;     // [x_stages][x_unit]
    JobInfo *jinfo = reinterpret_cast<JobInfo *>(x_ring + (size_t)kXRingBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(jinfo + kJobSlots);
    uint64_t *c_full = bars;
    uint64_t *c_empty = c_full + kCStages;
    uint64_t *x_raw = c_empty + kCStages;
    uint64_t *x_full = x_raw + kXMaxStages;
    // u_done[u % 8]: every MMA of unit u has completed (one commit per issuer
    // and unit); it frees the unit's activation slot and its two A items.
    uint64_t *u_done = x_full + kXMaxStages;
    uint64_t *a_full = u_done + kUnitSlots;
    uint64_t *d_full = a_full + kAStages;
    uint64_t *d_empty = d_full + 2;
    uint64_t *j_full = d_empty + 2;
    uint64_t *j_empty = j_full + kJobSlots;
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + 96);
    uint32_t *tmem_slot = misc;       // [0]
    int *ok_s = reinterpret_cast<int *>(misc + 1);
    int *last_s = reinterpret_cast<int *>(misc + 2);
    uint32_t *red_s = misc + 8;       // [8] reductions of the epilogue warps
    PlanHeader *hs = reinterpret_cast<PlanHeader *>(misc + 32);  // the plan header, copied once
    static_assert(2 * kCStages + 2 * kXMaxStages + kUnitSlots + kAStages + 4 + 2 * kJobSlots <= 96, "barrier count");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const PlanHeader *H = reinterpret_cast<const PlanHeader *>(plan);

    if (threadIdx.x == 0) {
        tc::griddep_launch_dependents();
        for (int s = 0; s < kCStages; ++s) {
            tc::mbar_init(&c_full[s], 1);
            tc::mbar_init(&c_empty[s], kReaders);
        }
        for (int s = 0; s < kXMaxStages; ++s) {
            tc::mbar_init(&x_raw[s], 1);
            tc::mbar_init(&x_full[s], 1);

        }
        for (int s = 0; s < kAStages; ++s) {
            tc::mbar_init(&a_full[s], 4);

        }
        for (int s = 0; s < kUnitSlots; ++s)
            tc::mbar_init(&u_done[s], kMmaWarps);
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&d_full[s], kMmaWarps);
            tc::mbar_init(&d_empty[s], kEpiThreads / 32);
        }
        for (int s = 0; s < kJobSlots; ++s) {
            tc::mbar_init(&j_full[s], 1);
            tc::mbar_init(&j_empty[s], 2);  // the epilogue and the converter
        }
        tc::fence_mbar_init();
        // The plan's constant part was written before any run; a plan built for
        // another grid size is refused.
        *ok_s = (H->magic == kPlanMagic && H->P == (int)gridDim.x) ? 1 : 0;
        *hs = *H;  // constant fields (the epoch is read after the grid dependency)
        if (!*ok_s && H->magic == kPlanMagic)
            fail(plan, 31);
    }
    if (warp == 0)
        tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_a = tmem;
    const uint32_t tmem_d = tmem + kAStages * kACols;
    const bool ok = *ok_s != 0;

    const PlanHeader &hd = *hs;
    const int N = hd.N, P = hd.P, n_jobs = hd.n_jobs;
    const int xrows = xrows_of(N);
    const int x_sub = xrows * 128;                 // bytes of one sub-box
    const int x_unit = 4 * x_sub;
    const int x_stages = kXRingBytes / x_unit;
    const Seg *segs;
    int n_seg;
    {
        const int32_t *seg_start = reinterpret_cast<const int32_t *>(plan + hd.off_seg_start);
        segs = reinterpret_cast<const Seg *>(plan + hd.off_segs) + (ok ? seg_start[b] : 0);
        n_seg = ok ? seg_start[b + 1] - seg_start[b] : 0;
    }
    const JobDesc *jobs = reinterpret_cast<const JobDesc *>(plan + hd.off_jobs);

    // The roles' context is the same for every thread of the CTA: one copy in
    // shared memory (a per-thread copy would live in local memory, written by
    // every thread and evicted to DRAM).
    __shared__ Ctx ctx_s;
    if (threadIdx.x == 0) {
        Ctx &c = ctx_s;
        c.plan = plan;
        c.H = H;
        c.hs = hs;
        c.c_ring = c_ring;
        c.x_ring = x_ring;
        c.jinfo = jinfo;
        c.c_full = c_full;
        c.c_empty = c_empty;
        c.x_raw = x_raw;
        c.x_full = x_full;
        c.u_done = u_done;
        c.a_full = a_full;
        c.d_full = d_full;
        c.d_empty = d_empty;
        c.j_full = j_full;
        c.j_empty = j_empty;
        c.last_s = last_s;
        c.red_s = red_s;
        c.segs = segs;
        c.jobs = jobs;
        c.tmem_a = tmem_a;
        c.tmem_d = tmem_d;
        c.n_seg = n_seg;
        c.N = N;
        c.P = P;
        c.n_jobs = n_jobs;
        c.xrows = xrows;
        c.x_sub = x_sub;
        c.x_unit = x_unit;
        c.x_stages = x_stages;
        c.b = b;
        c.ok = ok;
    }
    __syncthreads();
    CtxRef cr;
    cr.shared = &ctx_s;
    cr.warp = warp;
    cr.lane = lane;
    if (warp == kWProdWarp0 || warp == kWProdWarp0 + 1)
        role_wprod(cr);
    else if (warp == kXProdWarp)
        role_xprod(cr);
    else if (warp == kConvWarp)
        role_conv(cr);
    else if (warp < kMmaWarps)
        role_mma(cr);
    else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4)
        role_epi(cr);
    else
        role_dq(cr);

    // Lane 0 of the producer and MMA warps ran their loops alone: reconverge
    // each warp first, so the block-wide barrier really waits for every thread.
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && ok) {
        // the last CTA of the run advances the epoch (the next run's targets)
        __threadfence();
        uint32_t *fin = reinterpret_cast<uint32_t *>(plan + offsetof(PlanHeader, finished));
        if (atomicAdd(fin, 1u) == (uint32_t)P - 1) {
            *fin = 0;
            uint64_t *ep = reinterpret_cast<uint64_t *>(plan);
            *ep = *reinterpret_cast<volatile uint64_t *>(ep) + 1;
            __threadfence();
        }
    }
}

}  // namespace st
}  // namespace nvfp4

// ---------------------------------------------------------------------------
// host side: the plan
// ---------------------------------------------------------------------------

#include "../../include/nvfp4.h"

namespace nvfp4 {
namespace st {

static_assert(sizeof(JobDesc) % 64 == 0 && alignof(JobDesc) >= 64 && kHeaderBytes % alignof(JobDesc) == 0,
              "job descriptors keep their tensor maps 64-byte aligned");
constexpr int kMaxCtas = 256;

inline size_t align64(size_t v) { return (v + 63) / 64 * 64; }
inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Validated job list: phases, inputs, and the per-job sizes the plan needs.
struct JobsInfo {
    int n_phases = 0;
    std::vector<int> phase, feeds, nw, input;
    std::vector<int64_t> tiles, units_per_tile;
};

int check_jobs(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N, JobsInfo *ji)
{
    if (n_jobs < 1 || !jobs)
        return NVFP4_ERR_INVALID_ARG;
    if (N < 1 || N > kMaxN)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (n_jobs > (1 << 20))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    ji->phase.assign(n_jobs, 0);
    ji->feeds.assign(n_jobs, 0);
    ji->tiles.assign(n_jobs, 0);
    ji->units_per_tile.assign(n_jobs, 0);
    ji->nw.assign(n_jobs, 1);
    ji->input.assign(n_jobs, -1);
    int phase = 0;
    for (int j = 0; j < n_jobs; ++j) {
        const nvfp4_skinny_job &J = jobs[j];
        if (J.n_weights != 1 && J.n_weights != 2)
            return NVFP4_ERR_INVALID_ARG;
        if (J.out_dtype != NVFP4_OUT_F32 && J.out_dtype != NVFP4_OUT_BF16)
            return NVFP4_ERR_INVALID_ARG;
        if (J.M < 1 || J.K < 1 || J.x_ld < 0)
            return NVFP4_ERR_INVALID_ARG;
        // the tcgen05 units are 256 k wide; a tile holds at most 32767 units
        if (J.K % 256 != 0 || J.K / 256 * J.n_weights > 32767 || J.M > (INT64_C(1) << 31) - 128)
            return NVFP4_ERR_UNSUPPORTED_SHAPE;
        for (int i = 0; i < J.n_weights; ++i)
            if (!J.codes[i] || !J.scales[i] || !J.tensor_scale[i] || !aligned(J.codes[i], 16) ||
                !aligned(J.scales[i], 16) || !aligned(J.tensor_scale[i], 4))
                return NVFP4_ERR_INVALID_ARG;
        if (!J.y || !aligned(J.y, 16))
            return NVFP4_ERR_INVALID_ARG;
        if (J.input < 0) {
            const int64_t ld = J.x_ld ? J.x_ld : J.K;
            if (J.input != -1 || !J.x || !aligned(J.x, 16) || ld < J.K || ld % 8 != 0)
                return NVFP4_ERR_INVALID_ARG;
        } else {
            if (J.input >= j)
                return NVFP4_ERR_INVALID_ARG;
            const nvfp4_skinny_job &I = jobs[J.input];
            // x = the producing job's bf16 output, row stride its M
            if (I.out_dtype != NVFP4_OUT_BF16 || I.M < J.K || I.M % 8 != 0)
                return NVFP4_ERR_INVALID_ARG;
            ji->feeds[J.input] = 1;
            if (j > 0)
                ++phase;
        }
        ji->phase[j] = phase;
        ji->tiles[j] = (J.M + BM - 1) / BM;
        ji->units_per_tile[j] = J.K / 256 * J.n_weights;
        ji->nw[j] = J.n_weights;
        ji->input[j] = J.input;
    }
    ji->n_phases = phase + 1;
    return NVFP4_OK;
}

struct Layout {
    size_t jobs, phase_tiles, seg_start, segs, splits, slot_list, items, state, prep_cnt, phase_done, stats_in,
        stats_out, split_cnt, state_end, partials, images, total;
    std::vector<int64_t> img_off;  // per job: its f16 image (caller-buffer inputs), else -1
};

// Sizes of every section for P CTAs, with upper bounds on the segment and
// split counts (the build fills at most that many).
Layout layout(const JobsInfo &ji, const std::vector<int> &jobs_input, int n_jobs, int64_t N, int n_items, int P)
{
    int64_t tiles = 0;
    for (int j = 0; j < n_jobs; ++j)
        tiles += ji.tiles[j];
    const int64_t max_segs = tiles + (int64_t)ji.n_phases * P;
    const int64_t max_splits = (int64_t)ji.n_phases * P;
    Layout L;
    size_t o = kHeaderBytes;
    L.jobs = o;
    o = align64(o + (size_t)n_jobs * sizeof(JobDesc));
    L.phase_tiles = o;
    o = align64(o + (size_t)ji.n_phases * 8);
    L.seg_start = o;
    o = align64(o + (size_t)(P + 1) * 4);
    L.segs = o;
    o = align64(o + (size_t)max_segs * sizeof(Seg));
    L.splits = o;
    o = align64(o + (size_t)max_splits * sizeof(Split));
    L.slot_list = o;
    o = align64(o + (size_t)max_splits * 2 * 4);
    L.items = o;
    o = align64(o + (size_t)std::max(n_items, 1) * 4);
    L.state = o;
    L.prep_cnt = o;
    o = align64(o + (size_t)n_jobs * 8);
    L.phase_done = o;
    o = align64(o + (size_t)ji.n_phases * 8);
    L.stats_in = o;
    o = align64(o + (size_t)n_jobs * NTOK * sizeof(TokStat));
    L.stats_out = o;
    o = align64(o + (size_t)2 * n_jobs * NTOK * sizeof(TokStat));
    L.split_cnt = o;
    o = align64(o + (size_t)max_splits * 4);
    L.state_end = o;
    L.partials = (o + 255) / 256 * 256;
    L.images = L.partials + (size_t)4 * P * kPartialFloats * 4;
    // f16 images of the caller-provided activations: K / 256 units of four
    // sub-boxes of 8 (N <= 8) or 16 token rows of 128 bytes
    const size_t x_unit = (size_t)4 * (N <= 8 ? 8 : 16) * 128;
    size_t io = L.images;
    L.img_off.assign(n_jobs, -1);
    for (int j = 0; j < n_jobs; ++j)
        if (jobs_input[j] < 0) {
            L.img_off[j] = (int64_t)io;
            io += (size_t)(ji.units_per_tile[j] / ji.nw[j]) * x_unit;
            io = (io + 255) / 256 * 256;
        }
    L.total = io;
    return L;
}

int n_items_of(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N)
{
    int n = 0;
    for (int j = 0; j < n_jobs; ++j)
        if (jobs[j].input < 0)
            n += (int)N;
    return n;
}

int num_sms_now(int *out)
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0)
        return NVFP4_ERR_CUDA;
    *out = std::min(n, kMaxCtas);
    return NVFP4_OK;
}

}  // namespace st
}  // namespace nvfp4

namespace nvfp4 {
namespace st {

// Host image of a plan (constant part and zero-filled state).
struct Built {
    Layout L;
    std::vector<uint8_t> image;  // bytes [0, L.state_end)
};

int build_plan(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N, const JobsInfo &ji, int P, Built *out)
{
    const int n_items = n_items_of(jobs, n_jobs, N);
    const Layout L = layout(ji, ji.input, n_jobs, N, n_items, P);
    std::vector<uint8_t> img(L.state_end, 0);
    PlanHeader h{};
    h.magic = kPlanMagic;
    h.P = P;
    h.N = (int32_t)N;
    h.n_jobs = n_jobs;
    h.n_phases = ji.n_phases;
    h.n_items = n_items;
    h.off_jobs = (uint32_t)L.jobs;
    h.off_phase_tiles = (uint32_t)L.phase_tiles;
    h.off_seg_start = (uint32_t)L.seg_start;
    h.off_segs = (uint32_t)L.segs;
    h.off_splits = (uint32_t)L.splits;
    h.off_slot_list = (uint32_t)L.slot_list;
    h.off_items = (uint32_t)L.items;
    h.off_prep_cnt = (uint32_t)L.prep_cnt;
    h.off_phase_done = (uint32_t)L.phase_done;
    h.off_stats_in = (uint32_t)L.stats_in;
    h.off_stats_out = (uint32_t)L.stats_out;
    h.off_split_cnt = (uint32_t)L.split_cnt;
    h.off_partials = L.partials;
    if (L.state_end > UINT32_MAX)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;

    // jobs: tensor maps and scalars
    JobDesc *jd = reinterpret_cast<JobDesc *>(img.data() + L.jobs);
    for (int j = 0; j < n_jobs; ++j) {
        const nvfp4_skinny_job &J = jobs[j];
        JobDesc d;
        std::memset(&d, 0, sizeof(d));
        const int nw = J.n_weights;
        for (int i = 0; i < 2; ++i) {
            const int s = i < nw ? i : 0;
            if (!sk::make_map(&d.codes[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, J.codes[s], (uint64_t)J.K / 2,
                              (uint64_t)J.M, (uint64_t)J.K / 2, BKU / 2, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
                !sk::make_map(&d.scales[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, J.scales[s], (uint64_t)J.K / 16,
                              (uint64_t)J.M, (uint64_t)J.K / 16, BKU / 16, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
                return NVFP4_ERR_CUDA;
            d.ts[i] = J.tensor_scale[s];
        }
        const uint16_t *x = J.input < 0 ? J.x : reinterpret_cast<const uint16_t *>(jobs[J.input].y);
        const int64_t ld = J.input < 0 ? (J.x_ld ? J.x_ld : J.K) : jobs[J.input].M;
        if (!sk::make_map(&d.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)J.K, (uint64_t)N, (uint64_t)ld * 2,
                          64, (uint32_t)N, CU_TENSOR_MAP_SWIZZLE_128B))
            return NVFP4_ERR_CUDA;
        d.x_ptr = x;
        d.x_ld = ld;
        d.y = J.y;
        d.M = J.M;
        d.K = J.K;
        d.nw = nw;
        d.out_bf16 = J.out_dtype == NVFP4_OUT_BF16;
        d.C = (int32_t)(J.K / BKU);
        d.input = J.input;
        d.phase = ji.phase[j];
        d.wait_phase = ji.phase[j] - 1;
        d.feeds = ji.feeds[j];
        d.img_off = L.img_off[j];
        std::memcpy(&jd[j], &d, sizeof(d));
    }

    // phases: tile totals, and the stream-K split of each phase's unit list
    std::vector<std::vector<Seg>> per_cta(P);
    std::vector<Split> splits;
    std::vector<int32_t> slot_list;
    int64_t *phase_tiles = reinterpret_cast<int64_t *>(img.data() + L.phase_tiles);
    int j0 = 0;
    for (int p = 0; p < ji.n_phases; ++p) {
        int j1 = j0;
        while (j1 < n_jobs && ji.phase[j1] == p)
            ++j1;
        // tiles of the phase in order, with their first unit in the phase's list
        std::vector<int> t_job;
        std::vector<int32_t> t_tile;
        std::vector<int64_t> t_start;
        int64_t U = 0, T = 0;
        for (int j = j0; j < j1; ++j)
            for (int64_t t = 0; t < ji.tiles[j]; ++t) {
                t_job.push_back(j);
                t_tile.push_back((int32_t)t);
                t_start.push_back(U);
                U += ji.units_per_tile[j];
                ++T;
            }
        phase_tiles[p] = T;
        t_start.push_back(U);
        // contributors of each tile: (cta, segment index in that CTA's list)
        std::vector<std::vector<std::pair<int, size_t>>> contrib(T);
        for (int b = 0; b < P; ++b) {
            const int64_t lo = (int64_t)((__int128)U * b / P), hi = (int64_t)((__int128)U * (b + 1) / P);
            if (lo >= hi)
                continue;
            int64_t ti = std::upper_bound(t_start.begin(), t_start.end(), lo) - t_start.begin() - 1;
            for (int64_t pos = lo; pos < hi; ++ti) {
                const int64_t ts = t_start[ti], te = t_start[ti + 1];
                const int64_t qb = pos - ts, qe = std::min(hi, te) - ts;
                Seg sg;
                sg.job = t_job[ti];
                sg.tile = t_tile[ti];
                sg.qb = (int16_t)qb;
                sg.qe = (int16_t)qe;
                sg.split = -1;
                sg.slot = -1;
                sg.pad = 0;
                contrib[ti].push_back({b, per_cta[b].size()});
                per_cta[b].push_back(sg);
                pos = ts + qe;
            }
        }
        // tiles with several contributors: partial slots and the split list
        std::vector<int> n_split_of_cta(P, 0);
        for (int64_t ti = 0; ti < T; ++ti) {
            if (contrib[ti].size() < 2)
                continue;
            const int id = (int)splits.size();
            splits.push_back(Split{(int32_t)slot_list.size(), (int32_t)contrib[ti].size()});
            for (auto &c : contrib[ti]) {
                const int b = c.first;
                const int i = n_split_of_cta[b]++;
                if (i > 1)
                    return NVFP4_ERR_UNSUPPORTED_SHAPE;  // cannot happen with contiguous ranges
                Seg &sg = per_cta[b][c.second];
                sg.split = id;
                sg.slot = (p & 1) * 2 * P + 2 * b + i;
                slot_list.push_back(sg.slot);
            }
        }
        j0 = j1;
    }
    // flatten the per-CTA lists
    int32_t *seg_start = reinterpret_cast<int32_t *>(img.data() + L.seg_start);
    Seg *segs = reinterpret_cast<Seg *>(img.data() + L.segs);
    size_t ns = 0;
    const size_t max_segs = (L.splits - L.segs) / sizeof(Seg);
    for (int b = 0; b < P; ++b) {
        seg_start[b] = (int32_t)ns;
        if (ns + per_cta[b].size() > max_segs)
            return NVFP4_ERR_UNSUPPORTED_SHAPE;
        std::memcpy(segs + ns, per_cta[b].data(), per_cta[b].size() * sizeof(Seg));
        ns += per_cta[b].size();
    }
    seg_start[P] = (int32_t)ns;
    if (splits.size() > (L.slot_list - L.splits) / sizeof(Split) ||
        slot_list.size() > (L.items - L.slot_list) / 4)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    std::memcpy(img.data() + L.splits, splits.data(), splits.size() * sizeof(Split));
    std::memcpy(img.data() + L.slot_list, slot_list.data(), slot_list.size() * 4);
    h.n_splits = (int32_t)splits.size();
    // activation statistics of the caller buffers: one item per (job, token)
    int32_t *items = reinterpret_cast<int32_t *>(img.data() + L.items);
    int k = 0;
    for (int j = 0; j < n_jobs; ++j)
        if (jobs[j].input < 0)
            for (int n = 0; n < N; ++n)
                items[k++] = (j << 5) | n;
    std::memcpy(img.data(), &h, sizeof(h));
    out->L = L;
    out->image.swap(img);
    return NVFP4_OK;
}

cudaError_t set_smem_attr()
{
    static std::once_flag once[kMaxDevices];
    static cudaError_t err[kMaxDevices];
    return once_per_device(once, err, [] {
        return cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    });
}

}  // namespace st
}  // namespace nvfp4

extern "C" {

size_t nvfp4_stream_plan_bytes(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N)
{
    using namespace nvfp4::st;
    JobsInfo ji;
    if (check_jobs(jobs, n_jobs, N, &ji) != NVFP4_OK)
        return 0;
    return layout(ji, ji.input, n_jobs, N, n_items_of(jobs, n_jobs, N), kMaxCtas).total;
}

int nvfp4_stream_plan(const nvfp4_skinny_job *jobs, int n_jobs, int64_t N, void *plan, size_t plan_bytes,
                      nvfp4_stream_t stream)
{
    using namespace nvfp4::st;
    JobsInfo ji;
    int rc = check_jobs(jobs, n_jobs, N, &ji);
    if (rc != NVFP4_OK)
        return rc;
    if (plan_bytes < nvfp4_stream_plan_bytes(jobs, n_jobs, N))
        return NVFP4_ERR_WORKSPACE;
    if (!plan || !aligned(plan, 256))
        return NVFP4_ERR_INVALID_ARG;
    int P = 0;
    if ((rc = num_sms_now(&P)) != NVFP4_OK)
        return rc;
    Built bp;
    if ((rc = build_plan(jobs, n_jobs, N, ji, P, &bp)) != NVFP4_OK)
        return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(plan, bp.image.data(), bp.image.size(), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

int nvfp4_stream_run(void *plan, size_t plan_bytes, nvfp4_stream_t stream)
{
    using namespace nvfp4::st;
    if (!plan || !aligned(plan, 256) || plan_bytes < kHeaderBytes)
        return NVFP4_ERR_INVALID_ARG;
    int P = 0;
    int rc = num_sms_now(&P);
    if (rc != NVFP4_OK)
        return rc;
    if (set_smem_attr() != cudaSuccess)
        return NVFP4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_kernel, reinterpret_cast<uint8_t *>(plan)) == cudaSuccess
               ? NVFP4_OK
               : NVFP4_ERR_CUDA;
}

}  // extern "C"
