// gemv.cu -- skinny NVFP4 x bf16 products for N = 1..16 tokens, and the fused
// gate/up + SwiGLU variant.
//
// What it computes (the decode matvec and the batched verify of bw24 README,
// NVFP4 decode path and speculative decoding sections; qwentin README,
// "Highlights", verify reading each weight once for the whole draft tree):
//   y[n][m] = ts * sum_k e2m1(code[m][k]) * e4m3(scale[m][k/16]) * x[n][k]
//
// Design (GB300, HBM-bound: 0.5625 B of weights per multiply-add row):
//   * Work = row tiles of 16 rows x chunks of 128 k.  The (tile, chunk) grid is
//     cut into equal contiguous ranges, one per CTA (one wave: 2 CTAs per SM),
//     so every SM streams the same number of bytes whatever M and K are.
//   * Inside a CTA the 8 warps split the chunks of the current tile.  Each lane
//     streams 16 contiguous code bytes of rows g and g+8 (128-bit loads that
//     skip L1), i.e. a warp covers 16 rows x 128 k per chunk.
//   * Dequantisation is exact and in registers: the 3 magnitude bits of an E2M1
//     code are placed at bf16 bits 8..6 and the sign at bit 15, giving the bf16
//     value e2m1 * 2^-126 (code 1 = 0.5 lands on the bf16 subnormal 2^-127, as
//     E2M1's own subnormal does); one bf16x2 multiply by e4m3(scale) * 2^118
//     then gives e2m1 * scale * 2^-8, exact in bf16 (at most 6 significant
//     bits).  Products with bf16 x are exact in the fp32 accumulator of the
//     tensor-core MMA (mma.sync m16n8k16, weights as A, tokens as B).  The k
//     order inside an MMA is permuted (pairs k, k+4 share a register) in the
//     same way for A and B, which leaves the dot product unchanged.
//   * Reduction order is fixed by (M, K, grid): MMA accumulation over a warp's
//     chunks in order, then warps 0..7 in order, then CTAs in order for the
//     few tiles whose chunk range straddles two CTAs (partials go to the
//     workspace and a small fixup kernel adds them).  Results are deterministic
//     and identical for every N (the grid does not depend on N).
//   * Epilogue: y = acc * 2^8 * ts (fp32 or bf16), or for the gate/up pair
//     h = g / (1 + exp(-g)) * u with g and u from their own tensor scales.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTileRows = 16;
constexpr int kChunkK = 128;

struct GemvArgs {
    const uint16_t *x;
    int N;
    int64_t M, K;
    const uint8_t *codes[2];
    const uint8_t *scales[2];
    const float *ts[2];
    void *y;
    int out_bf16;
    float *partial;   // [P][2 slots][NW][16 rows][16 tokens]
    int64_t tiles, chunks, total;
    int P;
};

template <int NW>
struct Chunk {
    uint4 code[NW][2];     // rows g, g+8: 16 code bytes (32 k) each
    uint32_t scl[NW][2];   // rows g, g+8: 2 scale bytes
};

// Place codes of one 32-bit word (8 codes, k = 0..7) into four bf16x2 words
// holding the pairs (k, k+4) for k = 0..3, each value e2m1 * 2^-126, and scale
// them by `mult` (bf16x2 of e4m3(scale) * 2^118 in both halves).
NVFP4_DEVINL void dequant_word(uint32_t w, uint32_t mult, uint32_t (&out)[4])
{
    constexpr uint32_t kMag = 0x01C001C0u;  // bf16 bits 8..6 of both halves
    const uint32_t te = w & 0x08080808u;    // sign bits of codes 0, 2, 4, 6
    const uint32_t to = w & 0x80808080u;    // sign bits of codes 1, 3, 5, 7
    // (a & kMag) | (b & ~kMag): the b operands hold only sign bits at 15/31
    // (the other sign bits they carry fall on bits 7/23, inside kMag).
    const uint32_t p0 = ((w << 6) & kMag) | ((te << 12) & ~kMag);  // codes 0, 4
    const uint32_t p1 = ((w << 2) & kMag) | ((to << 8) & ~kMag);   // codes 1, 5
    const uint32_t p2 = ((w >> 2) & kMag) | ((te << 4) & ~kMag);   // codes 2, 6
    const uint32_t p3 = ((w >> 6) & kMag) | (to & ~kMag);          // codes 3, 7
    out[0] = bf16x2_mul(p0, mult);
    out[1] = bf16x2_mul(p1, mult);
    out[2] = bf16x2_mul(p2, mult);
    out[3] = bf16x2_mul(p3, mult);
}

NVFP4_DEVINL uint32_t scale_mult(uint32_t byte)
{
    return f32_to_bf16x2_bcast(__fmul_rn(e4m3_to_f32(byte & 0xFF), 0x1p118f));
}

NVFP4_DEVINL int valid_k(int64_t K, int64_t k0)
{
    const int64_t rem = K - k0;
    return rem >= 32 ? 32 : (rem >= 16 ? 16 : 0);
}

template <int NW, bool ALIGNED>
NVFP4_DEVINL void load_chunk(Chunk<NW> &ch, const GemvArgs &a, int64_t tile, int64_t c, int g, int t)
{
    const int64_t k0 = c * kChunkK + 32 * t;
    const int nvalid = valid_k(a.K, k0);
    const int64_t half_k = a.K >> 1, nblk = a.K >> 4;
#pragma unroll
    for (int mi = 0; mi < NW; ++mi) {
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            const int64_t r = tile * kTileRows + g + 8 * ri;
            uint4 cv = make_uint4(0, 0, 0, 0);
            uint32_t sv = 0;
            if (r < a.M && nvalid > 0) {
                const uint8_t *cp = a.codes[mi] + r * half_k + (k0 >> 1);
                const uint8_t *sp = a.scales[mi] + r * nblk + (k0 >> 4);
                if (nvalid == 32) {
                    if (ALIGNED) {
                        cv = ldg_stream_v4(cp);
                        sv = __ldg(reinterpret_cast<const uint16_t *>(sp));
                    } else {
                        uint2 lo = ldg_stream_v2(cp), hi = ldg_stream_v2(cp + 8);
                        cv = make_uint4(lo.x, lo.y, hi.x, hi.y);
                        sv = (uint32_t)__ldg(sp) | ((uint32_t)__ldg(sp + 1) << 8);
                    }
                } else {
                    uint2 lo = ldg_stream_v2(cp);
                    cv = make_uint4(lo.x, lo.y, 0, 0);
                    sv = (uint32_t)__ldg(sp);
                }
            }
            ch.code[mi][ri] = cv;
            ch.scl[mi][ri] = sv;
        }
    }
}

NVFP4_DEVINL uint32_t word_of(const uint4 &v, int q)
{
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

template <int NW, int NT>
NVFP4_DEVINL void compute_chunk(const Chunk<NW> &ch, const GemvArgs &a, int64_t c, int g, int t,
                                float (&acc)[NW][NT][4])
{
    // Activations for this lane's 32 k (token g + 8j): read-only path, L2 hits.
    const int64_t k0 = c * kChunkK + 32 * t;
    const int nvalid = valid_k(a.K, k0);
    uint4 xv[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int n = g + 8 * j;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            xv[j][q] = make_uint4(0, 0, 0, 0);
        if (n < a.N && nvalid > 0) {
            const uint16_t *xp = a.x + (int64_t)n * a.K + k0;
            xv[j][0] = ldg_v4(xp);
            xv[j][1] = ldg_v4(xp + 8);
            if (nvalid == 32) {
                xv[j][2] = ldg_v4(xp + 16);
                xv[j][3] = ldg_v4(xp + 24);
            }
        }
    }
    // B fragments: pairs (k, k+4) of each 8-k group, matching dequant_word.
    uint32_t xb[NT][4][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 r = xv[j][q];
            xb[j][q][0] = prmt(r.x, r.z, 0x5410);  // (k0, k4)
            xb[j][q][1] = prmt(r.x, r.z, 0x7632);  // (k1, k5)
            xb[j][q][2] = prmt(r.y, r.w, 0x5410);  // (k2, k6)
            xb[j][q][3] = prmt(r.y, r.w, 0x7632);  // (k3, k7)
        }
    }
#pragma unroll
    for (int mi = 0; mi < NW; ++mi) {
        uint32_t mult[2][2];
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            mult[ri][0] = scale_mult(ch.scl[mi][ri]);
            mult[ri][1] = scale_mult(ch.scl[mi][ri] >> 8);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t pa[4], pb[4];
            dequant_word(word_of(ch.code[mi][0], q), mult[0][q >> 1], pa);
            dequant_word(word_of(ch.code[mi][1], q), mult[1][q >> 1], pb);
            const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
            const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                mma_bf16_16816(acc[mi][j], a0, xb[j][q][0], xb[j][q][1]);
                mma_bf16_16816(acc[mi][j], a1, xb[j][q][2], xb[j][q][3]);
            }
        }
    }
}

// ---- FP6 E2M3 weights (one UE8M0 scale per 128 k = per chunk and row) ----
//
// A lane holds the same 32 k of rows g and g+8 as above (24 code bytes each).
// The codes unpack to bf16 pairs in natural k order (k, k+1), and the
// activations are used in natural order too: the MMA's logical k slot 2t,2t+1
// holds the lane's pair (k0, k1) of an 8-k group in both operands, slot
// 2t+8,2t+9 the pair (k2, k3); the second MMA of the group takes (k4,k5) and
// (k6,k7).  Each dequantised weight is e2m3 * 2^(s-127), exact in bf16.
template <int NW>
struct Chunk6 {
    uint2 code[NW][2][3];  // rows g, g+8: 24 code bytes (32 k) each
    uint32_t scl[NW][2];   // rows g, g+8: the chunk's scale byte
};

template <int NW>
NVFP4_DEVINL void load_chunk6(Chunk6<NW> &ch, const GemvArgs &a, int64_t tile, int64_t c, int g, int t)
{
    const int64_t row_bytes = a.K / 8 * 6, nblk = a.K / 128;
#pragma unroll
    for (int mi = 0; mi < NW; ++mi) {
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            const int64_t r = tile * kTileRows + g + 8 * ri;
            if (r < a.M) {
                const uint8_t *cp = a.codes[mi] + r * row_bytes + c * 96 + 24 * t;
#pragma unroll
                for (int i = 0; i < 3; ++i)
                    ch.code[mi][ri][i] = ldg_stream_v2(cp + 8 * i);
                ch.scl[mi][ri] = __ldg(a.scales[mi] + r * nblk + c);
            } else {
#pragma unroll
                for (int i = 0; i < 3; ++i)
                    ch.code[mi][ri][i] = make_uint2(0, 0);
                ch.scl[mi][ri] = 127;
            }
        }
    }
}

template <int NW, int NT>
NVFP4_DEVINL void compute_chunk6(const Chunk6<NW> &ch, const GemvArgs &a, int64_t c, int g, int t,
                                 float (&acc)[NW][NT][4])
{
    const int64_t k0 = c * kChunkK + 32 * t;  // K % 128 == 0: all 32 k are valid
    uint4 xv[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int n = g + 8 * j;
        if (n < a.N) {
            const uint16_t *xp = a.x + (int64_t)n * a.K + k0;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xv[j][q] = ldg_v4(xp + 8 * q);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xv[j][q] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int mi = 0; mi < NW; ++mi) {
        const Fp6Mult m0 = fp6_mult(ch.scl[mi][0]), m1 = fp6_mult(ch.scl[mi][1]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 pa = fp6_group(ch.code[mi][0], q, m0);
            const uint4 pb = fp6_group(ch.code[mi][1], q, m1);
            const uint32_t a0[4] = {pa.x, pb.x, pa.y, pb.y};
            const uint32_t a1[4] = {pa.z, pb.z, pa.w, pb.w};
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                mma_bf16_16816(acc[mi][j], a0, xv[j][q].x, xv[j][q].y);
                mma_bf16_16816(acc[mi][j], a1, xv[j][q].z, xv[j][q].w);
            }
        }
    }
}

NVFP4_DEVINL float silu_mul(float g, float u)
{
    return __fdiv_rn(g, 1.0f + expf(-g)) * u;
}

NVFP4_DEVINL void store_out(void *y, int out_bf16, int64_t idx, float v)
{
    if (out_bf16)
        reinterpret_cast<uint16_t *>(y)[idx] = f32_to_bf16(v);
    else
        reinterpret_cast<float *>(y)[idx] = v;
}

// FMT 0: NVFP4 (accumulators hold sum * 2^-8, times the tensor scale);
// FMT 1: FP6 (accumulators hold the sum itself).
template <int NW, int FMT>
NVFP4_DEVINL float finish(const float (&v)[NW], const float (&ts)[NW])
{
    if (FMT == 1)
        return NW == 1 ? v[0] : silu_mul(v[0], v[NW - 1]);
    if (NW == 1)
        return v[0] * 256.0f * ts[0];
    const float g = v[0] * 256.0f * ts[0];
    const float u = v[NW - 1] * 256.0f * ts[NW - 1];
    return silu_mul(g, u);
}

template <int NW, int NT, bool ALIGNED, int FMT>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(GemvArgs a)
{
    using Ch = typename std::conditional<FMT == 0, Chunk<NW>, Chunk6<NW>>::type;
    // Chunks of codes in flight per warp (registers): ~48 KB per SM at 2 CTAs.
    constexpr int kPrefetch = NW == 1 ? 3 : 2;
    __shared__ float red[kWarps][NW][kTileRows][16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int b = blockIdx.x;
    const int64_t lo = (int64_t)b * a.total / a.P;
    const int64_t hi = (int64_t)(b + 1) * a.total / a.P;
    if (lo >= hi)
        return;
    float ts[NW];
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
        ts[mi] = FMT == 0 ? __ldg(a.ts[mi]) : 1.0f;
    const int64_t first_tile = lo / a.chunks;

    for (int64_t tile = first_tile; tile * a.chunks < hi; ++tile) {
        const int64_t tbase = tile * a.chunks;
        const int64_t c0 = (lo > tbase ? lo : tbase) - tbase;
        const int64_t c1 = (hi < tbase + a.chunks ? hi : tbase + a.chunks) - tbase;

        float acc[NW][NT][4];
#pragma unroll
        for (int mi = 0; mi < NW; ++mi)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[mi][j][e] = 0.0f;

        Ch buf[kPrefetch];
        auto load = [&](Ch &dst, int64_t c) {
            if constexpr (FMT == 0)
                load_chunk<NW, ALIGNED>(dst, a, tile, c, g, t);
            else
                load_chunk6<NW>(dst, a, tile, c, g, t);
        };
#pragma unroll
        for (int s = 0; s < kPrefetch; ++s) {
            const int64_t c = c0 + warp + s * kWarps;
            if (c < c1)
                load(buf[s], c);
        }
        for (int64_t cb = c0 + warp; cb < c1; cb += kPrefetch * kWarps) {
#pragma unroll
            for (int s = 0; s < kPrefetch; ++s) {
                const int64_t c = cb + s * kWarps;
                if (c < c1) {
                    if constexpr (FMT == 0)
                        compute_chunk<NW, NT>(buf[s], a, c, g, t, acc);
                    else
                        compute_chunk6<NW, NT>(buf[s], a, c, g, t, acc);
                    const int64_t cn = c + kPrefetch * kWarps;
                    if (cn < c1)
                        load(buf[s], cn);
                }
            }
        }

        // Warp partials -> shared memory (row, token) layout.
#pragma unroll
        for (int mi = 0; mi < NW; ++mi)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                red[warp][mi][g][2 * t + 8 * j] = acc[mi][j][0];
                red[warp][mi][g][2 * t + 1 + 8 * j] = acc[mi][j][1];
                red[warp][mi][g + 8][2 * t + 8 * j] = acc[mi][j][2];
                red[warp][mi][g + 8][2 * t + 1 + 8 * j] = acc[mi][j][3];
            }
        if (NT == 1) {  // tokens 8..15 are not computed: keep them defined
#pragma unroll
            for (int mi = 0; mi < NW; ++mi) {
                red[warp][mi][g][8 + 2 * t] = 0.0f;
                red[warp][mi][g][9 + 2 * t] = 0.0f;
                red[warp][mi][g + 8][8 + 2 * t] = 0.0f;
                red[warp][mi][g + 8][9 + 2 * t] = 0.0f;
            }
        }
        __syncthreads();
        {
            const int tok = threadIdx.x >> 4, row = threadIdx.x & 15;
            const int64_t m = tile * kTileRows + row;
            float v[NW];
#pragma unroll
            for (int mi = 0; mi < NW; ++mi) {
                float s = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w)
                    s += red[w][mi][row][tok];
                v[mi] = s;
            }
            if (c0 == 0 && c1 == a.chunks) {
                if (tok < a.N && m < a.M)
                    store_out(a.y, a.out_bf16, (int64_t)tok * a.M + m, finish<NW, FMT>(v, ts));
            } else {
                const int slot = (tile == first_tile) ? 0 : 1;
#pragma unroll
                for (int mi = 0; mi < NW; ++mi)
                    a.partial[(((int64_t)b * 2 + slot) * NW + mi) * 256 + row * 16 + tok] = v[mi];
            }
        }
        __syncthreads();
    }
}

// CTA whose range contains flattened chunk q.
NVFP4_DEVINL int cta_of(int64_t q, int64_t total, int P)
{
    return (int)(((q + 1) * P - 1) / total);
}

// One block per CTA boundary: the tile holding boundary lo_b (if it lies
// strictly inside a tile and is that tile's first inner boundary) is summed
// over the CTAs that touch it, in CTA order.
template <int NW, int FMT>
__global__ void __launch_bounds__(256) gemv_fixup_kernel(GemvArgs a)
{
    const int b = blockIdx.x + 1;
    const int64_t lo = (int64_t)b * a.total / a.P;
    if (lo % a.chunks == 0 || lo >= a.total)
        return;
    const int64_t tile = lo / a.chunks;
    const int64_t prev = (int64_t)(b - 1) * a.total / a.P;
    if (prev > tile * a.chunks)
        return;  // an earlier boundary inside this tile handles it
    const int b_lo = cta_of(tile * a.chunks, a.total, a.P);
    const int b_hi = cta_of((tile + 1) * a.chunks - 1, a.total, a.P);
    const int tok = threadIdx.x >> 4, row = threadIdx.x & 15;
    const int64_t m = tile * kTileRows + row;
    float ts[NW];
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
        ts[mi] = FMT == 0 ? __ldg(a.ts[mi]) : 1.0f;
    float v[NW];
#pragma unroll
    for (int mi = 0; mi < NW; ++mi)
        v[mi] = 0.0f;
    for (int bb = b_lo; bb <= b_hi; ++bb) {
        const int64_t bfirst = ((int64_t)bb * a.total / a.P) / a.chunks;
        const int slot = (bfirst == tile) ? 0 : 1;
#pragma unroll
        for (int mi = 0; mi < NW; ++mi) {
            float *pp = a.partial + (((int64_t)bb * 2 + slot) * NW + mi) * 256 + row * 16 + tok;
            v[mi] += *pp;
            *pp = 0.0f;  // consumed: the workspace is left zero for the next call
        }
    }
    if (tok < a.N && m < a.M)
        store_out(a.y, a.out_bf16, (int64_t)tok * a.M + m, finish<NW, FMT>(v, ts));
}

template <int NW, int NT, bool ALIGNED, int FMT = 0>
static cudaError_t launch_t(const GemvArgs &a, cudaStream_t stream)
{
    gemv_kernel<NW, NT, ALIGNED, FMT><<<a.P, kThreads, 0, stream>>>(a);
    if (a.P > 1)
        gemv_fixup_kernel<NW, FMT><<<a.P - 1, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

size_t skinny_workspace_bytes(int64_t M, int64_t K, int n_weights)
{
    if (skinny_tc_supported(M, K))
        return skinny_tc_workspace_bytes(M, K, n_weights);
    return gemv_mma_workspace_bytes(n_weights);
}

int64_t gemv_grid(int64_t M, int64_t K, int num_sms)
{
    const int64_t tiles = (M + kTileRows - 1) / kTileRows;
    const int64_t chunks = (K + kChunkK - 1) / kChunkK;
    const int64_t total = tiles * chunks;
    return std::max<int64_t>(1, std::min<int64_t>(total, std::min<int64_t>(kGemvMaxCtas, 2LL * num_sms)));
}

cudaError_t launch_gemv(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                        const uint8_t *const *scales, const float *const *ts, int n_weights, void *y,
                        int out_bf16, void *workspace, int num_sms, cudaStream_t stream)
{
    GemvArgs a{};
    a.x = x;
    a.N = N;
    a.M = M;
    a.K = K;
    for (int i = 0; i < 2; ++i) {
        const int s = i < n_weights ? i : 0;
        a.codes[i] = codes[s];
        a.scales[i] = scales[s];
        a.ts[i] = ts[s];
    }
    a.y = y;
    a.out_bf16 = out_bf16;
    a.partial = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + 256);  // after the header
    a.tiles = (M + kTileRows - 1) / kTileRows;
    a.chunks = (K + kChunkK - 1) / kChunkK;
    a.total = a.tiles * a.chunks;
    a.P = (int)gemv_grid(M, K, num_sms);
    if (a.total == 0)
        return cudaSuccess;
    if (skinny_tc_supported(M, K))
        return launch_skinny_tc(x, N, M, K, codes, scales, ts, n_weights, y, out_bf16, workspace, num_sms, stream);
    const bool aligned = (K % 32) == 0;
    if (n_weights == 1) {
        if (N <= 8)
            return aligned ? launch_t<1, 1, true>(a, stream) : launch_t<1, 1, false>(a, stream);
        return aligned ? launch_t<1, 2, true>(a, stream) : launch_t<1, 2, false>(a, stream);
    }
    if (N <= 8)
        return aligned ? launch_t<2, 1, true>(a, stream) : launch_t<2, 1, false>(a, stream);
    return aligned ? launch_t<2, 2, true>(a, stream) : launch_t<2, 2, false>(a, stream);
}

size_t gemv_mma_workspace_bytes(int n_weights)
{
    return 256 + (size_t)kGemvMaxCtas * kGemvPartialFloatsPerCta * n_weights * 4;
}

cudaError_t launch_gemv_fp6(const uint16_t *x, int N, int64_t M, int64_t K, const uint8_t *const *codes,
                            const uint8_t *const *scales, int n_weights, void *y, int out_bf16, void *workspace,
                            int num_sms, cudaStream_t stream)
{
    GemvArgs a{};
    a.x = x;
    a.N = N;
    a.M = M;
    a.K = K;
    for (int i = 0; i < 2; ++i) {
        const int s = i < n_weights ? i : 0;
        a.codes[i] = codes[s];
        a.scales[i] = scales[s];
        a.ts[i] = nullptr;
    }
    a.y = y;
    a.out_bf16 = out_bf16;
    a.partial = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + 256);
    a.tiles = (M + kTileRows - 1) / kTileRows;
    a.chunks = K / kChunkK;  // K % 128 == 0
    a.total = a.tiles * a.chunks;
    a.P = (int)gemv_grid(M, K, num_sms);
    if (a.total == 0)
        return cudaSuccess;
    if (n_weights == 1)
        return N <= 8 ? launch_t<1, 1, true, 1>(a, stream) : launch_t<1, 2, true, 1>(a, stream);
    return N <= 8 ? launch_t<2, 1, true, 1>(a, stream) : launch_t<2, 2, true, 1>(a, stream);
}

}  // namespace nvfp4
