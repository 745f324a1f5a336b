// skinny.cuh -- device helpers shared by the skinny tcgen05 kernels (the
// per-call kernel of gemv_tc.cu and the persistent multi-product kernel of
// stream.cu): exact E2M1 x E4M3 dequantisation into f16 or bf16 operands,
// acquire-release counters, the SwiGLU epilogue, bulk copies, and the host
// helper that encodes TMA tensor maps.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace nvfp4 {
namespace sk {

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


NVFP4_DEVINL uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

NVFP4_DEVINL float silu_mul(float g, float u) { return __fdiv_rn(g, 1.0f + expf(-g)) * u; }

using tc::bulk_load;

// Host: encode a 2-D TMA tensor map (inner dimension first); false if the
// driver entry point is missing or the encoder rejects the arguments.
bool make_map(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

}  // namespace sk
}  // namespace nvfp4
