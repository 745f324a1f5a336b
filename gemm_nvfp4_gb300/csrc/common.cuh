// common.cuh -- small device helpers shared by the NVFP4 kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define NVFP4_DEVINL __device__ __forceinline__

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------

// Streaming 16-byte load that is not kept in L1 (weights are read once).
NVFP4_DEVINL uint4 ldg_stream_v4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

NVFP4_DEVINL uint2 ldg_stream_v2(const void *p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

// Read-only cached 16-byte load (activations, reused by many warps).
NVFP4_DEVINL uint4 ldg_v4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

NVFP4_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// ---------------------------------------------------------------------------
// Element conversions (hardware instructions; no arithmetic reimplemented)
// ---------------------------------------------------------------------------

// Two E4M3 bytes (low byte -> low half) to f16x2, exact.
NVFP4_DEVINL uint32_t e4m3x2_to_f16x2(uint16_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

// E4M3 byte to its exact fp32 value.
NVFP4_DEVINL float e4m3_to_f32(uint32_t byte)
{
    uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(byte & 0xFF));
    float f;
    asm("{ .reg .f16 lo, hi; mov.b32 {lo, hi}, %1; cvt.f32.f16 %0, lo; }" : "=f"(f) : "r"(h2));
    return f;
}

// fp32 -> E4M3 byte, round to nearest even, saturating to +-448.
NVFP4_DEVINL uint32_t f32_to_e4m3_satfinite(float v)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
    return r & 0xFF;
}

// Two fp32 -> one byte of two E2M1 codes: `lo` in bits 3..0, `hi` in bits 7..4;
// round to nearest even, saturating to +-6.
NVFP4_DEVINL uint32_t f32x2_to_e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------------------
// Tensor-core MMA (warp-level, bf16 x bf16 -> fp32)
// ---------------------------------------------------------------------------

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
NVFP4_DEVINL void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

NVFP4_DEVINL uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// fp32 -> bf16 (round to nearest even) in both halves of a 32-bit word.
NVFP4_DEVINL uint32_t f32_to_bf16x2_bcast(float v)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(v));
    return r;
}

NVFP4_DEVINL uint16_t f32_to_bf16(float v)
{
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

// ---------------------------------------------------------------------------
// FP6 E2M3 weights (block-scaled variant: UE8M0 scale per 128 k)
// ---------------------------------------------------------------------------

// Two E2M3 codes (bits 0..5 and 6..11 of u) -> bf16x2 holding e2m3 * 2^-126
// each.  The five magnitude bits (2 exponent, 3 mantissa) land on bf16 bits
// 8..4, so the bf16 exponent field is the E2M3 exponent field and the mantissa
// is m/8: a normal code reads 2^(e-127) * (1 + m/8) = e2m3 * 2^-126 and a
// subnormal code (e = 0) the bf16 subnormal 2^-126 * m/8 = e2m3 * 2^-126.
// The sign goes to bit 15.
NVFP4_DEVINL uint32_t e2m3x2_to_bf16x2(uint32_t u)
{
    return ((u << 4) & 0x000001F0u) | ((u << 10) & 0x00008000u) | ((u << 14) & 0x01F00000u) |
           ((u << 20) & 0x80000000u);
}

// Eight codes of a 48-bit little-endian group (lo = bits 0..31, hi = 32..47)
// -> four bf16x2 words in natural k order (k0k1, k2k3, k4k5, k6k7).
NVFP4_DEVINL uint4 e2m3x8_to_bf16(uint32_t lo, uint32_t hi)
{
    return make_uint4(e2m3x2_to_bf16x2(lo), e2m3x2_to_bf16x2(lo >> 12),
                      e2m3x2_to_bf16x2((lo >> 24) | (hi << 8)), e2m3x2_to_bf16x2(hi >> 4));
}

// Multipliers that turn e2m3 * 2^-126 into e2m3 * 2^(s-127) (s = UE8M0 byte)
// with exact bf16 multiplies: 2^(s-1) when s <= 128, else 2^127 then 2^(s-128)
// (every factor and product stays a bf16 value with at most 4 significant bits).
struct Fp6Mult {
    uint32_t m1, m2;
    bool two;
};

NVFP4_DEVINL Fp6Mult fp6_mult(uint32_t s)
{
    Fp6Mult r;
    r.two = s > 128u;
    const uint32_t b1 = ((r.two ? 127u : s - 1u) + 127u) << 7;  // s = 0 wraps to 2^-1
    const uint32_t b2 = ((s - 128u) + 127u) << 7;
    r.m1 = b1 | (b1 << 16);
    r.m2 = b2 | (b2 << 16);
    return r;
}

NVFP4_DEVINL uint32_t fp6_apply(uint32_t p, const Fp6Mult &m)
{
    p = bf16x2_mul(p, m.m1);
    return m.two ? bf16x2_mul(p, m.m2) : p;
}

// 8-k group q (0..3) of 32 consecutive codes held as 24 bytes (three uint2,
// little-endian 6-bit stream): bf16 pairs in natural k order, each value
// e2m3 * 2^(s-127).  Group q occupies bytes 6q .. 6q+5.
NVFP4_DEVINL uint4 fp6_group(const uint2 (&c)[3], int q, const Fp6Mult &mult)
{
    uint32_t lo, hi;
    if (q == 0) {
        lo = c[0].x;
        hi = c[0].y & 0xFFFFu;
    } else if (q == 1) {
        lo = (c[0].y >> 16) | (c[1].x << 16);
        hi = c[1].x >> 16;
    } else if (q == 2) {
        lo = c[1].y;
        hi = c[2].x & 0xFFFFu;
    } else {
        lo = (c[2].x >> 16) | (c[2].y << 16);
        hi = c[2].y >> 16;
    }
    const uint4 p = e2m3x8_to_bf16(lo, hi);
    return make_uint4(fp6_apply(p.x, mult), fp6_apply(p.y, mult), fp6_apply(p.z, mult), fp6_apply(p.w, mult));
}

}  // namespace nvfp4
