// hp_dequant.cuh -- 8-bit codes to bfloat16 for the dequantising gathers ("Block-Paged
// Layout -- Hurray Format Specification", Per-page-slot parameters, Per-scheme
// composition): exact integer-to-float conversion and the bfloat16 nearest the exact
// product (q - zero_point) * scale, used by the copy engine's dequantising mode
// (hp_copy.cu).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace hp {

// The bfloat16 nearest to the exact product q*s (ties to even).  The binary32
// product p = RN(q*s) rounds to the same bfloat16 as the exact value unless p is
// itself a bfloat16 midpoint (low 16 bits 0x8000): every midpoint is a binary32
// number, so a closer one cannot lie between q*s and p.  At a midpoint the sign of
// the exact residual q*s - p, which one fused multiply-add returns (the
// "TwoProduct" error-free transformation of Ogita, Rump and Oishi, "Accurate sum
// and dot product", 2005), decides the direction.
__device__ __forceinline__ unsigned dq_bf16(float q, float s)
{
    const float p = __fmul_rn(q, s);
    unsigned r = __bfloat16_as_ushort(__float2bfloat16_rn(p));
    const unsigned b = __float_as_uint(p);
    if ((b & 0xFFFFu) == 0x8000u && (b & 0x7F800000u) != 0x7F800000u) {
        const float e = __fmaf_rn(q, s, -p);
        if (e != 0.0f) r = (b >> 16) + (((e > 0.0f) == (p > 0.0f)) ? 1u : 0u);
    }
    return r;
}

// Quantization schemes of the dequantising gather; the copy kernel's Q template argument
// is scheme * 2 + (zero points present).
enum QScheme { kQSlot = 0, kQTensor = 1, kQHead = 2, kQDim = 3 };

// Byte k of w as a float, exactly: placed under the exponent of 2^23 a byte u reads
// 2^23 + u.  A signed byte x is first made x + 128 by flipping its sign bit.
__device__ __forceinline__ float byte_to_f32(uint32_t w, uint32_t k, float bias)
{
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u | k)) - bias;
}

// The eight 8-bit codes of q (signed or unsigned) as floats.
__device__ __forceinline__ void codes_to_f32(uint2 q, bool sgn, float f[8])
{
    const uint32_t flip = sgn ? 0x80808080u : 0u;
    const float bias = sgn ? 8388736.0f : 8388608.0f;  // 2^23 + 128, or 2^23
    const uint32_t w0 = q.x ^ flip, w1 = q.y ^ flip;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[k] = byte_to_f32(w0, k, bias);
        f[4 + k] = byte_to_f32(w1, k, bias);
    }
}

__device__ __forceinline__ float code_to_f32(unsigned char b, bool sgn)
{
    return sgn ? (float)(signed char)b : (float)b;
}

// Two fp32 values in one 64-bit register pair, for the packed f32x2 arithmetic (one
// instruction for two lanes' worth of IEEE round-to-nearest adds or multiplies).
using f32x2 = unsigned long long;
__device__ __forceinline__ f32x2 pack2(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The eight codes of q minus their zero points, times their scales, as eight bfloat16
// values, each the one nearest the exact product.  Each code is placed under the exponent
// of 2^23 (2^23 + u, or 2^23 + x + 128 for a signed x); one packed subtraction of
// (2^23 [+ 128] + zero point), exact because every operand and result is an integer below
// 2^24, leaves q - zp, and one packed multiply forms the two binary32 products that one
// packed conversion rounds.  A product whose low 16 bits are 0x8000 (a bfloat16 midpoint,
// found with a zero-halfword test over each packed pair) sends the group to dq_bf16.
__device__ __forceinline__ uint4 dequant8(uint2 q, bool sgn, const float zc[8], const float sc[8])
{
    const uint32_t flip = sgn ? 0x80808080u : 0u;
    const float bias = sgn ? 8388736.0f : 8388608.0f;  // 2^23 + 128, or 2^23
    const uint32_t w[2] = {q.x ^ flip, q.y ^ flip};
    float f[8], p[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t wk = w[k >> 1], b0 = (2 * k) & 3;
        const f32x2 x = pack2(__uint_as_float(__byte_perm(wk, 0x4B000000u, 0x7650u | b0)),
                              __uint_as_float(__byte_perm(wk, 0x4B000000u, 0x7650u | (b0 + 1))));
        const f32x2 v = sub2(x, pack2(bias + zc[2 * k], bias + zc[2 * k + 1]));
        unpack2(v, f[2 * k], f[2 * k + 1]);
        unpack2(mul2(v, pack2(sc[2 * k], sc[2 * k + 1])), p[2 * k], p[2 * k + 1]);
    }
    uint32_t o[4];
    uint32_t mid = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(p[2 * k], p[2 * k + 1]);
        o[k] = *reinterpret_cast<const uint32_t*>(&h);
        const uint32_t y =
            __byte_perm(__float_as_uint(p[2 * k]), __float_as_uint(p[2 * k + 1]), 0x5410u) ^
            0x80008000u;
        mid |= (y - 0x00010001u) & ~y & 0x80008000u;
    }
    if (mid) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = dq_bf16(f[2 * k], sc[2 * k]) | (dq_bf16(f[2 * k + 1], sc[2 * k + 1]) << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace hp
