// 4-bit KV codes to bf16 (sm_103a device helpers shared by the attention
// kernels).  A code c in [-7, 7] is stored as a two's-complement nibble; a
// token row of d codes (two per byte: byte j holds dims 2j in its low nibble
// and 2j + 1 in its high one) has one power-of-two exponent e, value c * 2^e.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

namespace kvp {
namespace {

// 4-bit codes to bf16 mma operands.  A code c in [-7, 7] stored as a
// two's-complement nibble u becomes bf16(136 + c) by placing u ^ 8 in the
// low mantissa bits of 128 (bits 0x4300); then fma(x, 2^e, -136 * 2^e) =
// c * 2^e exactly (one rounding of an exact, representable result) when
// 2^e and 136 * 2^e are normal bf16 numbers (-126 <= e <= 120); otherwise
// x - 136 = c (exact) and a multiply by 2^e.
__device__ __forceinline__ uint32_t bf16_exp2_bits(int e) {   // 2^e, e in [-127, 127]
    return e >= -126 ? (uint32_t)(e + 127) << 7 : 0x40u;
}
__device__ __forceinline__ uint32_t bf16_neg136_bits(int e) {   // -136 * 2^e, e in [-126, 120]
    return 0x8000u | ((uint32_t)(134 + e) << 7) | 0x08u;
}
// scale pair (2^ea, 2^eb) as bf16x2 with the -136 * 2^e pair packed above
// it: .x = scales, .y = constants (callers check the fused range)
__device__ __forceinline__ uint2 exp_pair2(int ea, int eb) {
    const int ca = min(max(ea, -126), 120), cb = min(max(eb, -126), 120);
    return make_uint2(bf16_exp2_bits(ea) | (bf16_exp2_bits(eb) << 16),
                      bf16_neg136_bits(ca) | (bf16_neg136_bits(cb) << 16));
}
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int i) {   // nibbles i and i + 4 as bf16(136 + c)
    return ((w >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
}
__device__ __forceinline__ uint32_t conv_pair(uint32_t x, uint2 sc, bool fused) {
    __nv_bfloat162 xv = *reinterpret_cast<__nv_bfloat162 *>(&x);
    const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162 *>(&sc.x);
    __nv_bfloat162 r;
    if (fused) {
        const __nv_bfloat162 c2 = *reinterpret_cast<const __nv_bfloat162 *>(&sc.y);
        r = __hfma2(xv, s2, c2);
    } else {
        const uint32_t k136 = 0x43084308u;
        r = __hmul2(__hsub2(xv, *reinterpret_cast<const __nv_bfloat162 *>(&k136)), s2);
    }
    return *reinterpret_cast<uint32_t *>(&r);
}
// One 32-bit word of codes (8 dims of one row, bytes b = dims 2b, 2b + 1)
// to four bf16 pairs v[i] = dims (2i, 2i + 1), times 2^e as packed in sc.
__device__ __forceinline__ void expand_word(uint32_t w, uint2 sc, bool fused, uint32_t (&v)[4]) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t pr = __byte_perm(lo, hi, b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12));
        v[b] = conv_pair((pr & 0x000F000Fu) ^ 0x43084308u, sc, fused);
    }
}

}  // namespace
}  // namespace kvp
