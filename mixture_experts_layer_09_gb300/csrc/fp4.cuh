// fp4.cuh -- e2m1 (MXFP4) code expansion for the expert kernels (colibri PR #418, the fmt=7
// note of its Kimi K3 tier: e2m1 nibbles decoded through a table, one scale per 32 inputs).
//
// An e2m1 code (OCP Microscaling formats) holds the sign in bit 3, a 2-bit exponent (bits 2..1,
// bias 1) and a 1-bit mantissa (bit 0); the magnitudes of codes 0..7 are 0, 0.5, 1, 1.5, 2, 3,
// 4, 6.  The kernels read a code as the integer 2v (0, 1, 2, 3, 4, 6, 8, 12 and negatives) and
// the group scale is halved at upload, so the GEMV's integer dot products and the tensor arm's
// fp16 operands both hold the weights exactly.  The tables are byte permutes indexed by the
// 3-bit magnitude code (selector nibbles always below 8); the sign is applied separately.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// 2v as signed bytes for magnitude codes 0..3 (first word) and 4..7 (second word)
constexpr uint32_t kE2m1PosLo = 0x03020100u, kE2m1PosHi = 0x0C080604u;
constexpr uint32_t kE2m1NegLo = 0xFDFEFF00u, kE2m1NegHi = 0xF4F8FAFCu;
// high byte of fp16(2v) for magnitude codes 0..3 and 4..7 (the low byte is 0 for all of them)
constexpr uint32_t kE2m1HalfLo = 0x42403C00u, kE2m1HalfHi = 0x4A484644u;

// The four codes in the low 16 bits of c (code j in bits 4j..4j+3) as signed bytes 2v,
// byte j from code j.
__device__ __forceinline__ uint32_t e2m1x4_to_i8(uint32_t c) {
    const uint32_t sel = c & 0x7777u;
    const uint32_t pos = __byte_perm(kE2m1PosLo, kE2m1PosHi, sel);
    const uint32_t neg = __byte_perm(kE2m1NegLo, kE2m1NegHi, sel);
    const uint32_t msk = __byte_perm(0u, 0xFFFFFFFFu, (c >> 1) & 0x4444u);  // 0xFF where the sign is set
    return (pos & ~msk) | (neg & msk);
}

// Eight codes (column j of the word in bits 4j..4j+3) as signed bytes 2v, split like the int4
// nibbles: lo = columns 0, 2, 4, 6, hi = columns 1, 3, 5, 7.
__device__ __forceinline__ void e2m1x8_to_i8(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t a = e2m1x4_to_i8(w);        // columns 0..3
    const uint32_t b = e2m1x4_to_i8(w >> 16);  // columns 4..7
    lo = __byte_perm(a, b, 0x6420u);
    hi = __byte_perm(a, b, 0x7531u);
}

// Eight codes times one fp16 scale -> eight fp16 values in the K order
// [c0 c4 c1 c5 c2 c6 c3 c7] of the tensor arm's operands.  Each half2 takes its two high bytes
// from the table (selector nibbles 1 and 3; nibbles 0 and 2 pick table byte 0, which is 0)
// and its two sign bits from the codes.
__device__ __forceinline__ uint4 e2m1x8_to_f16(uint32_t w, __half2 s2) {
    const uint32_t hx = __byte_perm(kE2m1HalfLo, kE2m1HalfHi, ((w << 4) & 0x70u) | ((w >> 4) & 0x7000u)) |
                        ((w << 12) & 0x80008000u);  // c0, c4
    const uint32_t hy = __byte_perm(kE2m1HalfLo, kE2m1HalfHi, (w & 0x70u) | ((w >> 8) & 0x7000u)) |
                        ((w << 8) & 0x80008000u);   // c1, c5
    const uint32_t hz = __byte_perm(kE2m1HalfLo, kE2m1HalfHi, ((w >> 4) & 0x70u) | ((w >> 12) & 0x7000u)) |
                        ((w << 4) & 0x80008000u);   // c2, c6
    const uint32_t hw = __byte_perm(kE2m1HalfLo, kE2m1HalfHi, ((w >> 8) & 0x70u) | ((w >> 16) & 0x7000u)) |
                        (w & 0x80008000u);          // c3, c7
    uint4 out;
    __half2 v;
    v = __hmul2(*reinterpret_cast<const __half2*>(&hx), s2);
    out.x = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(*reinterpret_cast<const __half2*>(&hy), s2);
    out.y = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(*reinterpret_cast<const __half2*>(&hz), s2);
    out.z = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(*reinterpret_cast<const __half2*>(&hw), s2);
    out.w = *reinterpret_cast<uint32_t*>(&v);
    return out;
}

}  // namespace moe
