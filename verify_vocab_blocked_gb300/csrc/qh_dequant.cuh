// qh_dequant.cuh -- register-level unpack of packed affine codes into fp16
// pairs, shared by the weight-streaming and tensor-core kernels.
//
// w = scale * q + bias (page "mlx-bun 0.0.4 -> 0.0.6", src/train/flash-cce.ts,
// the kernels' dequant): the code q is placed in the mantissa of an fp16 with
// a magic exponent, the magic value is subtracted exactly, and one fp16 FMA
// forms scale * q + bias with a single rounding.
#pragma once

#include "qh_internal.cuh"

namespace qh {

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 x) { return *reinterpret_cast<uint32_t*>(&x); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }

// fp16 value x broadcast to both halves of a 32-bit register.
__device__ __forceinline__ uint32_t bcast_h(__half x) {
    const uint32_t r = __half_as_ushort(x);
    return __byte_perm(r, r, 0x1010);
}

// (M + q_lo, M + q_hi) -> (s*q_lo + b, s*q_hi + b), fp16, one rounding: the
// subtraction of the magic M (1024 or 64) is exact for integers q < 256.
// The magic constant is passed as its fp16x2 bit pattern so it stays a
// compile-time immediate (0x64006400 = (1024, 1024), 0x54005400 = (64, 64)).
__device__ __forceinline__ uint32_t affine(uint32_t magic_pair, uint32_t magic, __half2 s,
                                           __half2 b) {
    const __half2 q = __hsub2(u32_as_h2(magic_pair), u32_as_h2(magic));
    return h2_as_u32(__hfma2(q, s, b));
}

// 4-bit codes of one word as fp16 pairs (q_k, q_k+4), k = 0..3, without a
// shift per pair: codes in bits 0-3 of each 16-bit half become the mantissa
// of 1024 + q (magic 0x6400), codes in bits 4-7 the mantissa of 64 + q (magic
// 0x5400: exponent 2^6, mantissa step 16 -> 1).  One shift by 8 brings codes
// 2, 3, 6, 7 down to the same two positions.
__device__ __forceinline__ void deq4_word(uint32_t w, __half2 s, __half2 b, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = affine(lop3_and_or(w, 0x000F000Fu, 0x64006400u), 0x64006400u, s, b);
    p[1] = affine(lop3_and_or(w, 0x00F000F0u, 0x54005400u), 0x54005400u, s, b);
    p[2] = affine(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), 0x64006400u, s, b);
    p[3] = affine(lop3_and_or(w8, 0x00F000F0u, 0x54005400u), 0x54005400u, s, b);
}

// 8-bit codes: prmt builds (1024 + q_a, 1024 + q_b) from two bytes of w.
__device__ __forceinline__ uint32_t deq8(uint32_t w, uint32_t sel, __half2 s, __half2 b) {
    return affine(__byte_perm(w, 0x64646464u, sel), 0x64006400u, s, b);
}

// Same, with the broadcast scale and bias held as fp16x2 bit patterns.
__device__ __forceinline__ void deq4_word(uint32_t w, uint32_t s2, uint32_t b2, uint32_t (&p)[4]) {
    deq4_word(w, u32_as_h2(s2), u32_as_h2(b2), p);
}

__device__ __forceinline__ uint32_t deq8(uint32_t w, uint32_t sel, uint32_t s2, uint32_t b2) {
    return deq8(w, sel, u32_as_h2(s2), u32_as_h2(b2));
}

}  // namespace qh
