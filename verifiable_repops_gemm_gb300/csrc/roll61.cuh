// roll61.cuh -- arithmetic modulo the Mersenne prime P = 2^61 - 1 for the
// rolling hash of uint32 rows with base B = 2^32 + 15, without 64-bit
// multiplies.
//
// Because 2^61 = 1 (mod P), multiplying a value below 2^61 by 2^s is a
// rotation of its 61 bits by s.  With B = 2^32 + 2^4 - 1, the Horner step
// h * B therefore becomes two rotations and a subtraction; the word leaving
// the window, w * B^W with w < 2^32 and B^W a residue, needs one 32 x 32 and
// one 32 x 29 bit product.  Each sum below stays under 8P < 2^64 and is
// folded once at the end, so every function returns the canonical residue in
// [0, P): the values of plain modular arithmetic, whatever the grouping.
#pragma once

#include <cstdint>

namespace repops {
namespace roll61 {

constexpr uint64_t P = (uint64_t(1) << 61) - 1;
constexpr uint64_t BASE = (uint64_t(1) << 32) + 15;

// x * 2^S mod P, up to a multiple of P, for x < 2^61: the result is < 2^61
template <int S>
__host__ __device__ __forceinline__ uint64_t rot(uint64_t x) {
    return ((x << S) & P) | (x >> (61 - S));
}

// the residue of s < 2^64: fold bits 61..63 (2^61 = 1), then subtract P once
__host__ __device__ __forceinline__ uint64_t fold(uint64_t s) {
    s = (s & P) + (s >> 61);   // <= P + 7
    return s >= P ? s - P : s;
}

// w * c mod P up to a multiple of P, for w < 2^32 and c < 2^61: < 2P + 8
__host__ __device__ __forceinline__ uint64_t mul_word_lazy(uint32_t w, uint64_t c) {
    const uint64_t t0 = uint64_t(w) * uint32_t(c);                 // < 2^64
    const uint64_t t1 = uint64_t(w) * uint32_t(c >> 32);           // < 2^61
    return (t0 & P) + (t0 >> 61) + rot<32>(t1);
}

// one Horner step, (h * B + w) mod P, for h < P: the sum is < 3P + 2^32
__host__ __device__ __forceinline__ uint64_t push(uint64_t h, uint32_t w) {
    return fold(rot<32>(h) + rot<4>(h) + (P - h) + w);
}

// one slide of a window of W words, (h * B - w_out * B^W + w_in) mod P, for
// h < P and bw = B^W mod P: 4P - (w_out * bw, lazy) lies in (2P - 8, 4P], so
// the sum is < 7P + 2^32
__host__ __device__ __forceinline__ uint64_t slide(uint64_t h, uint32_t w_out, uint32_t w_in, uint64_t bw) {
    return fold(rot<32>(h) + rot<4>(h) + (P - h) + (4 * P - mul_word_lazy(w_out, bw)) + w_in);
}

}  // namespace roll61
}  // namespace repops
