// fixed_math.cuh -- the library's own exp, erfc and GeLU: every operation one
// IEEE binary32 rounding in a fixed order, so the bits are the same on any
// hardware (CUDA's expf/erfcf are not specified to the bit).
//
// "Verde与RepOps" §3.3 and §4.3 name GeLU and ERF among the operators that need
// a reproducible form; the pages fix no algorithm, so:
//   - exp(x): k = rint(x * log2 e); r = (x - k*ln2_hi) - k*ln2_lo (Cody and
//     Waite's two-part ln 2, k*ln2_hi exact); e^r by the degree-7 Taylor
//     polynomial in Horner form; times 2^k by exact power-of-two scaling;
//   - erfc(z), z >= 0: the Chebyshev fit of Numerical Recipes §6.2 (Press,
//     Teukolsky, Vetterling, Flannery), with the exp above;
//   - GeLU(x) = 0.5*x*(1 + erf(x/sqrt 2)) with 1 + erf(z) = 2 - erfc(z) for
//     z >= 0 and erfc(-z) for z < 0.
// Used by the row operators and by the GEMM epilogue.
#pragma once

#include "packed_f32.cuh"

namespace repops {

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

__device__ inline float exp_fixed(float x) {
    if (x != x) return x;
    if (x > 88.72283935546875f) return __int_as_float(0x7f800000);
    if (x < -103.972084045410156f) return 0.0f;
    const float t = __fmul_rn(x, 1.44269502162933349609375f);
    // k = rint(t), ties to even: adding 1.5 * 2^23 leaves rint(t) in the low
    // mantissa bits (exact for |t| < 2^22; past the checks above |t| < 151),
    // and subtracting it back is exact
    const float big = __fadd_rn(t, 12582912.0f);
    const float kf = __fsub_rn(big, 12582912.0f);
    const int k = __float_as_int(big) - 0x4B400000;
    float r = __fsub_rn(x, __fmul_rn(kf, 0.693145751953125f));
    r = __fsub_rn(r, __fmul_rn(kf, 1.428606765330187045037746e-06f));
    float p = 1.98412701e-04f;
    p = __fadd_rn(__fmul_rn(p, r), 1.38888892e-03f);
    p = __fadd_rn(__fmul_rn(p, r), 8.33333377e-03f);
    p = __fadd_rn(__fmul_rn(p, r), 4.16666679e-02f);
    p = __fadd_rn(__fmul_rn(p, r), 1.66666672e-01f);
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    // p * 2^k as (p * 2^k1) * 2^k2: k1 = 127, k2 = k - 127 above the normal
    // range; k1 = k + 64, k2 = -64 below it (one rounding, at the end); else
    // k1 = k and the second factor is 1 (exact).  Selects, not branches.
    const int k2 = k > 127 ? k - 127 : (k < -126 ? -64 : 0);
    return __fmul_rn(__fmul_rn(p, pow2i(k - k2)), pow2i(k2));
}

__device__ inline float erfc_pos(float z) {
    // correctly rounded reciprocal: the same value as a correctly rounded 1/x
    const float t = __frcp_rn(__fadd_rn(1.0f, __fmul_rn(0.5f, z)));
    float q = 0.17087277f;
    q = __fadd_rn(__fmul_rn(q, t), -0.82215223f);
    q = __fadd_rn(__fmul_rn(q, t), 1.48851587f);
    q = __fadd_rn(__fmul_rn(q, t), -1.13520398f);
    q = __fadd_rn(__fmul_rn(q, t), 0.27886807f);
    q = __fadd_rn(__fmul_rn(q, t), -0.18628806f);
    q = __fadd_rn(__fmul_rn(q, t), 0.09678418f);
    q = __fadd_rn(__fmul_rn(q, t), 0.37409196f);
    q = __fadd_rn(__fmul_rn(q, t), 1.00002368f);
    q = __fmul_rn(q, t);
    const float zz = __fmul_rn(z, z);
    const float arg = __fadd_rn(__fadd_rn(-zz, -1.26551223f), q);
    return __fmul_rn(t, exp_fixed(arg));
}

// ---------------------------------------------------------------- pairs ----
// The same functions for two arguments at once: each lane goes through exactly
// the steps above (x - y computed as x + (-y) and fl(k * -c) as -fl(k * c), both
// exact identities of IEEE rounding to nearest), with every pair of additions
// issued as one packed add (packed_f32.cuh): the same bits, fewer instructions.

__device__ __forceinline__ void horner2(float &p0, float &p1, float r0, float r1, float c) {
    unpack2(add2_rn(pack2(__fmul_rn(p0, r0), __fmul_rn(p1, r1)), pack2(c, c)), p0, p1);
}

__device__ __forceinline__ float exp_finish(float x, float p, int k) {
    const int k2 = k > 127 ? k - 127 : (k < -126 ? -64 : 0);
    const float v = __fmul_rn(__fmul_rn(p, pow2i(k - k2)), pow2i(k2));
    return x != x ? x : (x > 88.72283935546875f ? __int_as_float(0x7f800000) : (x < -103.972084045410156f ? 0.0f : v));
}

__device__ inline float2 exp_fixed2(float x0, float x1) {
    float big0, big1, kf0, kf1, r0, r1;
    unpack2(add2_rn(pack2(__fmul_rn(x0, 1.44269502162933349609375f), __fmul_rn(x1, 1.44269502162933349609375f)),
                    pack2(12582912.0f, 12582912.0f)), big0, big1);
    unpack2(add2_rn(pack2(big0, big1), pack2(-12582912.0f, -12582912.0f)), kf0, kf1);
    const int k0 = __float_as_int(big0) - 0x4B400000, k1 = __float_as_int(big1) - 0x4B400000;
    unpack2(add2_rn(pack2(x0, x1), pack2(__fmul_rn(kf0, -0.693145751953125f), __fmul_rn(kf1, -0.693145751953125f))),
            r0, r1);
    unpack2(add2_rn(pack2(r0, r1), pack2(__fmul_rn(kf0, -1.428606765330187045037746e-06f),
                                         __fmul_rn(kf1, -1.428606765330187045037746e-06f))),
            r0, r1);
    float p0 = 1.98412701e-04f, p1 = 1.98412701e-04f;
    horner2(p0, p1, r0, r1, 1.38888892e-03f);
    horner2(p0, p1, r0, r1, 8.33333377e-03f);
    horner2(p0, p1, r0, r1, 4.16666679e-02f);
    horner2(p0, p1, r0, r1, 1.66666672e-01f);
    horner2(p0, p1, r0, r1, 0.5f);
    horner2(p0, p1, r0, r1, 1.0f);
    horner2(p0, p1, r0, r1, 1.0f);
    return make_float2(exp_finish(x0, p0, k0), exp_finish(x1, p1, k1));
}

__device__ inline float2 erfc_pos2(float z0, float z1) {
    float d0, d1;
    unpack2(add2_rn(pack2(1.0f, 1.0f), pack2(__fmul_rn(0.5f, z0), __fmul_rn(0.5f, z1))), d0, d1);
    const float t0 = __frcp_rn(d0), t1 = __frcp_rn(d1);
    float q0 = 0.17087277f, q1 = 0.17087277f;
    horner2(q0, q1, t0, t1, -0.82215223f);
    horner2(q0, q1, t0, t1, 1.48851587f);
    horner2(q0, q1, t0, t1, -1.13520398f);
    horner2(q0, q1, t0, t1, 0.27886807f);
    horner2(q0, q1, t0, t1, -0.18628806f);
    horner2(q0, q1, t0, t1, 0.09678418f);
    horner2(q0, q1, t0, t1, 0.37409196f);
    horner2(q0, q1, t0, t1, 1.00002368f);
    q0 = __fmul_rn(q0, t0);
    q1 = __fmul_rn(q1, t1);
    float a0, a1;
    unpack2(add2_rn(pack2(-__fmul_rn(z0, z0), -__fmul_rn(z1, z1)), pack2(-1.26551223f, -1.26551223f)), a0, a1);
    unpack2(add2_rn(pack2(a0, a1), pack2(q0, q1)), a0, a1);
    const float2 e = exp_fixed2(a0, a1);
    return make_float2(__fmul_rn(t0, e.x), __fmul_rn(t1, e.y));
}

__device__ __forceinline__ float2 gelu_fixed2(float x0, float x1) {
    const float z0 = __fmul_rn(x0, 0.707106769084930419921875f), z1 = __fmul_rn(x1, 0.707106769084930419921875f);
    const float2 e = erfc_pos2(fabsf(z0), fabsf(z1));
    const float phi0 = z0 >= 0.0f ? __fsub_rn(2.0f, e.x) : e.x;
    const float phi1 = z1 >= 0.0f ? __fsub_rn(2.0f, e.y) : e.y;
    return make_float2(__fmul_rn(__fmul_rn(0.5f, x0), phi0), __fmul_rn(__fmul_rn(0.5f, x1), phi1));
}

__device__ __forceinline__ float gelu_fixed(float x) {
    const float z = __fmul_rn(x, 0.707106769084930419921875f);
    // one erfc for either sign: no divergent branch
    const float e = erfc_pos(fabsf(z));
    const float phi2 = z >= 0.0f ? __fsub_rn(2.0f, e) : e;
    return __fmul_rn(__fmul_rn(0.5f, x), phi2);
}

}  // namespace repops
