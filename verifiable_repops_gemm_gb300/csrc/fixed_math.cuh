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

__device__ __forceinline__ float gelu_fixed(float x) {
    const float z = __fmul_rn(x, 0.707106769084930419921875f);
    // one erfc for either sign: no divergent branch
    const float e = erfc_pos(fabsf(z));
    const float phi2 = z >= 0.0f ? __fsub_rn(2.0f, e) : e;
    return __fmul_rn(__fmul_rn(0.5f, x), phi2);
}

}  // namespace repops
