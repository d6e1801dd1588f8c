// packed_f32.cuh -- Blackwell's packed binary32 add (add.rn.f32x2): two
// independent additions in one instruction, each rounded to nearest even on
// its own, so two values taken through the same steps side by side get the
// bits they would get one at a time.
//
// The products stay scalar (__fmul_rn, one rounding each) and one packed add
// folds two of them: 3 FP32 instructions per pair of multiply-adds instead of
// 4, the same per-lane operations and bits.  Packed multiplies are not used:
// ptxas has been measured fusing a packed multiply with a packed add into a
// fused multiply-add even with explicit round-to-nearest modifiers and
// -fmad=false.  Used by the GEMM's k-chains and by the exp, erfc and GeLU of
// fixed_math.cuh.
#pragma once

namespace repops {

using u64 = unsigned long long;

__device__ __forceinline__ u64 pack2(float lo, float hi) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(u64 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ u64 add2_rn(u64 a, u64 b) {
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// acc (two lanes) = (fl(acc.lo + fl(x0*y0)), fl(acc.hi + fl(x1*y1)))
__device__ __forceinline__ u64 fold2(u64 acc, float x0, float y0, float x1, float y1) {
    return add2_rn(acc, pack2(__fmul_rn(x0, y0), __fmul_rn(x1, y1)));
}

}  // namespace repops
