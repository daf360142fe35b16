// e4m3.cuh -- FP8 E4M3 conversions and the query scale rule of the
// quantised-K path (shared by its attention kernel and its commit).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace lucetree {
namespace e4m3 {

// two fp32 values -> two E4M3 codes, round to nearest even, saturating to
// +-448 (the callers keep |x| <= 448): lo -> low byte, hi -> high byte
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// two E4M3 codes (low byte first) -> two fp32 values (exact)
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t c) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// p with max * 2^p in (224, 448] (the quantised-K scale rule); 0 for max = 0
__device__ __forceinline__ int scale_exponent(float m) {
    if (!(m > 0.f)) return 0;
    int ex;
    const float mant = frexpf(m, &ex);  // m = mant * 2^ex, mant in [0.5, 1)
    return mant <= 0.875f ? 9 - ex : 8 - ex;
}

}  // namespace e4m3
}  // namespace lucetree
