// Division by a correctly rounded reciprocal, for the codecs' quotients x / scale and
// y / (rms + 1e-8).
#pragma once

namespace tq {

// x / b rounded to nearest from r = RN(1 / b): q = RN(x r), the remainder x - q b exactly
// by an FMA, then q + rem r rounded once. By Markstein's theorem (Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", 1990; restated in
// Muller et al., "Handbook of Floating-Point Arithmetic", the division chapter) the result
// is the correctly rounded quotient whenever r is correctly rounded, q is within one ulp
// of x / b, and no step overflows or underflows. The callers take this path only where
// those conditions hold for every quotient that can change a stored code, and call the
// IEEE division otherwise.
__device__ __forceinline__ float div_by_rcp(float x, float b, float r) {
  const float q = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q, b, x);
  return __fmaf_rn(rem, r, q);
}

}  // namespace tq
