// The one e4m3 quantisation rule every FP8 writer uses (activations, weights,
// K/V vectors): a power-of-two scale 2^e, e the smallest integer with
// 448 * 2^e >= amax (e = 0 for an all-zero block), and each value's code the
// e4m3fn value nearest to v / 2^e (ties to even, saturating at 448, sign kept).
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 and §4.2 ask that
// rollout and training quantise by the same rule; sharing it makes that so.
#pragma once
#include <cuda_fp8.h>

#include <cstdint>

namespace bi {

__device__ __forceinline__ int fp8_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = ilogbf(amax);  // amax in [2^e, 2^(e+1))
  return amax <= ldexpf(1.75f, e) ? e - 8 : e - 7;
}

__device__ __forceinline__ uint32_t fp8_code(float v, int e) {
  return (uint32_t)__nv_cvt_float_to_fp8(ldexpf(v, -e), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace bi
