// The one e4m3 quantisation rule every FP8 writer uses (activations, weights,
// K/V vectors): a power-of-two scale 2^e, e the smallest integer with
// 448 * 2^e >= amax (e = 0 for an all-zero block), and each value's code the
// e4m3fn value nearest to v / 2^e (ties to even, saturating at 448, sign kept).
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 and §4.2 ask that
// rollout and training quantise by the same rule; sharing it makes that so.
#pragma once
#include <cuda_bf16.h>
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

// bf16 pair of the e4m3 values of two codes sitting in bytes 1 and 3 of x.
// s eeee mmm placed at bf16 bits 15 and 10..4 is the bf16 (-1)^s 2^(e-127)
// (1 + m/8), or (-1)^s 2^-126 (m/8) for e = 0 (a bf16 subnormal): in both cases
// exactly the e4m3 value times 2^-120, so one bf16x2 multiply by 2^120 (exact:
// a power of two, results in [2^-9, 448]) gives the value, branch-free.
__device__ __forceinline__ uint32_t e4m3_pair_to_bf16x2(uint32_t x) {
  const uint32_t bits = (x & 0x80008000u) | ((x >> 4) & 0x07F007F0u);
  __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&bits);
  v = __hmul2(v, __nv_bfloat162(__float2bfloat16_rn(0x1p120f), __float2bfloat16_rn(0x1p120f)));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// bf16 values (unscaled) of the four e4m3 codes in w: byte i -> element i, two
// per 32-bit word.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  return make_uint2(e4m3_pair_to_bf16x2(__byte_perm(w, 0u, 0x1404)),   // [0, b0, 0, b1]
                    e4m3_pair_to_bf16x2(__byte_perm(w, 0u, 0x3424)));  // [0, b2, 0, b3]
}

}  // namespace bi
