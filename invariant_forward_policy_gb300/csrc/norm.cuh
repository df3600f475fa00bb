// The RMSNorm arithmetic of the norm kernels (plain, and with the FP8 quantisation
// of its output fused).
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §2 (a row's result depends on
// the row only) and §3.1 (RMSNorm is one of the forward operators whose values
// the inference kernels define).  Per row of d elements: r = bf16(residual + x)
// (or x), ss accumulated by norm_threads(d) "virtual threads", thread t over the
// 16-byte vectors t, t + nthr, ... element by element with one fma each, then a
// xor butterfly inside each warp of 32 virtual threads and the warps' sums added
// in warp order; inv = 1 / sqrt(ss / d + eps); y = bf16((r * inv) * g).
#pragma once
#include "common.cuh"

namespace bi {

// Virtual threads per row: d/8 (one vector each) capped at 256, at least 32,
// rounded up to a warp.  A function of d only.
__host__ __device__ constexpr int norm_threads(int64_t d) {
  return (int)((((d / 8) > 256 ? 256 : ((d / 8) < 32 ? 32 : (d / 8))) + 31) / 32 * 32);
}
constexpr int kNormMaxVec = 8;  // d <= 16384: at most 8 vectors per virtual thread

// r = bf16(res + x), elementwise over one vector of 8
__device__ __forceinline__ uint4 norm_residual_add(uint4 x, const uint4& res) {
  uint32_t* pa = reinterpret_cast<uint32_t*>(&x);
  const uint32_t* pb = reinterpret_cast<const uint32_t*>(&res);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = __fadd_rn(bf16lo(pb[j]), bf16lo(pa[j]));
    const float hi = __fadd_rn(bf16hi(pb[j]), bf16hi(pa[j]));
    pa[j] = pack_bf16x2(lo, hi);
  }
  return x;
}

// ss plus the squares of the vector's 8 elements, in element order
__device__ __forceinline__ float norm_ss_vec(const uint4& a, float ss) {
  const uint32_t* pa = reinterpret_cast<const uint32_t*>(&a);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = bf16lo(pa[j]), hi = bf16hi(pa[j]);
    ss = __fmaf_rn(lo, lo, ss);
    ss = __fmaf_rn(hi, hi, ss);
  }
  return ss;
}

// the fixed xor butterfly of one warp (every lane ends with the same sum)
__device__ __forceinline__ float norm_warp_sum(float ss) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return ss;
}

// 1 / sqrt(mean square + eps) from the sum of the warps' sums (taken in warp order)
__device__ __forceinline__ float norm_inv(float t, int d, float eps) {
  const float ms = __fdiv_rn(t, (float)d);
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// inv of a row from each thread's own sum of squares: the warps' butterflies,
// then thread 0 adds the warp sums in warp order.  Every thread of the block
// calls it; warp_ss holds blockDim / 32 floats, s_inv one.
__device__ __forceinline__ float norm_row_inv(float ss, int d, float eps, float* warp_ss, float* s_inv) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  ss = norm_warp_sum(ss);
  if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < nthr / 32; ++w) t += warp_ss[w];
    *s_inv = norm_inv(t, d, eps);
  }
  __syncthreads();
  return *s_inv;
}

// y = bf16((r * inv) * g) of one vector
__device__ __forceinline__ uint4 norm_apply(const uint4& r, const uint4& g, float inv) {
  const uint32_t* pa = reinterpret_cast<const uint32_t*>(&r);
  const uint32_t* pg = reinterpret_cast<const uint32_t*>(&g);
  uint4 o;
  uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = __fmul_rn(__fmul_rn(bf16lo(pa[j]), inv), bf16lo(pg[j]));
    const float hi = __fmul_rn(__fmul_rn(bf16hi(pa[j]), inv), bf16hi(pg[j]));
    po[j] = pack_bf16x2(lo, hi);
  }
  return o;
}

}  // namespace bi
