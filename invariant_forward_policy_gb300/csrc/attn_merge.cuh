// The merge of a row's attention split partials (the split merge kernel's
// per-element arithmetic).
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.2: the splits of the KV
// range are absolute and merged in one fixed order, the same for every phase.
// Split s of a row holds (m_s, l_s, acc_s) of positions [512 s, 512 (s + 1));
// the output is sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), M = max_s m_s,
// every sum taken in ascending s.
#pragma once
#include "common.cuh"

namespace bi {

constexpr int kMergeBatch = 16;  // split records loaded ahead of the in-order accumulation

// M = max_s m_s in ascending s
__device__ __forceinline__ float merge_max(const float2* ml, int ns) {
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, ml[s].x);
  return M;
}
// weight of a split record
__device__ __forceinline__ float merge_weight(float m_s, float M) { return exp2f(__fsub_rn(m_s, M)); }
// one term of L or O: acc + v * w
__device__ __forceinline__ float merge_term(float acc, float v, float w) { return __fadd_rn(acc, __fmul_rn(v, w)); }

// Output element d of one (row, head) whose partials start at record `base`
// ((row * Hq + head) * nsplit) of part_o [.., hd] / part_ml [.., 2].
__device__ __forceinline__ float merge_split_element(const float* __restrict__ part_o,
                                                     const float* __restrict__ part_ml, int64_t base, int ns, int hd,
                                                     int d) {
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + base;
  const float* po = part_o + base * hd + d;
  const float M = merge_max(ml, ns);
  float L = 0.f, O = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kMergeBatch) {
    float2 r[kMergeBatch];
    float o[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const bool in = s0 + k < ns;
      r[k] = in ? ml[s0 + k] : make_float2(-INFINITY, 0.f);
      o[k] = in ? po[(int64_t)(s0 + k) * hd] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      if (s0 + k >= ns) break;
      const float w = merge_weight(r[k].x, M);
      L = merge_term(L, r[k].y, w);
      O = merge_term(O, o[k], w);
    }
  }
  return __fdiv_rn(O, L);
}

// Splits of a row at position pos (clamped to nsplit, which a position beyond
// the call's max_ctx bound would exceed: reported as a bad index)
__device__ __forceinline__ int merge_split_count(int pos, int split, int nsplit, int* status, bool report_it) {
  int ns = pos / split + 1;
  if (ns > nsplit) {
    if (report_it) report(status, DEV_BAD_INDEX);
    ns = nsplit;
  }
  return ns;
}

}  // namespace bi
