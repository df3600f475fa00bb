// Pieces of the block-FP8 layer the model driver runs (bi_model_config.fp8):
// RoPE with the FP8 K/V cache write, and the SwiGLU of an FP8 gate/up GEMM's
// bf16 output.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 (W8A8 block-FP8
// linear layers on both sides) and §4.2 (K and V make the same FP8 round trip
// in rollout and training: the same fused kernel writes them, the same
// dequantisation reads them).  The arithmetic is term for term that of the
// bf16 path: RoPE as in bi_rope_kv_write, K and V quantised exactly as
// bi_kv_fp8_write does, SwiGLU as the GEMM epilogue computes it.
#include <cuda_fp8.h>

#include "common.cuh"

namespace bi {

__device__ __forceinline__ int fp8_vec_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = ilogbf(amax);
  return amax <= ldexpf(1.75f, e) ? e - 8 : e - 7;
}

// One CTA per row, one warp per head at a time.  q heads: rotated, bf16, to
// q_out.  k heads: rotated, bf16, then e4m3 codes with a power-of-two scale per
// (row, head) into the row's page slot.  v heads: bf16 values quantised the same way.
__global__ void __launch_bounds__(256) rope_kv_write_fp8_kernel(
    const __nv_bfloat16* __restrict__ qkv, const int32_t* __restrict__ row_seq, const int32_t* __restrict__ row_pos,
    int Hq, int Hkv, int hd, const float* __restrict__ table, int64_t max_pos, const int32_t* __restrict__ block_table,
    int64_t max_blk, int64_t n_blocks, __nv_bfloat16* __restrict__ q_out, uint8_t* __restrict__ k8,
    float* __restrict__ ks, uint8_t* __restrict__ v8, float* __restrict__ vs, int* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pos = row_pos[row];
  const int seq = row_seq[row];
  if (pos < 0 || pos >= max_pos) {
    if (threadIdx.x == 0) report(status, DEV_BAD_INDEX);
    return;
  }
  const int32_t b = pos / 64 < max_blk ? block_table[(int64_t)seq * max_blk + pos / 64] : -1;
  const bool blk_ok = b >= 0 && b < n_blocks;
  if (!blk_ok && threadIdx.x == 0) report(status, DEV_BAD_INDEX);
  const int half = hd / 2, nq = Hq + 2 * Hkv;
  const __nv_bfloat16* src = qkv + row * (int64_t)nq * hd;
  const float* cs = table + pos * hd;
  for (int h = warp; h < nq; h += blockDim.x >> 5) {
    float val[4];  // this lane's values of the head: pairs (j, j + half) for q / k, plain for v
    int col[4];
    int nv = 0;
    if (h < Hq + Hkv) {
      for (int j = lane; j < half; j += 32) {
        const float x1 = bf2f(src[h * hd + j]);
        const float x2 = bf2f(src[h * hd + j + half]);
        const float c = cs[j], s = cs[half + j];
        val[nv] = bf2f(f2bf(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s))));
        col[nv++] = j;
        val[nv] = bf2f(f2bf(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s))));
        col[nv++] = j + half;
      }
    } else {
      for (int j = lane; j < hd; j += 32) {
        val[nv] = bf2f(src[h * hd + j]);
        col[nv++] = j;
      }
    }
    if (h < Hq) {
      __nv_bfloat16* dst = q_out + (row * Hq + h) * hd;
      for (int u = 0; u < nv; ++u) dst[col[u]] = f2bf(val[u]);
      continue;
    }
    float m = 0.f;
    for (int u = 0; u < nv; ++u) m = fmaxf(m, fabsf(val[u]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!blk_ok) continue;
    const bool is_v = h >= Hq + Hkv;
    const int kh = is_v ? h - Hq - Hkv : h - Hq;
    const int e = fp8_vec_scale_exp(m);
    const int64_t slot = ((int64_t)b * Hkv + kh) * 64 + pos % 64;
    uint8_t* dst = (is_v ? v8 : k8) + slot * hd;
    for (int u = 0; u < nv; ++u)
      dst[col[u]] = (uint8_t)__nv_cvt_float_to_fp8(ldexpf(val[u], -e), __NV_SATFINITE, __NV_E4M3);
    if (lane == 0) (is_v ? vs : ks)[slot] = ldexpf(1.f, e);
  }
}

__device__ __forceinline__ float silu_ref(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }

// act[t, j] = bf16(silu(g) u) with g = g13[t, j], u = g13[t, F + j] (both bf16).
__global__ void swiglu_rows_kernel(const __nv_bfloat16* __restrict__ g13, int64_t T, int64_t F,
                                   __nv_bfloat16* __restrict__ act) {
  pdl_trigger();
  pdl_wait();
  const int64_t n = T * F;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / F, j = i % F;
    const float g = bf2f(g13[t * 2 * F + j]);
    const float u = bf2f(g13[t * 2 * F + F + j]);
    act[i] = f2bf(__fmul_rn(silu_ref(g), u));
  }
}

bi_status rope_kv_write_fp8(const void* qkv, int64_t T, const int32_t* row_seq, const int32_t* row_pos, int Hq,
                            int Hkv, int hd, const float* table, int64_t max_pos, const int32_t* block_table,
                            int64_t max_blk, int64_t n_blocks, void* q_out, void* k8, float* ks, void* v8, float* vs,
                            cudaStream_t st) {
  if (T == 0) return BI_OK;
  BI_REQUIRE(T <= 0x7fffffff, "too many rows");
  return launched(launch_pdl(rope_kv_write_fp8_kernel, dim3((unsigned)T), dim3(256), 0, st,
                             static_cast<const __nv_bfloat16*>(qkv), row_seq, row_pos, Hq, Hkv, hd, table, max_pos,
                             block_table, max_blk, n_blocks, static_cast<__nv_bfloat16*>(q_out),
                             static_cast<uint8_t*>(k8), ks, static_cast<uint8_t*>(v8), vs, device_status_ptr()),
                  "rope_kv_write_fp8");
}

bi_status swiglu_rows(const void* g13, int64_t T, int64_t F, void* act, cudaStream_t st) {
  if (T == 0) return BI_OK;
  const int blocks = (int)std::min<int64_t>(cdiv(T * F, 256), 8 * (int64_t)num_sms());
  return launched(launch_pdl(swiglu_rows_kernel, dim3(blocks), dim3(256), 0, st,
                             static_cast<const __nv_bfloat16*>(g13), T, F, static_cast<__nv_bfloat16*>(act)),
                  "swiglu_rows");
}

}  // namespace bi
