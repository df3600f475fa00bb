// Pieces of the block-FP8 layer the model driver runs (bi_model_config.fp8):
// RoPE with the FP8 K/V cache write, and SwiGLU with the quantisation of its
// output fused.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 (W8A8 block-FP8
// linear layers on both sides) and §4.2 (K and V make the same FP8 round trip
// in rollout and training: the same fused kernel writes them, the same
// dequantisation reads them).  The arithmetic is term for term that of the
// bf16 path: RoPE as in bi_rope_kv_write, K and V quantised exactly as
// bi_kv_fp8_write does, SwiGLU as the GEMM epilogue computes it, every
// quantisation by the one rule of fp8.cuh.
#include <cuda_fp8.h>

#include "common.cuh"
#include "fp8.cuh"

namespace bi {

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
    const int e = fp8_scale_exp(m);
    const int64_t slot = ((int64_t)b * Hkv + kh) * 64 + pos % 64;
    uint8_t* dst = (is_v ? v8 : k8) + slot * hd;
    for (int u = 0; u < nv; ++u)
      dst[col[u]] = (uint8_t)fp8_code(val[u], e);
    if (lane == 0) (is_v ? vs : ks)[slot] = ldexpf(1.f, e);
  }
}

__device__ __forceinline__ float silu_ref(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }

// SiLU(gate) x up with the activation quantisation fused (the SiLU-mul-quant
// step): a[t, j] = bf16(silu(g) u), g = g13[t, j], u = g13[t, F + j] (bf16), then
// the row's 1 x 128 blocks of a to e4m3 codes q and power-of-two scales qs.
// One warp per (row, block), 4 consecutive columns per lane.
__global__ void __launch_bounds__(256) swiglu_fp8_kernel(const __nv_bfloat16* __restrict__ g13, int64_t T,
                                                         int64_t F, uint8_t* __restrict__ q,
                                                         float* __restrict__ qs) {
  pdl_trigger();
  pdl_wait();
  const int64_t nb = F / 128;
  const int64_t blk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (blk >= T * nb) return;
  const int lane = threadIdx.x & 31;
  const int64_t t = blk / nb, c0 = (blk % nb) * 128 + lane * 4;
  const uint2 graw = *reinterpret_cast<const uint2*>(g13 + t * 2 * F + c0);
  const uint2 uraw = *reinterpret_cast<const uint2*>(g13 + t * 2 * F + F + c0);
  const uint32_t gw[2] = {graw.x, graw.y}, uw[2] = {uraw.x, uraw.y};
  float a[4];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float g = (i & 1) ? bf16hi(gw[i >> 1]) : bf16lo(gw[i >> 1]);
    const float u = (i & 1) ? bf16hi(uw[i >> 1]) : bf16lo(uw[i >> 1]);
    a[i] = bf2f(f2bf(__fmul_rn(silu_ref(g), u)));
    m = fmaxf(m, fabsf(a[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int e = fp8_scale_exp(m);
  if (lane == 0) qs[blk] = ldexpf(1.f, e);
  *reinterpret_cast<uint32_t*>(q + t * F + c0) =
      fp8_code(a[0], e) | fp8_code(a[1], e) << 8 | fp8_code(a[2], e) << 16 | fp8_code(a[3], e) << 24;
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

bi_status swiglu_fp8(const void* g13, int64_t T, int64_t F, void* q, float* qs, cudaStream_t st) {
  if (T == 0) return BI_OK;
  BI_REQUIRE(T > 0 && F > 0 && F % 128 == 0, "F must be a multiple of 128");
  BI_REQUIRE(g13 && q && qs, "null pointer");
  BI_REQUIRE(aligned16(g13) && ((uintptr_t)q & 3) == 0, "g13 must be 16-byte and q 4-byte aligned");
  const int64_t blocks = cdiv(T * (F / 128), 8);
  BI_REQUIRE(blocks <= 0x7fffffff, "too many rows");
  return launched(launch_pdl(swiglu_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                             static_cast<const __nv_bfloat16*>(g13), T, F, static_cast<uint8_t*>(q), qs),
                  "swiglu_fp8");
}

}  // namespace bi

extern "C" bi_status bi_swiglu_fp8(const void* g13, int64_t T, int64_t F, void* q, float* q_scale, void* stream) {
  return bi::swiglu_fp8(g13, T, F, q, q_scale, bi::as_stream(stream));
}
