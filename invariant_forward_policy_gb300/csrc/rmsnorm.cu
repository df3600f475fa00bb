// RMSNorm with optional fused residual add: one CTA per row, fixed reduction tree.
//
// Batch-invariance source: "vLLM Achieves Bitwise-Consistent RL Training ..."
// §2 (batch independence: the row result may not depend on batch-mates) and
// §3.1 (RMSNorm is a forward operator whose values come from this kernel on
// both the rollout and the training side).
#include "common.cuh"
#include "fp8.cuh"
#include "norm.cuh"

namespace bi {

// Threads per row: norm_threads(d) (norm.cuh); a thread walks its vectors with
// stride 8*blockDim, so the per-thread order depends on d only.

// Row r of y is the norm of row src(r) of x (+ residual), src(r) = idx ? idx[r] : r;
// x + residual goes to res_out (the residual rows themselves, or another buffer).
// kFp8: the bf16 output row is also quantised in 1 x 128 blocks into codes q and
// scales qs (the 16 threads holding a block's 16 vectors reduce its amax); y may
// then be null.
// kOut: res_out is a buffer of its own; otherwise the sum goes back to the residual rows.
template <bool kResidual, bool kFp8, bool kOut = false>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                      __nv_bfloat16* __restrict__ residual,
                                                      __nv_bfloat16* __restrict__ res_out,
                                                      const __nv_bfloat16* __restrict__ gamma,
                                                      __nv_bfloat16* __restrict__ y, int d, float eps,
                                                      const int32_t* __restrict__ idx, uint8_t* __restrict__ q,
                                                      float* __restrict__ qs) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int64_t src = idx ? (int64_t)idx[row] : row;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int nvec = d / 8;
  constexpr int kMaxVec = kNormMaxVec;
  uint4 sv[kMaxVec];
  float ss = 0.f;
  const uint4* xr = reinterpret_cast<const uint4*>(x + src * d);
  uint4* rr = reinterpret_cast<uint4*>(residual + src * d);
  uint4* ro = kOut ? reinterpret_cast<uint4*>(res_out + src * d) : rr;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int v = tid + i * nthr;
    if (v < nvec) {
      uint4 a = xr[v];
      if (kResidual) {
        a = norm_residual_add(a, rr[v]);
        ro[v] = a;
      }
      sv[i] = a;
      ss = norm_ss_vec(a, ss);
    }
  }
  // fixed xor-butterfly inside the warp, then warps summed in index order
  __shared__ float warp_ss[8];
  __shared__ float s_inv;
  const float inv = norm_row_inv(ss, d, eps, warp_ss, &s_inv);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    if (i * nthr >= nvec) break;  // the same for every thread of the block
    const int v = tid + i * nthr;
    const bool on = v < nvec;
    uint4 o = make_uint4(0, 0, 0, 0);
    if (on) {
      o = norm_apply(sv[i], gr[v], inv);
      if (y) reinterpret_cast<uint4*>(y + row * d)[v] = o;
    }
    if (kFp8) {
      // a 128-column block is 16 consecutive vectors held by 16 consecutive lanes
      const uint32_t* po = reinterpret_cast<const uint32_t*>(&o);
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16lo(po[j])), fabsf(bf16hi(po[j]))));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const int e = fp8_scale_exp(m);
      if (on) {
        uint2 c;
        c.x = fp8_code(bf16lo(po[0]), e) | fp8_code(bf16hi(po[0]), e) << 8 | fp8_code(bf16lo(po[1]), e) << 16 |
              fp8_code(bf16hi(po[1]), e) << 24;
        c.y = fp8_code(bf16lo(po[2]), e) | fp8_code(bf16hi(po[2]), e) << 8 | fp8_code(bf16lo(po[3]), e) << 16 |
              fp8_code(bf16hi(po[3]), e) << 24;
        reinterpret_cast<uint2*>(q + row * d)[v] = c;
        if ((v & 15) == 0) qs[row * (d / 128) + v / 16] = ldexpf(1.f, e);
      }
    }
  }
}

bi_status rmsnorm_rows(const void* x, void* residual, const void* gamma, void* y, int64_t rows, int64_t d, float eps,
                       const int32_t* idx, void* stream) {
  return rmsnorm_rows_to(x, residual, residual, gamma, y, rows, d, eps, idx, stream);
}

bi_status rmsnorm_rows_to(const void* x, const void* residual, void* res_out, const void* gamma, void* y, int64_t rows,
                          int64_t d, float eps, const int32_t* idx, void* stream) {
  BI_REQUIRE(rows >= 0, "rows < 0");
  if (rows == 0) return BI_OK;
  BI_REQUIRE(x && gamma && y, "null pointer");
  BI_REQUIRE(d >= 8 && d <= 16384 && d % 8 == 0, "d must be a multiple of 8 in [8, 16384]");
  BI_REQUIRE(!residual == !res_out, "residual and res_out go together");
  BI_REQUIRE(aligned16(x) && aligned16(gamma) && aligned16(y) && (!residual || (aligned16(residual) && aligned16(res_out))),
             "pointers must be 16-byte aligned");
  BI_REQUIRE(rows <= 0x7fffffff, "rows too large");
  const int thr = norm_threads(d);
  auto* xp = static_cast<const __nv_bfloat16*>(x);
  auto* rp = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(residual));  // written only in place
  auto* op = static_cast<__nv_bfloat16*>(res_out);
  auto* gp = static_cast<const __nv_bfloat16*>(gamma);
  auto* yp = static_cast<__nv_bfloat16*>(y);
  cudaError_t e;
  if (residual && res_out != residual)
    e = launch_pdl(rmsnorm_kernel<true, false, true>, dim3((unsigned)rows), dim3(thr), 0, as_stream(stream), xp, rp,
                   op, gp, yp, (int)d, eps, idx, nullptr, nullptr);
  else if (residual)
    e = launch_pdl(rmsnorm_kernel<true, false>, dim3((unsigned)rows), dim3(thr), 0, as_stream(stream), xp, rp,
                   static_cast<__nv_bfloat16*>(nullptr), gp, yp, (int)d, eps, idx, nullptr, nullptr);
  else
    e = launch_pdl(rmsnorm_kernel<false, false>, dim3((unsigned)rows), dim3(thr), 0, as_stream(stream), xp, rp,
                   static_cast<__nv_bfloat16*>(nullptr), gp, yp, (int)d, eps, idx, nullptr, nullptr);
  return launched(e, "rmsnorm_kernel");
}

bi_status rmsnorm_fp8_rows(const void* x, void* residual, const void* gamma, void* y, void* q, float* qs,
                           int64_t rows, int64_t d, float eps, void* stream) {
  BI_REQUIRE(rows >= 0, "rows < 0");
  if (rows == 0) return BI_OK;
  BI_REQUIRE(x && gamma && q && qs, "null pointer");
  BI_REQUIRE_SHAPE(d >= 128 && d <= 16384 && d % 128 == 0, "d must be a multiple of 128 in [128, 16384]");
  BI_REQUIRE(aligned16(x) && aligned16(gamma) && (!y || aligned16(y)) && (!residual || aligned16(residual)) &&
                 ((uintptr_t)q & 7) == 0,
             "x, gamma, y, residual must be 16-byte and q 8-byte aligned");
  BI_REQUIRE(rows <= 0x7fffffff, "rows too large");
  const int thr = norm_threads(d);
  auto* xp = static_cast<const __nv_bfloat16*>(x);
  auto* rp = static_cast<__nv_bfloat16*>(residual);
  auto* gp = static_cast<const __nv_bfloat16*>(gamma);
  auto* yp = static_cast<__nv_bfloat16*>(y);
  auto* qp = static_cast<uint8_t*>(q);
  cudaError_t e;
  if (residual)
    e = launch_pdl(rmsnorm_kernel<true, true>, dim3((unsigned)rows), dim3(thr), 0, as_stream(stream), xp, rp,
                   static_cast<__nv_bfloat16*>(nullptr), gp, yp, (int)d, eps, nullptr, qp, qs);
  else
    e = launch_pdl(rmsnorm_kernel<false, true>, dim3((unsigned)rows), dim3(thr), 0, as_stream(stream), xp, rp,
                   static_cast<__nv_bfloat16*>(nullptr), gp, yp, (int)d, eps, nullptr, qp, qs);
  return launched(e, "rmsnorm_fp8_kernel");
}

}  // namespace bi

extern "C" bi_status bi_rmsnorm(const void* x, void* residual, const void* gamma, void* y, int64_t rows, int64_t d,
                                float eps, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  return rmsnorm_rows(x, residual, gamma, y, rows, d, eps, nullptr, stream);
}

extern "C" bi_status bi_rmsnorm_fp8(const void* x, void* residual, const void* gamma, void* y, void* q,
                                    float* q_scale, int64_t rows, int64_t d, float eps, void* stream) {
  return bi::rmsnorm_fp8_rows(x, residual, gamma, y, q, q_scale, rows, d, eps, stream);
}
