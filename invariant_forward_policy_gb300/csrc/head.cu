// Embedding gather, vocab-wide log-softmax + gather (+ greedy argmax), rollout bookkeeping.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §2: diff is measured on
// each sampled token's logprob and the discrete choices (here the greedy
// argmax) need a fixed tie-break; §3.1 lists "the final logprob" as a fused
// output of the forward.  The logprob kernel gives each row one CTA whose
// thread count depends on V only; every thread walks a fixed index stride
// keeping an online (max, sum-exp, argmax), and the threads are merged by a
// fixed xor-butterfly and then warps in index order.
#include <algorithm>

#include "common.cuh"

namespace bi {

__global__ void embed_kernel(const int32_t* __restrict__ ids, const __nv_bfloat16* __restrict__ table, int64_t V,
                             int64_t d, __nv_bfloat16* __restrict__ out, int* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t t = blockIdx.x;
  const int32_t id = ids[t];
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) report(status, DEV_BAD_INDEX);
  const uint4* src = reinterpret_cast<const uint4*>(table + (int64_t)(ok ? id : 0) * d);
  uint4* dst = reinterpret_cast<uint4*>(out + t * d);
  for (int64_t v = threadIdx.x; v < d / 8; v += blockDim.x) dst[v] = ok ? src[v] : make_uint4(0, 0, 0, 0);
}

struct LseState {
  float m, s, best;
  int idx;
};

__device__ __forceinline__ LseState lse_merge(const LseState& a, const LseState& b) {
  LseState r;
  r.m = fmaxf(a.m, b.m);
  if (r.m == -INFINITY) {
    r.s = 0.f;
  } else {
    const float ea = (a.m == r.m) ? 1.f : expf(__fsub_rn(a.m, r.m));
    const float eb = (b.m == r.m) ? 1.f : expf(__fsub_rn(b.m, r.m));
    r.s = __fadd_rn(__fmul_rn(a.s, ea), __fmul_rn(b.s, eb));
  }
  if (a.best > b.best || (a.best == b.best && a.idx < b.idx)) {
    r.best = a.best;
    r.idx = a.idx;
  } else {
    r.best = b.best;
    r.idx = b.idx;
  }
  return r;
}

__device__ __forceinline__ void lse_step4(LseState& st, float4 x, int base) {
  const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
  if (mx > st.m) {
    st.s = (st.m == -INFINITY) ? 0.f : __fmul_rn(st.s, expf(__fsub_rn(st.m, mx)));
    st.m = mx;
  }
  st.s = __fadd_rn(st.s, expf(__fsub_rn(x.x, st.m)));
  st.s = __fadd_rn(st.s, expf(__fsub_rn(x.y, st.m)));
  st.s = __fadd_rn(st.s, expf(__fsub_rn(x.z, st.m)));
  st.s = __fadd_rn(st.s, expf(__fsub_rn(x.w, st.m)));
  if (x.x > st.best) { st.best = x.x; st.idx = base; }
  if (x.y > st.best) { st.best = x.y; st.idx = base + 1; }
  if (x.z > st.best) { st.best = x.z; st.idx = base + 2; }
  if (x.w > st.best) { st.best = x.w; st.idx = base + 3; }
}

// Reduce over the CTA: butterfly inside warps, then warps 0..W-1 in order.
template <int NT>
__device__ __forceinline__ LseState lse_block_reduce(LseState st) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    LseState b;
    b.m = __shfl_xor_sync(0xffffffffu, st.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, st.s, o);
    b.best = __shfl_xor_sync(0xffffffffu, st.best, o);
    b.idx = __shfl_xor_sync(0xffffffffu, st.idx, o);
    st = lse_merge(st, b);
  }
  __shared__ LseState ws[NT / 32];
  __shared__ LseState total;
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    LseState r = ws[0];
    for (int w = 1; w < NT / 32; ++w) r = lse_merge(r, ws[w]);
    total = r;
  }
  __syncthreads();
  return total;
}

__device__ __forceinline__ LseState lse_init() { return LseState{-INFINITY, 0.f, -INFINITY, 0x7fffffff}; }

// Visit x4[v] for v = v0, v0 + NT, ... < end in that order; the loads of four
// consecutive visits are issued before any of them is used.
template <int NT>
__device__ __forceinline__ void lse_walk(LseState& st, const float4* __restrict__ x4, int64_t v0, int64_t end) {
  constexpr int U = 4;
  for (; v0 < end; v0 += (int64_t)NT * U) {
    float4 xs[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + (int64_t)u * NT;
      if (v < end) xs[u] = __ldg(x4 + v);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + (int64_t)u * NT;
      if (v < end) lse_step4(st, xs[u], (int)(v * 4));
    }
  }
}

// One CTA per row (invariant path).  Results go to index dst[row] (or row).
template <int NT>
__global__ void __launch_bounds__(NT) logprob_kernel(const float* __restrict__ logits, const int32_t* __restrict__ ids,
                                                     int64_t V, float* __restrict__ lp_out,
                                                     int32_t* __restrict__ argmax_out, const int32_t* __restrict__ dst,
                                                     int* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const float4* x4 = reinterpret_cast<const float4*>(logits + row * V);
  const int64_t n4 = V / 4;
  LseState st = lse_init();
  lse_walk<NT>(st, x4, threadIdx.x, n4);
  st = lse_block_reduce<NT>(st);
  if (threadIdx.x == 0) {
    int32_t id = st.idx;
    if (ids) {
      id = ids[row];
      if (id < 0 || id >= V) {
        report(status, DEV_BAD_INDEX);
        id = st.idx;
      }
    }
    const float xid = logits[row * V + id];
    const int64_t o = dst ? (int64_t)dst[row] : row;
    lp_out[o] = __fsub_rn(__fsub_rn(xid, st.m), logf(st.s));
    if (argmax_out) argmax_out[o] = st.idx;
  }
}

// BI_FAST: the vocab of each row is split over `chunks` CTAs (chosen from T),
// then merged.  Results depend on T (not batch invariant).
template <int NT>
__global__ void __launch_bounds__(NT) logprob_partial_kernel(const float* __restrict__ logits, int64_t V, int chunks,
                                                             LseState* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x / chunks;
  const int c = blockIdx.x % chunks;
  const int64_t n4 = V / 4;
  const int64_t per = (n4 + chunks - 1) / chunks;
  const int64_t b = c * per, e = min(n4, b + per);
  const float4* x4 = reinterpret_cast<const float4*>(logits + row * V);
  LseState st = lse_init();
  lse_walk<NT>(st, x4, b + threadIdx.x, e);
  st = lse_block_reduce<NT>(st);
  if (threadIdx.x == 0) part[blockIdx.x] = st;
}

__global__ void logprob_combine_kernel(const float* __restrict__ logits, const int32_t* __restrict__ ids, int64_t V,
                                       int chunks, const LseState* __restrict__ part, float* __restrict__ lp_out,
                                       int32_t* __restrict__ argmax_out, const int32_t* __restrict__ dst, int64_t T) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (row >= T) return;
  LseState st = part[row * chunks];
  for (int c = 1; c < chunks; ++c) st = lse_merge(st, part[row * chunks + c]);
  int32_t id = st.idx;
  if (ids) {
    id = ids[row];
    if (id < 0 || id >= V) id = st.idx;
  }
  const int64_t o = dst ? (int64_t)dst[row] : row;
  lp_out[o] = __fsub_rn(__fsub_rn(logits[row * V + id], st.m), logf(st.s));
  if (argmax_out) argmax_out[o] = st.idx;
}

// Fused head: merge the vocab-tile partials of one row, thread t taking tiles
// t, t + 128, ... in order, then the fixed butterfly / warp-order tree.
__global__ void __launch_bounds__(128) lse_tiles_merge_kernel(const TileLse* __restrict__ part, int n_tiles,
                                                              int tile_n, const int32_t* __restrict__ ids,
                                                              float* __restrict__ lp_out,
                                                              int32_t* __restrict__ argmax_out,
                                                              const int32_t* __restrict__ dst, int* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const TileLse* pr = part + row * n_tiles;
  LseState st = lse_init();
  for (int t = threadIdx.x; t < n_tiles; t += 128) {
    const TileLse q = pr[t];
    st = lse_merge(st, LseState{q.m, q.s, q.best, q.idx});
  }
  st = lse_block_reduce<128>(st);
  if (threadIdx.x == 0) {
    float xt = st.best;
    if (ids) {
      int32_t id = ids[row];
      if (id < 0 || id / tile_n >= n_tiles) {
        report(status, DEV_BAD_INDEX);
      } else {
        xt = pr[id / tile_n].xt;
      }
    }
    const int64_t o = dst ? (int64_t)dst[row] : row;
    lp_out[o] = __fsub_rn(__fsub_rn(xt, st.m), logf(st.s));
    if (argmax_out) argmax_out[o] = st.idx;
  }
}

bi_status lse_tiles_merge(const TileLse* part, int64_t T, int n_tiles, int tile_n, const int32_t* ids,
                          float* logprob_out, int32_t* argmax_out, const int32_t* dst, void* stream) {
  if (T == 0) return BI_OK;
  return launched(launch_pdl(lse_tiles_merge_kernel, dim3((unsigned)T), dim3(128), 0, as_stream(stream), part, n_tiles,
                             tile_n, ids, logprob_out, argmax_out, dst, device_status_ptr()),
                  "lse_tiles_merge_kernel");
}

static int fast_chunks(int64_t T, int64_t V) {
  if (T >= num_sms()) return 1;
  int64_t c = cdiv(2 * (int64_t)num_sms(), T);
  c = std::min<int64_t>(c, std::max<int64_t>(1, V / 4096));
  return (int)std::max<int64_t>(c, 1);
}

// One CTA: record the step, feed the sampled tokens back, advance positions and the step counter.
__global__ void decode_advance_kernel(const int32_t* __restrict__ sampled, const float* __restrict__ lp,
                                      int32_t* __restrict__ tokens, int32_t* __restrict__ pos, int64_t B,
                                      int32_t* __restrict__ step_counter, int32_t* __restrict__ hist_ids,
                                      float* __restrict__ hist_lp, int64_t max_steps, int* status) {
  pdl_trigger();
  pdl_wait();
  const int32_t step = *step_counter;
  const bool in_range = step >= 0 && step < max_steps;
  for (int64_t b = threadIdx.x; b < B; b += blockDim.x) {
    if (in_range) {
      hist_ids[(int64_t)step * B + b] = sampled[b];
      hist_lp[(int64_t)step * B + b] = lp[b];
    }
    tokens[b] = sampled[b];
    pos[b] = pos[b] + 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!in_range) report(status, DEV_BAD_INDEX);
    *step_counter = step + 1;
  }
}

bi_status logprob_gather_to(const float* logits, const int32_t* ids, int64_t T, int64_t V, float* logprob_out,
                            int32_t* argmax_out, const int32_t* dst, int mode, void* workspace, size_t ws_bytes,
                            void* stream) {
  BI_REQUIRE(T >= 0, "T < 0");
  if (T == 0) return BI_OK;
  BI_REQUIRE(logits && logprob_out, "null pointer");
  BI_REQUIRE(V >= 4 && V % 4 == 0 && V < (1ll << 31), "V must be a multiple of 4");
  BI_REQUIRE(aligned16(logits), "logits must be 16-byte aligned");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  BI_REQUIRE(T <= 0x7fffffff, "T too large");
  cudaStream_t st = as_stream(stream);
  const int chunks = mode == BI_FAST ? fast_chunks(T, V) : 1;
  if (chunks > 1) {
    BI_REQUIRE(workspace && ws_bytes >= (size_t)T * chunks * sizeof(LseState),
               "BI_FAST logprob needs workspace (bi_logprob_workspace_size)");
    auto* part = static_cast<LseState*>(workspace);
    BI_TRY(launched(launch_pdl(logprob_partial_kernel<256>, dim3((unsigned)(T * chunks)), dim3(256), 0, st, logits,
                               V, chunks, part),
                    "logprob_partial_kernel"));
    return launched(launch_pdl(logprob_combine_kernel, dim3((unsigned)cdiv(T, 128)), dim3(128), 0, st, logits, ids, V,
                               chunks, (const LseState*)part, logprob_out, argmax_out, dst, T),
                    "logprob_combine_kernel");
  }
  if (V <= 16384)
    return launched(launch_pdl(logprob_kernel<256>, dim3((unsigned)T), dim3(256), 0, st, logits, ids, V, logprob_out,
                               argmax_out, dst, device_status_ptr()),
                    "logprob_kernel");
  return launched(launch_pdl(logprob_kernel<512>, dim3((unsigned)T), dim3(512), 0, st, logits, ids, V, logprob_out,
                             argmax_out, dst, device_status_ptr()),
                  "logprob_kernel");
}

}  // namespace bi

extern "C" {

bi_status bi_embed(const int32_t* ids, int64_t T, const void* table, int64_t V, int64_t d, void* out, void* stream) {
  using namespace bi;
  BI_REQUIRE(T >= 0, "T < 0");
  if (T == 0) return BI_OK;
  BI_REQUIRE(ids && table && out, "null pointer");
  BI_REQUIRE(V > 0 && d > 0 && d % 8 == 0, "d must be a multiple of 8");
  BI_REQUIRE(aligned16(table) && aligned16(out), "pointers must be 16-byte aligned");
  BI_REQUIRE(T <= 0x7fffffff, "T too large");
  return launched(launch_pdl(embed_kernel, dim3((unsigned)T), dim3(128), 0, as_stream(stream), ids,
                             static_cast<const __nv_bfloat16*>(table), V, d, static_cast<__nv_bfloat16*>(out),
                             device_status_ptr()),
                  "bi_embed");
}

size_t bi_logprob_workspace_size(int64_t T, int64_t V, int mode) {
  if (mode != BI_FAST || T <= 0) return 0;
  return (size_t)T * bi::fast_chunks(T, V) * sizeof(bi::LseState);
}

bi_status bi_logprob_gather(const float* logits, const int32_t* ids, int64_t T, int64_t V, float* logprob_out,
                            int32_t* argmax_out, int mode, void* workspace, size_t ws_bytes, void* stream) {
  return bi::logprob_gather_to(logits, ids, T, V, logprob_out, argmax_out, nullptr, mode, workspace, ws_bytes, stream);
}

bi_status bi_decode_advance(const int32_t* sampled, const float* logprob, int32_t* tokens, int32_t* pos, int64_t B,
                            int32_t* step_counter, int32_t* hist_ids, float* hist_lp, int64_t max_steps,
                            void* stream) {
  using namespace bi;
  BI_REQUIRE(B >= 0, "B < 0");
  if (B == 0) return BI_OK;
  BI_REQUIRE(sampled && logprob && tokens && pos && step_counter && hist_ids && hist_lp, "null pointer");
  BI_REQUIRE(max_steps > 0, "max_steps <= 0");
  return launched(launch_pdl(decode_advance_kernel, dim3(1), dim3(256), 0, as_stream(stream), sampled, logprob, tokens,
                             pos, B, step_counter, hist_ids, hist_lp, max_steps, device_status_ptr()),
                  "decode_advance_kernel");
}

}  // extern "C"
