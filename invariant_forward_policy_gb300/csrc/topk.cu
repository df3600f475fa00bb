// Deterministic Top-K with a unique (score, in-request position) key.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.3 ("Top-K in sparse
// attention: fix ties and order"): a default Top-K breaks ties by thread
// scheduling; the consistent one makes the key unique by appending the
// candidate's in-request position to the score bits, so a tie goes to the
// larger position, and returns the selected positions sorted by descending
// position with invalid entries last.
//
// With few rows, a row is split over a cluster of kTopkCluster CTAs (with many
// rows, one CTA takes a whole row the same way), CTA r holding the r-th
// contiguous chunk of positions (its keys cached in shared memory when the
// chunk fits).  The score of every candidate maps to an order-preserving
// 32-bit key (-0 first made +0, so equal scores give equal keys).  A 4-pass
// 8-bit radix select finds the exact key of the K-th largest score and how
// many candidates holding exactly that key belong to the selection (kk): each
// CTA histograms its chunk, then every CTA sums the cluster's histograms
// through distributed shared memory (integer sums, the same in every CTA) and
// takes the same decision.  The output pass walks positions from the top: a
// CTA learns from the higher chunks how many keys above the threshold and how
// many ties they hold, then walks its own chunk downward in tiles, prefix-
// summing per-thread counts over the block, and writes each selected position
// to its final slot.  A key above the threshold is always selected, a key equal
// to it while fewer than kk of those lie at higher positions; so the output is
// in descending position order without a sort.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace bi {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCluster = 8;
constexpr int kTopkMaxK = 4096;
constexpr int kTopkChunkKeys = 32 * 1024;  // chunks up to this many positions are cached in shared memory
constexpr int kTopkRowThreads = 512;       // one-CTA-per-row kernel
constexpr int kTopkRowWarps = kTopkRowThreads / 32;

__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one packed value per thread (thread 0 first);
// returns the exclusive prefix and writes the block total to *total.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_sum(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? warp_sums[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    if (lane < kWarps) warp_sums[lane] = wi - w;  // exclusive over warps
    if (lane == kWarps - 1) *total = wi;
  }
  __syncthreads();
  const uint32_t r = warp_sums[warp] + inc - v;
  __syncthreads();  // warp_sums is reused by the next call
  return r;
}

// Rows that alone fill the GPU: one CTA per row, the row re-read from L2 by
// each radix pass, the same selection and ordered write as below.
template <bool FAST>
__global__ void __launch_bounds__(kTopkRowThreads) topk_row_kernel(const float* __restrict__ scores, int64_t ld,
                                                            const int32_t* __restrict__ n_valid, int K,
                                                            int32_t* __restrict__ out, int* status) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[kTopkRowWarps];
  __shared__ uint32_t s_prefix, s_kk, s_total;
  __shared__ int s_slot_gt, s_slot_tie;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const float* s = scores + row * ld;
  int32_t* o = out + row * (int64_t)K;
  int64_t n = n_valid[row];
  if (n < 0 || n > ld) {
    if (tid == 0) report(status, DEV_BAD_INDEX);
    n = n < 0 ? 0 : ld;
  }
  if (n <= K) {  // every candidate is selected
    for (int i = tid; i < K; i += kTopkRowThreads) o[i] = i < n ? (int32_t)(n - 1 - i) : -1;
    return;
  }

  // ---- radix select: exact key of the K-th largest and the ties to take
  uint32_t prefix = 0, mask = 0, kk = (uint32_t)K;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkRowThreads) hist[i] = 0u;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kTopkRowThreads) {
      const uint32_t u = score_key(s[i]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l holds bins 8l .. 8l+7; find the bin where the count from the top reaches kk
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hist[tid * 8 + b];
        sum += c[b];
      }
      uint32_t above = sum;  // inclusive suffix over lanes >= tid
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t u = __shfl_down_sync(0xffffffffu, above, off);
        if (tid + off < 32) above += u;
      }
      uint32_t acc = above - sum;  // candidates in bins of higher lanes
      if (acc < kk && acc + sum >= kk) {
#pragma unroll
        for (int b = 7; b >= 0; --b) {
          if (acc + c[b] >= kk) {
            s_prefix = prefix | ((uint32_t)(tid * 8 + b) << shift);
            s_kk = kk - acc;
            break;
          }
          acc += c[b];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    kk = s_kk;
    mask |= 255u << shift;
  }
  const uint32_t thr = prefix;  // kk candidates with key == thr are selected, all with key > thr

  if (FAST) {
    // arrival order: the first kk ties to claim a slot win; output unsorted
    if (tid == 0) {
      s_slot_gt = 0;
      s_slot_tie = 0;
    }
    __syncthreads();
    const int n_gt = K - (int)kk;
    for (int64_t i = tid; i < n; i += kTopkRowThreads) {
      const uint32_t u = score_key(s[i]);
      if (u > thr) {
        o[atomicAdd(&s_slot_gt, 1)] = (int32_t)i;
      } else if (u == thr) {
        const int t = atomicAdd(&s_slot_tie, 1);
        if (t < (int)kk) o[n_gt + t] = (int32_t)i;
      }
    }
    return;
  }

  // ---- descending walk: tile of 4 positions per thread, thread 0 at the top
  uint32_t G = 0, E = 0;  // selected-above-threshold and ties met at higher positions
  const int64_t tile = 4 * kTopkRowThreads;
  for (int64_t hi = n; hi > 0; hi -= tile) {
    int32_t pos[4];
    uint32_t key[4];
    uint32_t gt = 0, tie = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t p = hi - 1 - (int64_t)tid * 4 - e;
      pos[e] = (int32_t)p;
      key[e] = p >= 0 ? score_key(s[p]) : 0u;
      if (p >= 0) {
        gt += key[e] > thr;
        tie += key[e] == thr;
      }
    }
    const uint32_t ex = block_exclusive_sum<kTopkRowThreads>(gt | (tie << 16), warp_sums, &s_total);
    uint32_t g = G + (ex & 0xffffu), t = E + (ex >> 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (pos[e] < 0) continue;
      if (key[e] > thr) {
        o[g + (t < kk ? t : kk)] = pos[e];
        ++g;
      } else if (key[e] == thr) {
        if (t < kk) o[g + t] = pos[e];
        ++t;
      }
    }
    const uint32_t tot = s_total;
    G += tot & 0xffffu;
    E += tot >> 16;
    if (G + (E < kk ? E : kk) >= (uint32_t)K) break;  // all K written
    __syncthreads();  // s_total is rewritten by the next tile
  }
}

// Few rows: a cluster of kTopkCluster CTAs per row.
template <bool FAST, bool CACHED>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int64_t ld,
                                                            const int32_t* __restrict__ n_valid, int K,
                                                            int32_t* __restrict__ out, int* status) {
  __shared__ uint32_t hist[2][256];  // this CTA's histogram, double-buffered across passes
  __shared__ uint32_t total[256];    // the cluster's histogram
  __shared__ uint32_t warp_sums[kTopkWarps];
  __shared__ uint32_t s_prefix, s_kk, s_total;
  __shared__ uint32_t s_counts[2];   // this chunk's (keys above threshold, ties)
  __shared__ int s_slot[2];          // BI_FAST: slot counters (used in cluster rank 0)
  extern __shared__ uint32_t keys[];  // CACHED: this chunk's keys
  cg::cluster_group cluster = cg::this_cluster();
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int rank = (int)cluster.block_rank();
  const int64_t row = blockIdx.x / kTopkCluster;
  const float* s = scores + row * ld;
  int32_t* o = out + row * (int64_t)K;
  int64_t n = n_valid[row];
  if (n < 0 || n > ld) {
    if (tid == 0 && rank == 0) report(status, DEV_BAD_INDEX);
    n = n < 0 ? 0 : ld;
  }
  if (n <= K) {  // every candidate is selected (the whole cluster returns here)
    if (rank == 0)
      for (int i = tid; i < K; i += kTopkThreads) o[i] = i < n ? (int32_t)(n - 1 - i) : -1;
    return;
  }
  const int64_t cs = (n + kTopkCluster - 1) / kTopkCluster;
  const int64_t lo = std::min<int64_t>(n, rank * cs), hi = std::min<int64_t>(n, lo + cs);
  const int m = (int)(hi - lo);
  auto key_at = [&](int i) -> uint32_t { return CACHED ? keys[i] : score_key(s[lo + i]); };
  if (CACHED) {
    for (int i = tid; i < m; i += kTopkThreads) keys[i] = score_key(s[lo + i]);
  }
  if (tid == 0) s_slot[0] = s_slot[1] = 0;

  // ---- radix select over the cluster
  uint32_t prefix = 0, mask = 0, kk = (uint32_t)K;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* h = hist[pass & 1];
    h[tid] = 0u;  // 256 threads, 256 bins
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < m; i += kTopkThreads) {
      const uint32_t u = key_at(i);
      if ((u & mask) == prefix) atomicAdd(&h[(u >> shift) & 255u], 1u);
    }
    cluster.sync();  // every chunk's histogram is complete
    uint32_t t = 0;
#pragma unroll
    for (int r = 0; r < kTopkCluster; ++r) t += cluster.map_shared_rank(h, r)[tid];
    total[tid] = t;
    __syncthreads();
    if (tid < 32) {
      // lane l holds bins 8l .. 8l+7; find the bin where the count from the top reaches kk
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = total[tid * 8 + b];
        sum += c[b];
      }
      uint32_t above = sum;  // inclusive suffix over lanes >= tid
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t u = __shfl_down_sync(0xffffffffu, above, off);
        if (tid + off < 32) above += u;
      }
      uint32_t acc = above - sum;  // candidates in bins of higher lanes
      if (acc < kk && acc + sum >= kk) {
#pragma unroll
        for (int b = 7; b >= 0; --b) {
          if (acc + c[b] >= kk) {
            s_prefix = prefix | ((uint32_t)(tid * 8 + b) << shift);
            s_kk = kk - acc;
            break;
          }
          acc += c[b];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    kk = s_kk;
    mask |= 255u << shift;
    // the other buffer is zeroed next pass: every CTA has read it, since all
    // passed this pass's cluster.sync after reading it in the previous pass
  }
  const uint32_t thr = prefix;  // kk candidates with key == thr are selected, all with key > thr

  if (FAST) {
    // arrival order across the cluster: slots claimed on rank 0's counters; output unsorted
    int* slot = cluster.map_shared_rank(s_slot, 0);
    const int n_gt = K - (int)kk;
    for (int i = tid; i < m; i += kTopkThreads) {
      const uint32_t u = key_at(i);
      if (u > thr) {
        o[atomicAdd(&slot[0], 1)] = (int32_t)(lo + i);
      } else if (u == thr) {
        const int q = atomicAdd(&slot[1], 1);
        if (q < (int)kk) o[n_gt + q] = (int32_t)(lo + i);
      }
    }
    cluster.sync();  // rank 0's counters stay alive until every CTA is done with them
    return;
  }

  // ---- counts of this chunk, then of the chunks above it
  uint32_t gt = 0, tie = 0;
  for (int i = tid; i < m; i += kTopkThreads) {
    const uint32_t u = key_at(i);
    gt += u > thr;
    tie += u == thr;
  }
  block_exclusive_sum<kTopkThreads>(gt | (tie << 16), warp_sums, &s_total);
  if (tid == 0) {
    s_counts[0] = s_total & 0xffffu;
    s_counts[1] = s_total >> 16;
  }
  cluster.sync();
  uint32_t G = 0, E = 0;  // above-threshold keys and ties at higher positions
  for (int r = rank + 1; r < kTopkCluster; ++r) {
    const uint32_t* c = cluster.map_shared_rank(s_counts, r);
    G += c[0];
    E += c[1];
  }
  cluster.sync();  // no CTA leaves while another still reads its counts

  // ---- descending walk of this chunk: 4 positions per thread per tile, thread 0 at the top
  const int tile = 4 * kTopkThreads;
  for (int top = m; top > 0; top -= tile) {
    if (G + (E < kk ? E : kk) >= (uint32_t)K) break;  // all K are out (uniform across the block)
    int idx[4];
    uint32_t key[4];
    gt = 0;
    tie = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      idx[e] = top - 1 - tid * 4 - e;
      key[e] = idx[e] >= 0 ? key_at(idx[e]) : 0u;
      if (idx[e] >= 0) {
        gt += key[e] > thr;
        tie += key[e] == thr;
      }
    }
    const uint32_t ex = block_exclusive_sum<kTopkThreads>(gt | (tie << 16), warp_sums, &s_total);
    uint32_t g = G + (ex & 0xffffu), t = E + (ex >> 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (idx[e] < 0) continue;
      if (key[e] > thr) {
        o[g + (t < kk ? t : kk)] = (int32_t)(lo + idx[e]);
        ++g;
      } else if (key[e] == thr) {
        if (t < kk) o[g + t] = (int32_t)(lo + idx[e]);
        ++t;
      }
    }
    const uint32_t tot = s_total;
    G += tot & 0xffffu;
    E += tot >> 16;
    __syncthreads();  // s_total is rewritten by the next tile
  }
}

template <bool FAST, bool CACHED>
static bi_status launch_topk(const float* scores, int64_t T, int64_t ld, const int32_t* n_valid, int K,
                             int32_t* idx_out, cudaStream_t st) {
  const int64_t chunk = (ld + kTopkCluster - 1) / kTopkCluster;
  const int dyn = CACHED ? (int)(std::max<int64_t>(chunk, 1) * 4) : 0;
  if (CACHED) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
      err = cudaFuncSetAttribute(topk_kernel<FAST, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kTopkChunkKeys * 4);
    });
    if (err != cudaSuccess) return fail(BI_ERR_CUDA, std::string("bi_topk smem attribute: ") + cudaGetErrorString(err));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(T * kTopkCluster));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTopkCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return launched(cudaLaunchKernelEx(&cfg, topk_kernel<FAST, CACHED>, scores, ld, n_valid, K, idx_out,
                                     device_status_ptr()),
                  "bi_topk");
}

}  // namespace bi

extern "C" bi_status bi_topk(const float* scores, int64_t T, int64_t ld, const int32_t* n_valid, int K,
                             int32_t* idx_out, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(T >= 0 && ld >= 0, "bad shape");
  BI_REQUIRE(K >= 1 && K <= kTopkMaxK, "K must be in [1, 4096]");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  if (T == 0) return BI_OK;
  BI_REQUIRE(scores && n_valid && idx_out, "null pointer");
  BI_REQUIRE(T <= 0x7fffffff / kTopkCluster && ld <= 0x7fffffff, "too many rows or positions");
  cudaStream_t st = as_stream(stream);
  // Both kernels return the one selection the key order defines; rows that
  // fill the GPU on their own take one CTA each, fewer rows a cluster each.
  if (T >= 2 * (int64_t)num_sms()) {
    auto kern = mode == BI_FAST ? topk_row_kernel<true> : topk_row_kernel<false>;
    return launched(launch_pdl(kern, dim3((unsigned)T), dim3(kTopkRowThreads), 0, st, scores, ld, n_valid, K,
                               idx_out, device_status_ptr()),
                    "bi_topk");
  }
  const bool cached = (ld + kTopkCluster - 1) / kTopkCluster <= kTopkChunkKeys;
  if (mode == BI_FAST)
    return cached ? launch_topk<true, true>(scores, T, ld, n_valid, K, idx_out, st)
                  : launch_topk<true, false>(scores, T, ld, n_valid, K, idx_out, st);
  return cached ? launch_topk<false, true>(scores, T, ld, n_valid, K, idx_out, st)
                : launch_topk<false, false>(scores, T, ld, n_valid, K, idx_out, st);
}
