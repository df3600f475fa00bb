// Deterministic Top-K with a unique (score, in-request position) key.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.3 ("Top-K in sparse
// attention: fix ties and order"): a default Top-K breaks ties by thread
// scheduling; the consistent one makes the key unique by appending the
// candidate's in-request position to the score bits, so a tie goes to the
// larger position, and returns the selected positions sorted by descending
// position with invalid entries last.
//
// One CTA per row.  The score of every candidate maps to an order-preserving
// 32-bit key (-0 first made +0, so equal scores give equal keys).  A 4-pass
// 8-bit radix select finds the exact key of the K-th largest score and how
// many of the candidates holding exactly that key belong to the selection
// (kk).  One more pass walks the positions from the top in tiles of
// 4 x blockDim.x, counting per thread and prefix-summing over the block, and
// writes each selected position to its final slot: a key above the threshold
// is always selected, a key equal to it is selected while fewer than kk of
// those have been met at higher positions.  Writing in descending position
// order needs no sort; the walk stops once K positions are out.
#include <string>

#include "common.cuh"

namespace bi {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkMaxK = 4096;

__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one packed value per thread (thread 0 first);
// returns the exclusive prefix and writes the block total to *total.
__device__ __forceinline__ uint32_t block_exclusive_sum(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
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
    uint32_t w = lane < kTopkWarps ? warp_sums[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    if (lane < kTopkWarps) warp_sums[lane] = wi - w;  // exclusive over warps
    if (lane == kTopkWarps - 1) *total = wi;
  }
  __syncthreads();
  const uint32_t r = warp_sums[warp] + inc - v;
  __syncthreads();  // warp_sums is reused by the next call
  return r;
}

template <bool FAST>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int64_t ld,
                                                            const int32_t* __restrict__ n_valid, int K,
                                                            int32_t* __restrict__ out, int* status) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[kTopkWarps];
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
    for (int i = tid; i < K; i += kTopkThreads) o[i] = i < n ? (int32_t)(n - 1 - i) : -1;
    return;
  }

  // ---- radix select: exact key of the K-th largest and the ties to take
  uint32_t prefix = 0, mask = 0, kk = (uint32_t)K;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kTopkThreads) {
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
    for (int64_t i = tid; i < n; i += kTopkThreads) {
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
  const int64_t tile = 4 * kTopkThreads;
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
    const uint32_t ex = block_exclusive_sum(gt | (tie << 16), warp_sums, &s_total);
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

}  // namespace bi

extern "C" bi_status bi_topk(const float* scores, int64_t T, int64_t ld, const int32_t* n_valid, int K,
                             int32_t* idx_out, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(T >= 0 && ld >= 0, "bad shape");
  BI_REQUIRE(K >= 1 && K <= kTopkMaxK, "K must be in [1, 4096]");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  if (T == 0) return BI_OK;
  BI_REQUIRE(scores && n_valid && idx_out, "null pointer");
  BI_REQUIRE(T <= 0x7fffffff && ld <= 0x7fffffff, "too many rows or positions");
  auto kern = mode == BI_FAST ? topk_kernel<true> : topk_kernel<false>;
  return launched(launch_pdl(kern, dim3((unsigned)T), dim3(kTopkThreads), 0, as_stream(stream), scores, ld, n_valid,
                             K, idx_out, device_status_ptr()),
                  "bi_topk");
}
