// Block-FP8 (e4m3) quantisation and the W8A8 tcgen05 GEMM.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 ("Dense GEMM: keep
// FP8, one accumulation order for every M"): the deployment GEMM is block-FP8
// W8A8 and every training forward quantises the bf16 master weights to block
// FP8 by the deployment rule, then calls the same GEMM.  The pages fix neither
// the block sizes nor the scale format; this file takes 128 x 128 weight
// blocks, 1 x 128 activation blocks and power-of-two scales
// s = 2^ceil(log2(amax / 448)), which make dequantisation exact.
//
// GEMM: C[m, n] = sum over K blocks kb of sa[m, kb] sw[n/128, kb] P_kb[m, n],
// P_kb the e4m3 product over the 128 K of block kb.  One persistent CTA per
// SM walks 128 x 256 output tiles: warp 0 streams A (128 x 128 bytes) and W
// (256 x 128 bytes) tiles with TMA, warp 1 issues four tcgen05 kind::f8f6f4
// MMAs (N = 256, K = 32 each) per K block into one of two 256-column TMEM
// partial buffers, and warps 2..9 (two per TMEM lane quarter, one per
// 128-column half, i.e. per weight block) add each finished partial, times
// the exact power-of-two scale product, to an fp32 accumulator held in
// registers, in ascending kb.  The tile shape and the K order are the same for
// every M, so every row's result is batch invariant.  Calls of at most 16
// rows run the same MMA with the operands' roles exchanged (weight tiles as its
// M side; see gemm_fp8_dec_kernel), which leaves every element's bits as they are.
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "common.cuh"
#include "fp8.cuh"

namespace bi {

constexpr int kF8Block = 128;   // K block = weight block rows
constexpr int kF8BN = 256;      // output tile width: two weight blocks
constexpr int kF8Stages = 4;
constexpr int kF8TileBytes = 128 * kF8Block;       // A: 128 rows x 128 fp8
constexpr int kF8BTileBytes = kF8BN * kF8Block;    // W: 256 rows x 128 fp8
// acc (two fp32 lanes) += (x0, x1) * (s, s) with one rounding each: a packed fp32 FMA.
__device__ __forceinline__ void fma2_acc(unsigned long long& acc, uint32_t x0, uint32_t x1, unsigned long long ss) {
  unsigned long long x;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(x0), "r"(x1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(x), "l"(ss));
}
__device__ __forceinline__ float lo_f32(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f32(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }

constexpr int kF8Threads = 320;                    // TMA, MMA, 8 promotion warps
constexpr int kF8SmemBytes = 1024 + kF8Stages * (kF8TileBytes + kF8BTileBytes) + 256;

// Activations (1 x 128 blocks): one warp per block, 4 consecutive elements per
// lane, amax by warp shuffles; 8 blocks per CTA.
__global__ void __launch_bounds__(256) quantize_fp8_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t R,
                                                                int64_t C, uint8_t* __restrict__ q,
                                                                float* __restrict__ scales) {
  pdl_trigger();
  pdl_wait();
  const int64_t nb = C / kF8Block;
  const int64_t blk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (blk >= R * nb) return;
  const int lane = threadIdx.x & 31;
  const int64_t r = blk / nb, c0 = (blk % nb) * kF8Block + lane * 4;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + r * C + c0);
  float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u), __uint_as_float(raw.y << 16),
                __uint_as_float(raw.y & 0xffff0000u)};
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int e = fp8_scale_exp(m);
  if (lane == 0) scales[blk] = ldexpf(1.f, e);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    packed |= fp8_code(v[i], e) << (8 * i);
  *reinterpret_cast<uint32_t*>(q + r * C + c0) = packed;
}

// Weights (128 x 128 blocks): one CTA of 256 threads per block; thread t takes
// 4 consecutive columns (t % 32) of rows t / 32, t / 32 + 8, ...
__global__ void __launch_bounds__(256) quantize_fp8_blocks_kernel(const __nv_bfloat16* __restrict__ x, int64_t R,
                                                                  int64_t C, uint8_t* __restrict__ q,
                                                                  float* __restrict__ scales) {
  __shared__ float wmax[8];
  pdl_trigger();
  pdl_wait();
  const int64_t r0 = (int64_t)blockIdx.x * kF8Block;
  const int64_t c0 = (int64_t)blockIdx.y * kF8Block + (threadIdx.x & 31) * 4;
  const int rsub = threadIdx.x >> 5;
  float m = 0.f;
  for (int i = rsub; i < kF8Block && r0 + i < R; i += 8) {
    const uint2 raw = *reinterpret_cast<const uint2*>(x + (r0 + i) * C + c0);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(raw.x << 16)), fabsf(__uint_as_float(raw.x & 0xffff0000u))),
                       fmaxf(fabsf(__uint_as_float(raw.y << 16)), fabsf(__uint_as_float(raw.y & 0xffff0000u)))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[rsub] = m;
  __syncthreads();
  float amax = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
  const int e = fp8_scale_exp(amax);
  if (threadIdx.x == 0) scales[(int64_t)blockIdx.x * (C / kF8Block) + blockIdx.y] = ldexpf(1.f, e);
  for (int i = rsub; i < kF8Block && r0 + i < R; i += 8) {
    const uint2 raw = *reinterpret_cast<const uint2*>(x + (r0 + i) * C + c0);
    const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                        __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      packed |= fp8_code(v[k], e) << (8 * k);
    *reinterpret_cast<uint32_t*>(q + (r0 + i) * C + c0) = packed;
  }
}

struct F8Args {
  const float* sa;  // [M, nkb]
  const float* sw;  // [N / 128, nkb]
  void* C;
  int* status;
  int M, N, nkb, m_tiles, n_tiles, a_box_rows, c_fp32;
};

__global__ void __launch_bounds__(kF8Threads, 1) gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA,
                                                          const __grid_constant__ CUtensorMap tmB, const F8Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kF8Stages * kF8TileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kF8Stages * kF8BTileBytes);
  uint64_t* empty = full + kF8Stages;
  uint64_t* pfull = empty + kF8Stages;   // [2] MMA -> epilogue: a K block's partial is in TMEM
  uint64_t* pempty = pfull + 2;          // [2] epilogue -> MMA (8 warp arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr uint32_t kTmemCols = 2 * kF8BN;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = args.m_tiles * args.n_tiles;
  const int nk = args.nkb;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], 8);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // tiles walk M fastest, so consecutive CTAs share a weight tile in L2
  auto tile_mn = [&](int t, int& mt, int& nt) {
    mt = t % args.m_tiles;
    nt = t / args.m_tiles;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      pdl_wait();
      const uint32_t stage_bytes = (uint32_t)args.a_box_rows * kF8Block + kF8BTileBytes;
      int kb_total = 0;
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        int mt, nt;
        tile_mn(t, mt, nt);
        for (int kb = 0; kb < nk; ++kb, ++kb_total) {
          const int s = kb_total % kF8Stages;
          const uint32_t ph = (kb_total / kF8Stages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1) || *abort_flag) {
            report(args.status, DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          tma_load_2d(sA + s * kF8TileBytes, &tmA, &full[s], kb * kF8Block, mt * 128);
          tma_load_2d(sB + s * kF8BTileBytes, &tmB, &full[s], kb * kF8Block, nt * kF8BN);
        }
      }
      for (int i = 0; i < kF8Stages && i < kb_total; ++i) {  // let the last copies land
        const int kb = kb_total - 1 - i;
        mbar_wait(&full[kb % kF8Stages], (kb / kF8Stages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: one TMEM partial per K block, two buffers
      constexpr uint32_t idesc = idesc_e4m3_f32(128, kF8BN);
      int kb_total = 0, pb = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok && !*abort_flag; t += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb, ++kb_total, ++pb) {
          const int j = pb & 1;
          const int s = kb_total % kF8Stages;
          if (!mbar_wait(&pempty[j], ((pb >> 1) & 1) ^ 1) ||
              !mbar_wait(&full[s], (kb_total / kF8Stages) & 1) || *abort_flag) {
            report(args.status, DEV_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + s * kF8TileBytes);
          const uint32_t b_addr = smem_u32(sB + s * kF8BTileBytes);
          const uint32_t d = tmem_base + j * kF8BN;
#pragma unroll
          for (int k = 0; k < kF8Block / 32; ++k)
            tc_mma_f8(d, sw128_kmajor_desc(a_addr + k * 32), sw128_kmajor_desc(b_addr + k * 32), idesc,
                      k != 0 ? 1u : 0u);
          tc_commit(&empty[s]);
          tc_commit(&pfull[j]);
        }
      }
    }
  } else {
    // ---------------- promotion and store: warps 2..9; lane quarter q = warp % 4,
    // column half (= weight block within the tile) hf = (warp - 2) / 4
    const int q = warp & 3, hf = (warp - 2) >> 2;
    pdl_wait();
    int pb = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      int mt, nt;
      tile_mn(t, mt, nt);
      const int row = mt * 128 + q * 32 + lane;
      const int wblk = nt * 2 + hf;                       // weight block row of this half
      const bool valid = row < args.M && wblk * kF8Block < args.N;
      unsigned long long acc2[kF8Block / 2];  // fp32 pairs (columns 2i, 2i + 1)
#pragma unroll
      for (int c = 0; c < kF8Block / 2; ++c) acc2[c] = 0ull;
      for (int kb = 0; kb < nk; ++kb, ++pb) {
        const int j = pb & 1;
        const float sc = valid ? args.sa[(int64_t)row * nk + kb] * args.sw[(int64_t)wblk * nk + kb] : 0.f;
        // decided for the whole warp: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&pfull[j], (pb >> 1) & 1))) {
          report(args.status, DEV_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + j * kF8BN + hf * kF8Block + ((uint32_t)(q * 32) << 16);
        // acc += partial * (scale_a * scale_w), one rounding per element (paired fp32 FMA);
        // 16 columns per TMEM round trip
        const unsigned long long sc2 = ((unsigned long long)__float_as_uint(sc) << 32) | __float_as_uint(sc);
#pragma unroll
        for (int c = 0; c < kF8Block / 16; ++c) {
          uint32_t p[16];
          tmem_ld_32x32b_x16(taddr + c * 16, p);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; i += 2) fma2_acc(acc2[(c * 16 + i) / 2], p[i], p[i + 1], sc2);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[j]);
      }
      if (!ok || !valid || *abort_flag) continue;
      const int64_t base = (int64_t)row * args.N + (int64_t)wblk * kF8Block;
      if (args.c_fp32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(args.C) + base);
#pragma unroll
        for (int v = 0; v < kF8Block / 4; ++v)
          dst[v] = make_float4(lo_f32(acc2[2 * v]), hi_f32(acc2[2 * v]), lo_f32(acc2[2 * v + 1]),
                               hi_f32(acc2[2 * v + 1]));
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.C) + base);
#pragma unroll
        for (int v = 0; v < kF8Block / 8; ++v)
          dst[v] = make_uint4(pack_bf16x2(lo_f32(acc2[4 * v]), hi_f32(acc2[4 * v])),
                              pack_bf16x2(lo_f32(acc2[4 * v + 1]), hi_f32(acc2[4 * v + 1])),
                              pack_bf16x2(lo_f32(acc2[4 * v + 2]), hi_f32(acc2[4 * v + 2])),
                              pack_bf16x2(lo_f32(acc2[4 * v + 3]), hi_f32(acc2[4 * v + 3])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ decode-size calls
// Calls of at most 16 rows (decode steps) on the same tensor-core MMA with the
// operands' roles exchanged: a tile of BM (64 or 128) weight rows is the MMA's
// M side and the call's rows, zero-filled by the TMA copy up to R = 16, are its
// N side, so one CTA per BM output columns streams its weight rows once (N / BM
// CTAs where the 128-row tile above gives N / 256).  (R = 32 and 64 were
// measured at 64-row calls of the long-context decoder: slower there than the
// 128 x 256 tiles, whose 44 and 8 CTAs stream the weights at least as fast.)  An element's partial per K
// block is the same sum of the same products in the same K order as in the
// large kernel (which operand is which does not enter a product), and the
// promotion is the same fp32 fma in ascending kb, so the rows are the same bits
// (the row-invariance test compares them across M).  Weights are copied before
// the dependency wait and the call's codes after it; a ring of up to
// f8dec_max_stages K blocks holds the whole K of the usual decode shapes, so
// every copy is in flight at once.  The scale products sa[m, kb] sw[n/128, kb]
// of the CTA's weight block are formed once, before the K loop, into shared
// memory (the same fp32 product the large kernel forms per block).
constexpr int kF8DecMaxRows = 16;   // the MMA's N: rows of the call, zero past M
constexpr int kF8DecBufs = 4;       // TMEM partial buffers (R columns each)
constexpr int kF8DecThreads = 192;  // TMA, MMA, four promotion warps (one per lane quarter)
constexpr size_t kF8DecMaxSmem = 220 * 1024;
__host__ __device__ constexpr int f8dec_stage_bytes(int bm, int r) { return (bm + r) * kF8Block; }
__host__ __device__ constexpr int f8dec_max_stages(int bm, int r) {
  return 196608 / f8dec_stage_bytes(bm, r) < 16 ? 196608 / f8dec_stage_bytes(bm, r) : 16;
}
__host__ constexpr size_t f8dec_smem(int bm, int r, int stages, int nkb) {
  return 1024 + (size_t)stages * f8dec_stage_bytes(bm, r) + (size_t)r * nkb * 4 + 512;
}

struct F8DecArgs {
  const float* sa;  // [M, nkb]
  const float* sw;  // [N / 128, nkb]
  void* C;
  int* status;
  int M, N, nkb, stages, c_fp32;
};

template <int BM, int R>
__global__ void __launch_bounds__(kF8DecThreads, 1) gemm_fp8_dec_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                 const __grid_constant__ CUtensorMap tmX,
                                                                 const F8DecArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = args.stages, nk = args.nkb;
  uint8_t* sW = smem;                              // [S][BM rows x 128 codes], 128-byte swizzle
  uint8_t* sX = smem + S * BM * kF8Block;          // [S][16 rows x 128 codes]
  float* sc_s = reinterpret_cast<float*>(sX + S * R * kF8Block);  // [nk][R] scale products
  uint64_t* full = reinterpret_cast<uint64_t*>(sc_s + nk * R);
  uint64_t* empty = full + S;
  uint64_t* pfull = empty + S;                     // [kF8DecBufs] MMA -> promotion
  uint64_t* pempty = pfull + kF8DecBufs;           // [kF8DecBufs] promotion -> MMA (4 warp arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pempty + kF8DecBufs);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr uint32_t kTmemCols = kF8DecBufs * R;
  constexpr uint32_t kStageW = BM * kF8Block, kStageX = R * kF8Block;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BM;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kF8DecBufs; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: the first ring's weights before the
      // dependency wait, its codes after it; later blocks reuse freed stages
      const int first = min(nk, S);
      for (int kb = 0; kb < first; ++kb) {
        mbar_arrive_expect_tx(&full[kb], kStageW + kStageX);
        tma_load_2d(sW + kb * kStageW, &tmW, &full[kb], kb * kF8Block, n0);
      }
      pdl_wait();
      for (int kb = 0; kb < first; ++kb) tma_load_2d(sX + kb * kStageX, &tmX, &full[kb], kb * kF8Block, 0);
      for (int kb = first; kb < nk; ++kb) {
        const int s = kb % S;
        if (!mbar_wait(&empty[s], ((kb / S) & 1) ^ 1) || *abort_flag) {
          report(args.status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kStageW + kStageX);
        tma_load_2d(sW + s * kStageW, &tmW, &full[s], kb * kF8Block, n0);
        tma_load_2d(sX + s * kStageX, &tmX, &full[s], kb * kF8Block, 0);
      }
      for (int i = 0; i < S && i < nk; ++i) {  // let the last copies land
        const int kb = nk - 1 - i;
        mbar_wait(&full[kb % S], (kb / S) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: one TMEM partial (BM x 16) per K block
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, R);
      for (int kb = 0; kb < nk; ++kb) {
        const int j = kb % kF8DecBufs, s = kb % S;
        if (!mbar_wait(&pempty[j], ((kb / kF8DecBufs) & 1) ^ 1) || !mbar_wait(&full[s], (kb / S) & 1) ||
            *abort_flag) {
          report(args.status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t w_addr = smem_u32(sW + s * kStageW), x_addr = smem_u32(sX + s * kStageX);
#pragma unroll
        for (int k = 0; k < kF8Block / 32; ++k)
          tc_mma_f8(tmem_base + j * R, sw128_kmajor_desc(w_addr + k * 32), sw128_kmajor_desc(x_addr + k * 32),
                    idesc, k != 0 ? 1u : 0u);
        tc_commit(&empty[s]);
        tc_commit(&pfull[j]);
      }
    }
  } else {
    // ---------------- promotion and store: warps 2..5, lane quarter q = warp % 4;
    // thread (q, lane) owns output column n0 + c (c = its tile row) for the R rows
    const int q = warp & 3;
    const int c = BM == 128 ? 32 * q + lane : 16 * q + lane;
    const bool col_ok = (BM == 128 || lane < 16) && n0 + c < args.N;
    const int wblk = n0 / kF8Block;  // BM divides 128: the tile lies in one weight block
    const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
    float acc[R];
#pragma unroll
    for (int m = 0; m < R; ++m) acc[m] = 0.f;
    pdl_wait();  // the row scales come from the preceding kernel
    // the scale products of every (kb, row): sa * sw, one rounding (0 past M)
    for (int i = threadIdx.x - 64; i < nk * R; i += 128) {
      const int kb = i / R, m = i % R;
      sc_s[i] = m < args.M ? __fmul_rn(args.sa[(int64_t)m * nk + kb], args.sw[(int64_t)wblk * nk + kb]) : 0.f;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");  // the four promotion warps
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int j = kb % kF8DecBufs;
      // decided for the whole warp: the TMEM load below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&pfull[j], (kb / kF8DecBufs) & 1) && !*abort_flag)) {
        report(args.status, DEV_TIMEOUT);
        *abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      // acc += partial * (scale_a * scale_w), one rounding per element; 16 rows per
      // TMEM load
#pragma unroll
      for (int c16 = 0; c16 < R; c16 += 16) {
        uint32_t p[16];
        tmem_ld_32x32b_x16(tq + j * R + c16, p);
        tmem_ld_wait();
        const float4* sc4 = reinterpret_cast<const float4*>(sc_s + kb * R + c16);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 sc = sc4[i / 4];
          acc[c16 + i] = __fmaf_rn(__uint_as_float(p[i]), sc.x, acc[c16 + i]);
          acc[c16 + i + 1] = __fmaf_rn(__uint_as_float(p[i + 1]), sc.y, acc[c16 + i + 1]);
          acc[c16 + i + 2] = __fmaf_rn(__uint_as_float(p[i + 2]), sc.z, acc[c16 + i + 2]);
          acc[c16 + i + 3] = __fmaf_rn(__uint_as_float(p[i + 3]), sc.w, acc[c16 + i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pempty[j]);
    }
    if (ok && col_ok && !*abort_flag) {
      const int col = n0 + c;
#pragma unroll
      for (int m = 0; m < R; ++m) {
        if (m >= args.M) break;
        if (args.c_fp32)
          static_cast<float*>(args.C)[(int64_t)m * args.N + col] = acc[m];
        else
          static_cast<__nv_bfloat16*>(args.C)[(int64_t)m * args.N + col] = __float2bfloat16_rn(acc[m]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace bi

extern "C" {

bi_status bi_quantize_fp8(const void* x, int64_t R, int64_t C, int block_rows, void* q, float* scales,
                          void* stream) {
  using namespace bi;
  BI_REQUIRE(R >= 0 && C >= 0, "bad shape");
  BI_REQUIRE(block_rows == 1 || block_rows == 128, "block_rows must be 1 (activations) or 128 (weights)");
  BI_REQUIRE_SHAPE(C % kF8Block == 0, "columns must be a multiple of 128");
  if (R == 0 || C == 0) return BI_OK;
  BI_REQUIRE(x && q && scales, "null pointer");
  BI_REQUIRE(aligned16(x) && ((uintptr_t)q & 3) == 0, "x must be 16-byte and q 4-byte aligned");
  cudaStream_t st = as_stream(stream);
  if (block_rows == 1) {
    const int64_t blocks = R * (C / kF8Block);
    BI_REQUIRE(cdiv(blocks, 8) <= 0x7fffffff, "too many blocks");
    return launched(launch_pdl(quantize_fp8_rows_kernel, dim3((unsigned)cdiv(blocks, 8)), dim3(256), 0, st,
                               static_cast<const __nv_bfloat16*>(x), R, C, static_cast<uint8_t*>(q), scales),
                    "bi_quantize_fp8");
  }
  const int64_t rb = cdiv(R, block_rows);
  BI_REQUIRE(rb <= 0x7fffffff && C / kF8Block <= 65535, "too many blocks");
  return launched(launch_pdl(quantize_fp8_blocks_kernel, dim3((unsigned)rb, (unsigned)(C / kF8Block)), dim3(256), 0,
                             st, static_cast<const __nv_bfloat16*>(x), R, C, static_cast<uint8_t*>(q), scales),
                  "bi_quantize_fp8");
}

bi_status bi_gemm_fp8(const void* Aq, const float* sa, int64_t M, int64_t K, const void* Wq, const float* sw,
                      int64_t N, void* C, int c_dtype, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(M >= 0 && N >= 0 && K >= 0, "bad shape");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  BI_REQUIRE(c_dtype == BI_DTYPE_BF16 || c_dtype == BI_DTYPE_FP32, "bad output dtype");
  BI_REQUIRE_SHAPE(K % kF8Block == 0 && N % kF8Block == 0, "N and K must be multiples of 128");
  if (M == 0 || N == 0) return BI_OK;
  BI_REQUIRE(K > 0 && Aq && sa && Wq && sw && C, "null pointer");
  BI_REQUIRE(aligned16(Aq) && aligned16(Wq) && aligned16(C), "pointers must be 16-byte aligned");
  BI_REQUIRE(M <= 0x7fffffff && N <= 0x7fffffff, "shape too large");
  const int nkb = (int)(K / kF8Block);
  // decode sizes: weight tiles as the MMA's M side (the same bits); 128-row tiles
  // once 64-row ones would fill the GPU twice
  const int bm = N / 64 >= 2 * (int64_t)num_sms() ? 128 : 64;
  constexpr int rr = kF8DecMaxRows;
  const int dec_stages = std::min(nkb, f8dec_max_stages(bm, rr));
  if (M <= kF8DecMaxRows && f8dec_smem(bm, rr, dec_stages, nkb) <= kF8DecMaxSmem) {
    static std::once_flag once_dec;
    static cudaError_t attr_dec = cudaSuccess;
    std::call_once(once_dec, [] {
      const int smax = (int)kF8DecMaxSmem;
      cudaError_t e = cudaSuccess;
      auto set = [&](auto fn) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smax);
      };
      set(gemm_fp8_dec_kernel<64, rr>);
      set(gemm_fp8_dec_kernel<128, rr>);
      attr_dec = e;
    });
    if (attr_dec != cudaSuccess)
      return fail(BI_ERR_CUDA, std::string("bi_gemm_fp8 decode smem attribute: ") + cudaGetErrorString(attr_dec));
    CUtensorMap tw, tx;
    if (!encode_tmap_2d_u8(&tw, Wq, K, N, K, kF8Block, bm) || !encode_tmap_2d_u8(&tx, Aq, K, M, K, kF8Block, rr))
      return fail(BI_ERR_CUDA, "bi_gemm_fp8: TMA descriptor failed");
    F8DecArgs da{sa, sw, C, device_status_ptr(), (int)M, (int)N, nkb, dec_stages, c_dtype == BI_DTYPE_FP32};
    const dim3 grid((unsigned)(N / bm)), block(kF8DecThreads);
    const size_t smem = f8dec_smem(bm, rr, dec_stages, nkb);
    cudaStream_t st = as_stream(stream);
    const cudaError_t le = bm == 64 ? launch_pdl(gemm_fp8_dec_kernel<64, rr>, grid, block, smem, st, tw, tx, da)
                                    : launch_pdl(gemm_fp8_dec_kernel<128, rr>, grid, block, smem, st, tw, tx, da);
    return launched(le, "bi_gemm_fp8");
  }
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8SmemBytes);
  });
  if (attr_err != cudaSuccess)
    return fail(BI_ERR_CUDA, std::string("bi_gemm_fp8 smem attribute: ") + cudaGetErrorString(attr_err));
  // a call with M < 128 copies only its rows of A (rounded up to 8); rows >= M are never stored
  const int a_rows = M < 128 ? (int)std::max<int64_t>(8, cdiv(M, 8) * 8) : 128;
  CUtensorMap ta, tb;
  if (!encode_tmap_2d_u8(&ta, Aq, K, M, K, kF8Block, a_rows) ||
      !encode_tmap_2d_u8(&tb, Wq, K, N, K, kF8Block, kF8BN))
    return fail(BI_ERR_CUDA, "bi_gemm_fp8: TMA descriptor failed");
  F8Args a;
  a.sa = sa;
  a.sw = sw;
  a.C = C;
  a.status = device_status_ptr();
  a.M = (int)M;
  a.N = (int)N;
  a.nkb = (int)(K / kF8Block);
  a.m_tiles = (int)cdiv(M, 128);
  a.n_tiles = (int)cdiv(N, kF8BN);
  a.a_box_rows = a_rows;
  a.c_fp32 = c_dtype == BI_DTYPE_FP32;
  const int64_t tiles = (int64_t)a.m_tiles * a.n_tiles;
  BI_REQUIRE_SHAPE(tiles < (1ll << 31), "too many tiles");
  return launched(launch_pdl(gemm_fp8_kernel, dim3((unsigned)std::min<int64_t>(tiles, num_sms())), dim3(kF8Threads),
                             kF8SmemBytes, as_stream(stream), ta, tb, a),
                  "bi_gemm_fp8");
}

}  // extern "C"
