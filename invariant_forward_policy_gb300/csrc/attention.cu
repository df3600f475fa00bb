// RoPE + paged KV write, fixed-split paged attention and the ascending-order split merge.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.2 ("FP8 KV cache: keep
// FP8 storage, unify the read path"): decode gives up its own batch-partitioned
// kernel and goes through prefill's algorithm, and training writes and reads a
// private cache the same way.  The zero-mismatch-rl README lists "fixed-split
// attention" for the hybrid model.  Here there is one attention kernel for
// prefill chunks and decode steps alike:
//   * a CTA owns (piece, 64-row query tile, kv head, split); rows are
//     (token, q head of the group) pairs;
//   * splits cover ABSOLUTE positions [s*S, (s+1)*S), S = kv_split, and inside a
//     split 64-key tiles (one cache block each) are taken in ascending order;
//   * scores and P*V run on bf16 mma.sync tensor-core tiles (row-independent),
//     the online softmax is fp32 with masking by select, so a key tile that is
//     fully masked for a row leaves that row's (m, l, acc) bit-for-bit unchanged;
//   * keys beyond the CTA's last query position are zero-filled, so stale cache
//     contents never reach the arithmetic;
//   * partials (m, l, acc) are merged per row in ascending split order.
// A decode row therefore reproduces its prefill row exactly.
#include <algorithm>
#include <mutex>
#include <string>
#include <type_traits>

#include "attn_merge.cuh"
#include "common.cuh"
#include "fp8.cuh"

namespace bi {

// ------------------------------------------------------------------ RoPE table
__global__ void rope_table_kernel(float* table, int64_t max_pos, int hd, double theta) {
  pdl_trigger();
  pdl_wait();
  const int half = hd / 2;
  const int64_t total = max_pos * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = idx / half;
    const int i = (int)(idx % half);
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)hd);
    const double ang = (double)p * inv_freq;
    table[p * hd + i] = (float)cos(ang);
    table[p * hd + half + i] = (float)sin(ang);
  }
}

// ------------------------------------------------------ RoPE + KV cache write
struct PieceMeta {
  const int32_t* seq;   // [P] sequence of each piece
  const int32_t* row0;  // [P+1] first row of each piece (row0[P] = T)
  const int32_t* pos0;  // [P] absolute position of each piece's first row
};

__global__ void rope_kv_write_kernel(const __nv_bfloat16* __restrict__ qkv, PieceMeta pm, int Hq, int Hkv, int hd,
                                     const float* __restrict__ table, int64_t max_pos,
                                     const int32_t* __restrict__ block_table, int64_t max_blk, int64_t n_blocks,
                                     __nv_bfloat16* __restrict__ q_out, __nv_bfloat16* __restrict__ k_cache,
                                     __nv_bfloat16* __restrict__ v_cache, int* status) {
  pdl_trigger();
  pdl_wait();
  const int p = blockIdx.y;
  const int i = blockIdx.x;
  const int row0 = pm.row0[p];
  if (i >= pm.row0[p + 1] - row0) return;
  const int64_t row = row0 + i;
  const int64_t pos = (int64_t)pm.pos0[p] + i;
  const int seq = pm.seq[p];
  const int half = hd / 2;
  const int nqkv = (Hq + 2 * Hkv) * hd;
  const __nv_bfloat16* src = qkv + row * nqkv;
  if (pos < 0 || pos >= max_pos) {
    report(status, DEV_BAD_INDEX);
    return;
  }
  const bool tab_ok = pos / 64 < max_blk;
  const int32_t blk = tab_ok ? block_table[(int64_t)seq * max_blk + pos / 64] : -1;
  const bool blk_ok = blk >= 0 && blk < n_blocks;
  if (!blk_ok && threadIdx.x == 0) report(status, DEV_BAD_INDEX);
  const float* cs = table + pos * hd;
  const int slot = (int)(pos % 64);
  // q and k heads: rotate pairs (j, j + hd/2)
  for (int idx = threadIdx.x; idx < (Hq + Hkv) * half; idx += blockDim.x) {
    const int h = idx / half;
    const int j = idx % half;
    const float x1 = bf2f(src[h * hd + j]);
    const float x2 = bf2f(src[h * hd + j + half]);
    const float c = cs[j], s = cs[half + j];
    const __nv_bfloat16 o1 = f2bf(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s)));
    const __nv_bfloat16 o2 = f2bf(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s)));
    if (h < Hq) {
      __nv_bfloat16* dst = q_out + (row * Hq + h) * hd;
      dst[j] = o1;
      dst[j + half] = o2;
    } else if (blk_ok) {
      const int kh = h - Hq;
      __nv_bfloat16* dst = k_cache + (((int64_t)blk * Hkv + kh) * 64 + slot) * hd;
      dst[j] = o1;
      dst[j + half] = o2;
    }
  }
  if (blk_ok) {
    for (int idx = threadIdx.x; idx < Hkv * hd; idx += blockDim.x) {
      const int kh = idx / hd, j = idx % hd;
      v_cache[(((int64_t)blk * Hkv + kh) * 64 + slot) * hd + j] = src[(Hq + Hkv) * hd + idx];
    }
  }
}

// ------------------------------------------------------------------ attention
struct AttnArgs {
  const __nv_bfloat16* q;  // [T, Hq, hd]
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;  // [n_blocks, Hkv, 64, hd]
  // FP8 cache (the KV8 kernels): e4m3 codes [n_blocks, Hkv, 64, hd] and one
  // fp32 scale per (block, kv head, slot)
  const uint8_t* k8;
  const uint8_t* v8;
  const float* ks;
  const float* vs;
  const int32_t* block_table;
  float* part_o;  // [T, Hq, nsplit, hd]
  float* part_ml; // [T, Hq, nsplit, 2]
  int* status;
  PieceMeta pm;
  int64_t max_blk, n_blocks;
  int Hq, Hkv, group, nsplit, split;  // split = positions per split
  float scale_log2;
  __nv_bfloat16* out;  // [T, Hq * hd]: FUSED decode only (the splits merged in the kernel)
};

constexpr int kRows = 64;   // query rows per CTA (4 warps x 16)
constexpr std::integral_constant<int, 32> kThr32{};    // copy loops of one warp
constexpr std::integral_constant<int, 128> kThr128{};  // copy loops of four warps
constexpr int kKeys = 64;   // keys per tile = cache block

// Per-row arithmetic (shared by the decode and the prefill schedule below):
// a split of S positions is cut into at most four "lanes" of lane_len =
// roundup(S / 4, 64) positions.  Inside a lane, 64-key tiles are taken in
// ascending order with an fp32 online softmax from a fresh (m, l, acc); the
// lane results are then merged in lane order 0, 1, 2, 3 (lanes with no key
// at or before the row's position are skipped).  The schedule decides only
// who computes a lane (all four warps in parallel for a decode tile, one warp
// after another for a prefill tile), never the arithmetic.

// Shared-memory byte offset of 16-byte chunk `ch` of key row `key` inside a
// 64-key tile: HD/64 boxes of 64 keys x 128 bytes, the chunks of each row
// XOR-swizzled by (key mod 8).  This is the layout a TMA copy with 128-byte
// swizzle writes for a 64x64 bf16 box at a 1024-byte aligned address, and the
// one the cp.async loader below reproduces; ldmatrix reads of 8 consecutive
// keys at one chunk hit 8 different bank groups.
template <int HD>
__device__ __forceinline__ uint32_t kv_off(int key, int ch) {
  return (uint32_t)((ch >> 3) * (kKeys * 128) + key * 128 + (((ch & 7) ^ (key & 7)) << 4));
}

// P = 2^x for the attention probabilities: the hardware's ex2 with results
// below 2^-126 flushed to zero (and 2^-inf = +0).  Every schedule, decode and
// prefill, takes P through this one instruction, so their bits stay equal.
__device__ __forceinline__ float exp2_p(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The warp's query rows: NH = 2 holds 16 rows per tile (thread (g, qd) rows g and
// g + 8), NH = 1 only rows 0..7 (decode tiles of at most 8 rows: GQA group x
// tokens).  At NH = 1 the m16n8k16 MMAs get zero A rows 8..15 and their D rows
// 8..15 are discarded; a D element depends only on its own A row and B column, so
// rows 0..7 are the same bits either way.
template <int NH>
__device__ __forceinline__ void mma_rows(float (&d)[2 * NH], const uint32_t (&a)[2 * NH], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (NH == 2) {
    mma_bf16_16816(d, a, b0, b1);
  } else {
    float t2, t3;  // rows 8..15 of D: discarded
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%10,%11};"
        : "+f"(d[0]), "+f"(d[1]), "=f"(t2), "=f"(t3)
        : "r"(a[0]), "r"(0u), "r"(a[1]), "r"(0u), "r"(b0), "r"(b1), "f"(0.f), "f"(0.f));
  }
}

// S = Q K^T for the warp's query rows and one 64-key tile (fp32, unscaled).
// qf[kk]: the rows' A fragment of head dims 16 kk .. 16 kk + 15 (h-th row half
// at [h] for dims + 0..7 and at [NH + h] for dims + 8..15).
template <int HD, int NH = 2>
__device__ __forceinline__ void attn_scores(uint32_t sk, const uint32_t (&qf)[HD / 16][2 * NH], int lane,
                                            float (&sc)[8][2 * NH]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int c = 0; c < 2 * NH; ++c) sc[j][c] = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int kk = 0; kk < HD / 16; kk += 2) {
      const int key = j * 8 + (lane & 7);
      const int ch = kk * 2 + (lane >> 3);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sk + kv_off<HD>(key, ch), b0, b1, b2, b3);
      mma_rows<NH>(sc[j], qf[kk], b0, b1);
      mma_rows<NH>(sc[j], qf[kk + 1], b2, b3);
    }
  }
}

// Fold one tile's scores into the online-softmax state of the warp's rows:
// masking by select, fp32 rescaling, then O += P V with P rounded to bf16.
// vsm (FP8 cache only): the tile's V scales; P is then multiplied by its key's
// scale before the bf16 rounding (exact: a power of two), so that P' V_codes has
// the products P (V_codes scale) term for term.
template <int HD, int NH = 2>
__device__ __forceinline__ void attn_update(uint32_t sv, float (&sc)[8][2 * NH], int key0, const bool (&row_valid)[2],
                                            const int (&row_pos)[2], float scale_log2, int lane, float (&m)[2],
                                            float (&l)[2], float (&acc)[HD / 8][2 * NH],
                                            const float* vsm = nullptr) {
  const int tq = lane & 3;
  float pr[8][2 * NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kp = key0 + j * 8 + tq * 2 + e;
        const bool ok = row_valid[h] && kp <= row_pos[h];
        const float v = ok ? __fmul_rn(sc[j][h * 2 + e], scale_log2) : -INFINITY;
        sc[j][h * 2 + e] = v;
        tmax = fmaxf(tmax, v);
      }
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m[h], tmax);
    const float alpha = (m_new == m[h]) ? 1.0f : exp2f(__fsub_rn(m[h], m_new));
    float rs = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = sc[j][h * 2 + e];
        const float pv = (v == -INFINITY) ? 0.f : exp2_p(__fsub_rn(v, m_new));
        pr[j][h * 2 + e] = pv;
        rs = __fadd_rn(rs, pv);
      }
    }
    rs = __fadd_rn(rs, __shfl_xor_sync(0xffffffffu, rs, 1));
    rs = __fadd_rn(rs, __shfl_xor_sync(0xffffffffu, rs, 2));
    l[h] = __fadd_rn(__fmul_rn(l[h], alpha), rs);
    m[h] = m_new;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
      acc[j][h * 2] = __fmul_rn(acc[j][h * 2], alpha);
      acc[j][h * 2 + 1] = __fmul_rn(acc[j][h * 2 + 1], alpha);
    }
  }
  if (vsm) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 vv = *reinterpret_cast<const float2*>(vsm + j * 8 + tq * 2);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        pr[j][h * 2] = __fmul_rn(pr[j][h * 2], vv.x);
        pr[j][h * 2 + 1] = __fmul_rn(pr[j][h * 2 + 1], vv.y);
      }
    }
  }
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {  // 64 keys = 4 k-steps of 16
    uint32_t pa[2 * NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      pa[h] = pack_bf16x2(pr[2 * kk][h * 2], pr[2 * kk][h * 2 + 1]);
      pa[NH + h] = pack_bf16x2(pr[2 * kk + 1][h * 2], pr[2 * kk + 1][h * 2 + 1]);
    }
#pragma unroll
    for (int j = 0; j < HD / 8; j += 2) {
      const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int ch = j + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sv + kv_off<HD>(key, ch), b0, b1, b2, b3);
      mma_rows<NH>(acc[j], pa, b0, b1);
      mma_rows<NH>(acc[j + 1], pa, b2, b3);
    }
  }
}

// One 64-key tile into the online-softmax state of 16 query rows (one warp).
// ksm / vsm (FP8 cache only): the tile holds unscaled e4m3 values and these are
// its per-key K and V scales.  A score column is multiplied by its key's K
// scale: Q (codes x 2^k)^T = 2^k (Q codes^T) exactly.
template <int HD, int NH = 2>
__device__ __forceinline__ void attn_tile(uint32_t sk, uint32_t sv, int key0, const uint32_t (&qf)[HD / 16][2 * NH],
                                          const bool (&row_valid)[2], const int (&row_pos)[2], float scale_log2,
                                          int lane, float (&m)[2], float (&l)[2], float (&acc)[HD / 8][2 * NH],
                                          const float* ksm = nullptr, const float* vsm = nullptr) {
  float sc[8][2 * NH];
  attn_scores<HD, NH>(sk, qf, lane, sc);
  if (ksm) {
    const int tq = lane & 3;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 kk = *reinterpret_cast<const float2*>(ksm + j * 8 + tq * 2);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        sc[j][h * 2] = __fmul_rn(sc[j][h * 2], kk.x);
        sc[j][h * 2 + 1] = __fmul_rn(sc[j][h * 2 + 1], kk.y);
      }
    }
  }
  attn_update<HD, NH>(sv, sc, key0, row_valid, row_pos, scale_log2, lane, m, l, acc, vsm);
}

// Per-thread state of one lane (its NH row halves), as stored in shared memory
// between lanes.
template <int HD, int NH = 2>
struct LaneState {
  float m[NH], l[NH];
  float acc[HD / 8][2 * NH];
};

// P <- P (+) Q for the rows a thread holds; an empty Q leaves P unchanged, an
// empty P takes Q as it is.
template <int HD, int NH = 2>
__device__ __forceinline__ void lane_merge(LaneState<HD, NH>& P, const float* mq, const float* lq,
                                           const float (&accq)[HD / 8][2 * NH]) {
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (mq[h] == -INFINITY) continue;
    if (P.m[h] == -INFINITY) {
      P.m[h] = mq[h];
      P.l[h] = lq[h];
#pragma unroll
      for (int j = 0; j < HD / 8; ++j) {
        P.acc[j][h * 2] = accq[j][h * 2];
        P.acc[j][h * 2 + 1] = accq[j][h * 2 + 1];
      }
      continue;
    }
    const float M = fmaxf(P.m[h], mq[h]);
    const float a = (P.m[h] == M) ? 1.0f : exp2f(__fsub_rn(P.m[h], M));
    const float b = (mq[h] == M) ? 1.0f : exp2f(__fsub_rn(mq[h], M));
    P.l[h] = __fadd_rn(__fmul_rn(P.l[h], a), __fmul_rn(lq[h], b));
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = h * 2 + e;
        P.acc[j][c] = __fadd_rn(__fmul_rn(P.acc[j][c], a), __fmul_rn(accq[j][c], b));
      }
    }
    P.m[h] = M;
  }
}

// Split partial of the rows a thread holds to the workspace.
template <int HD, int NH = 2>
__device__ __forceinline__ void write_partial(const AttnArgs& a, const LaneState<HD, NH>& P, const bool (&row_valid)[2],
                                              const int (&row_pos)[2], const int (&row_tok)[2],
                                              const int (&row_head)[2], int kv_begin, int s, int tq) {
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (!row_valid[h] || row_pos[h] < kv_begin) continue;
    const int64_t pidx = ((int64_t)row_tok[h] * a.Hq + row_head[h]) * a.nsplit + s;
    float* po = a.part_o + pidx * HD;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
      *reinterpret_cast<float2*>(po + j * 8 + tq * 2) = make_float2(P.acc[j][h * 2], P.acc[j][h * 2 + 1]);
    }
    if (tq == 0) *reinterpret_cast<float2*>(a.part_ml + pidx * 2) = make_float2(P.m[h], P.l[h]);
  }
}

// Query fragments (mma A layout) of the rows a thread holds; zero for invalid rows.
template <int HD, int NH = 2>
__device__ __forceinline__ void load_q_frags(const AttnArgs& a, const bool (&row_valid)[2], const int (&row_tok)[2],
                                             const int (&row_head)[2], int tq, uint32_t (&qf)[HD / 16][2 * NH]) {
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const __nv_bfloat16* qr = a.q + ((int64_t)row_tok[h] * a.Hq + row_head[h]) * HD + kk * 16 + tq * 2;
      qf[kk][h] = row_valid[h] ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
      qf[kk][NH + h] = row_valid[h] ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
    }
  }
}

// FUSED decode: the output of the two rows a thread holds from the partials of
// split 0 (P0) and split 1 (P1), with the split merge's arithmetic: M = max_s
// m_s, then L and O summed over s = 0, 1 in that order (a row whose position
// is before split 1 has only split 0), out = bf16(O / L).
template <int HD, int NH = 2>
__device__ __forceinline__ void fused_split_merge(const AttnArgs& a, const LaneState<HD, NH>& P0,
                                                  const LaneState<HD, NH>* P1, const bool (&row_valid)[2],
                                                  const int (&row_pos)[2], const int (&row_tok)[2],
                                                  const int (&row_head)[2], int tq) {
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (!row_valid[h]) continue;
    const int ns = merge_split_count(row_pos[h], a.split, a.nsplit, a.status, tq == 0);
    float M = fmaxf(-INFINITY, P0.m[h]);
    if (ns > 1) M = fmaxf(M, P1->m[h]);
    const float w0 = merge_weight(P0.m[h], M);
    const float w1 = ns > 1 ? merge_weight(P1->m[h], M) : 0.f;
    float L = merge_term(0.f, P0.l[h], w0);
    if (ns > 1) L = merge_term(L, P1->l[h], w1);
    __nv_bfloat16* orow = a.out + ((int64_t)row_tok[h] * a.Hq + row_head[h]) * HD;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
      float o[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        o[e] = merge_term(0.f, P0.acc[j][h * 2 + e], w0);
        if (ns > 1) o[e] = merge_term(o[e], P1->acc[j][h * 2 + e], w1);
        o[e] = __fdiv_rn(o[e], L);
      }
      __nv_bfloat162 v;
      v.x = f2bf(o[0]);
      v.y = f2bf(o[1]);
      *reinterpret_cast<__nv_bfloat162*>(orow + j * 8 + tq * 2) = v;
    }
  }
}

// One CTA per (piece, query tile, kv head, split), two schedules:
// PREFILL (64-row query tiles): warp w owns rows 16w..16w+15 and walks the
// split's tiles in order from a shared two-stage cp.async ring, folding each
// finished lane into a running state at every lane boundary.
// DECODE (query tiles of at most 16 rows, short contexts): warp w computes
// lane w of the split from its own buffers (bf16 caches: a three-tile cp.async
// ring of the lane's K and V tiles, two ahead of the one in use), then warp 0
// merges the lanes in order.  Tiles of at most 8 rows keep one row half.
// FUSED (DECODE with at most two splits): one CTA per (piece, query tile, kv
// head) covers both splits with eight warps, warp w computing lane w % 4 of
// split w / 4; warps 0 and 4 fold their split's lanes in order, and warp 0
// merges the two split partials with the split merge's formulas (ascending
// split order) and writes the output rows: no partials leave the CTA and no
// merge kernel runs.
// KV8: the cache holds e4m3 codes and per-(slot, kv head) scales.  Each tile's
// codes and scales are copied (cp.async) into a staging area, then expanded
// into the same swizzled bf16 tile the bf16 cache gives (code x power-of-two
// scale is exact in bf16), so every later step, and every bit, is unchanged.
template <int HD>
struct Kv8Stage {
  static constexpr int kCodes = kKeys * HD;                  // one page of K or V codes
  static constexpr int kBytes = 2 * kCodes + 2 * kKeys * 4;  // K codes, V codes, K scales, V scales
};

// Decode schedules: 64-key tiles of shared memory per warp (bf16 caches: a
// three-tile K/V ring; FP8 caches: the expanded K and V of one page).
template <bool KV8>
constexpr int kDecWarpTiles = KV8 ? 2 : 3;

template <int HD, bool DECODE, bool KV8, bool FUSED = false, int NH = 2>
__global__ void __launch_bounds__(FUSED ? 256 : 128) attention_kernel(const AttnArgs a) {
  static_assert(!FUSED || DECODE, "the fused split merge is a decode schedule");
  static_assert(NH == 2 || DECODE, "one row half only in decode tiles (at most 8 rows)");
  constexpr int CH = HD / 8;  // 16-byte chunks per key row
  constexpr int TILE_BYTES = kKeys * HD * 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_trigger();
  pdl_wait();
  const int p = blockIdx.y;
  const int kvh = FUSED ? (int)blockIdx.z : (int)blockIdx.z % a.Hkv;
  const int s = FUSED ? (int)(threadIdx.x >> 7) : (int)blockIdx.z / a.Hkv;
  const int row0 = a.pm.row0[p];
  const int n_tok = a.pm.row0[p + 1] - row0;
  const int tok_per_tile = (DECODE ? 8 * NH : kRows) / a.group;
  const int tok0 = blockIdx.x * tok_per_tile;
  if (tok0 >= n_tok) return;
  const int pos_first = a.pm.pos0[p];
  const int tok_last = min(n_tok, tok0 + tok_per_tile) - 1;
  const int max_pos = pos_first + tok_last;  // last query position in this CTA
  const int kv_begin = s * a.split;
  // a split entirely in the future of every row here: nothing to do (FUSED: this
  // half of the CTA only skips its lanes; split 0 always holds position 0)
  if (!FUSED && kv_begin > max_pos) return;
  const bool split_live = kv_begin <= max_pos;
  const int kv_end = min(kv_begin + a.split, max_pos + 1);  // exclusive
  const int lane_len = ((a.split + 3) / 4 + kKeys - 1) / kKeys * kKeys;
  const int seq = a.pm.seq[p];
  const int32_t* bt = a.block_table + (int64_t)seq * a.max_blk;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;

  // rows of this thread: r = (DECODE ? 0 : 16 * warp) + g + 8h
  int row_pos[2], row_tok[2], row_head[2];
  bool row_valid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = (DECODE ? 0 : warp * 16) + g + h * 8;
    const int ti = tok0 + r / a.group;
    row_valid[h] = h < NH && ti < n_tok && (r / a.group) < tok_per_tile;
    row_tok[h] = row0 + ti;
    row_pos[h] = pos_first + ti;
    row_head[h] = kvh * a.group + (r % a.group);
  }
  uint32_t qf[HD / 16][2 * NH];
  load_q_frags<HD, NH>(a, row_valid, row_tok, row_head, tq, qf);

  // copy one 64-key tile of K and V into (sk, sv) with threads t0, t0 + nthr, ...;
  // keys after max_pos are zero-filled.  nthr is a compile-time constant
  // (std::integral_constant) so that the copy loops unroll: a loop with
  // run-time bounds around each copy costs more issue slots than the copies.
  auto load_tile = [&](int key0, uint8_t* sk, uint8_t* sv, int t0, auto nthr_c) {
    constexpr int nthr = decltype(nthr_c)::value;
    const bool tab_ok = key0 / kKeys < a.max_blk;
    const int32_t blk = tab_ok ? bt[key0 / kKeys] : -1;
    const bool blk_ok = blk >= 0 && blk < a.n_blocks;
    if (!blk_ok && t0 == 0) report(a.status, DEV_BAD_INDEX);
    const int64_t base = ((int64_t)(blk_ok ? blk : 0) * a.Hkv + kvh) * kKeys * HD;
#pragma unroll
    for (int i = 0; i < kKeys * CH / nthr; ++i) {
      const int c = t0 + i * nthr;
      const int key = c / CH, ch = c % CH;
      const bool valid = blk_ok && (key0 + key) <= max_pos;
      const int off = (int)kv_off<HD>(key, ch);
      const int64_t src = base + (int64_t)key * HD + ch * 8;
      cp_async16(sk + off, a.k_cache + (valid ? src : 0), valid);
      cp_async16(sv + off, a.v_cache + (valid ? src : 0), valid);
    }
    cp_async_commit();
  };

  // one 64-key tile of K (v false) or V into dst (bf16 decode ring), as load_tile
  auto load_one = [&](int key0, uint8_t* dst, bool v, int t0, auto nthr_c) {
    constexpr int nthr = decltype(nthr_c)::value;
    const bool tab_ok = key0 / kKeys < a.max_blk;
    const int32_t blk = tab_ok ? bt[key0 / kKeys] : -1;
    const bool blk_ok = blk >= 0 && blk < a.n_blocks;
    if (!blk_ok && t0 == 0) report(a.status, DEV_BAD_INDEX);
    const int64_t base = ((int64_t)(blk_ok ? blk : 0) * a.Hkv + kvh) * kKeys * HD;
    const __nv_bfloat16* cache = v ? a.v_cache : a.k_cache;
#pragma unroll
    for (int i = 0; i < kKeys * CH / nthr; ++i) {
      const int c = t0 + i * nthr;
      const int key = c / CH, ch = c % CH;
      const bool valid = blk_ok && (key0 + key) <= max_pos;
      const int64_t src = base + (int64_t)key * HD + ch * 8;
      cp_async16(dst + kv_off<HD>(key, ch), cache + (valid ? src : 0), valid);
    }
    cp_async_commit();
  };

  // KV8: one tile's codes and scales into the staging area `stg`
  // (zero-filled where the block-table entry is bad or the key is in the future)
  auto load_tile8 = [&](int key0, uint8_t* stg, int t0, auto nthr_c) {
    constexpr int nthr = decltype(nthr_c)::value;
    constexpr int C16 = HD / 16;  // 16-code chunks per key row
    const bool tab_ok = key0 / kKeys < a.max_blk;
    const int32_t blk = tab_ok ? bt[key0 / kKeys] : -1;
    const bool blk_ok = blk >= 0 && blk < a.n_blocks;
    if (!blk_ok && t0 == 0) report(a.status, DEV_BAD_INDEX);
    const int64_t page = (int64_t)(blk_ok ? blk : 0) * a.Hkv + kvh;
#pragma unroll
    for (int i = 0; i < kKeys * C16 / nthr; ++i) {
      const int c = t0 + i * nthr;
      const bool valid = blk_ok && (key0 + c / C16) <= max_pos;
      const int64_t src = page * Kv8Stage<HD>::kCodes + (int64_t)c * 16;
      cp_async16(stg + c * 16, a.k8 + (valid ? src : 0), valid);
      cp_async16(stg + Kv8Stage<HD>::kCodes + c * 16, a.v8 + (valid ? src : 0), valid);
    }
    for (int c = t0; c < kKeys / 4; c += nthr) {  // 64 scales = 16 chunks of 4
      const int64_t src = page * kKeys + c * 4;
      cp_async16(stg + 2 * Kv8Stage<HD>::kCodes + c * 16, a.ks + (blk_ok ? src : 0), blk_ok);
      cp_async16(stg + 2 * Kv8Stage<HD>::kCodes + kKeys * 4 + c * 16, a.vs + (blk_ok ? src : 0), blk_ok);
    }
    cp_async_commit();
  };
  // KV8: expand a staged tile into swizzled bf16 K and V tiles of the unscaled
  // e4m3 values (the scales are applied to the scores and to P); keys after
  // max_pos become zeros with zero scales, whatever their slot holds
  auto expand_tile8 = [&](int key0, uint8_t* stg, uint8_t* sk, uint8_t* sv, int t0, auto nthr_c) {
    constexpr int nthr = decltype(nthr_c)::value;
    constexpr int C16 = HD / 16;
#pragma unroll 4
    for (int i = 0; i < 2 * kKeys * C16 / nthr; ++i) {
      const int c = t0 + i * nthr;
      const int which = c >= kKeys * C16;
      const int cc = which ? c - kKeys * C16 : c;
      const int key = cc / C16, c16 = cc % C16;
      const uint4 raw = *reinterpret_cast<const uint4*>(stg + which * Kv8Stage<HD>::kCodes + cc * 16);
      uint2 b0 = e4m3x4_to_bf16x4(raw.x), b1 = e4m3x4_to_bf16x4(raw.y);
      uint2 b2 = e4m3x4_to_bf16x4(raw.z), b3 = e4m3x4_to_bf16x4(raw.w);
      if (key0 + key > max_pos) b0 = b1 = b2 = b3 = make_uint2(0u, 0u);
      uint8_t* dst = which ? sv : sk;
      *reinterpret_cast<uint4*>(dst + kv_off<HD>(key, 2 * c16)) = make_uint4(b0.x, b0.y, b1.x, b1.y);
      *reinterpret_cast<uint4*>(dst + kv_off<HD>(key, 2 * c16 + 1)) = make_uint4(b2.x, b2.y, b3.x, b3.y);
    }
    float* sc8 = reinterpret_cast<float*>(stg + 2 * Kv8Stage<HD>::kCodes);  // K scales, then V scales
    for (int key = t0; key < kKeys; key += nthr)
      if (key0 + key > max_pos) sc8[key] = sc8[kKeys + key] = 0.f;
  };
  auto stage_ks = [&](const uint8_t* stg) {
    return reinterpret_cast<const float*>(stg + 2 * Kv8Stage<HD>::kCodes);
  };

  float m[2] = {-INFINITY, -INFINITY};
  float l[2] = {0.f, 0.f};
  float acc[HD / 8][2 * NH];
#pragma unroll
  for (int j = 0; j < HD / 8; ++j)
#pragma unroll
    for (int c = 0; c < 2 * NH; ++c) acc[j][c] = 0.f;

  LaneState<HD, NH> P;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    P.m[h] = -INFINITY;
    P.l[h] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < HD / 8; ++j)
#pragma unroll
    for (int c = 0; c < 2 * NH; ++c) P.acc[j][c] = 0.f;

  if constexpr (DECODE) {
    // ---- lane `warp` (FUSED: lane warp % 4 of split warp / 4), from this warp's own buffers
    constexpr int kWarps = FUSED ? 8 : 4;
    constexpr int kRegion = kDecWarpTiles<KV8> * TILE_BYTES;  // this warp's shared memory
    const int lb = kv_begin + (warp & 3) * lane_len;
    const int le = split_live ? min(lb + lane_len, kv_end) : lb;
    if constexpr (KV8) {
      uint8_t* sk = smem + warp * kRegion;
      uint8_t* sv = sk + TILE_BYTES;
      uint8_t* stg = smem + kWarps * kRegion + warp * Kv8Stage<HD>::kBytes;
      for (int key0 = lb; key0 < le; key0 += kKeys) {
        load_tile8(key0, stg, lane, kThr32);
        cp_async_wait<0>();
        __syncwarp();
        expand_tile8(key0, stg, sk, sv, lane, kThr32);
        __syncwarp();
        attn_tile<HD, NH>(smem_u32(sk), smem_u32(sv), key0, qf, row_valid, row_pos, a.scale_log2, lane, m, l, acc,
                          stage_ks(stg), stage_ks(stg) + kKeys);
        __syncwarp();
      }
    } else {
      // the lane's tiles K, V of each page in turn, tile j in buffer j % 3: two tiles
      // are in flight while one is used, and a buffer is refilled once it is read
      uint8_t* buf = smem + warp * kRegion;
      const int n_t = le > lb ? 2 * ((le - lb + kKeys - 1) / kKeys) : 0;
      auto issue = [&](int j) { load_one(lb + (j >> 1) * kKeys, buf + (j % 3) * TILE_BYTES, j & 1, lane, kThr32); };
      for (int j = 0; j < 3 && j < n_t; ++j) issue(j);
      float sc[8][2 * NH];
      for (int j = 0; j < n_t; ++j) {
        const int ahead = min(n_t, j + 3) - (j + 1);  // copy groups issued after tile j
        if (ahead >= 2) cp_async_wait<2>();
        else if (ahead == 1) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
        const uint32_t t = smem_u32(buf + (j % 3) * TILE_BYTES);
        if ((j & 1) == 0) attn_scores<HD, NH>(t, qf, lane, sc);
        else attn_update<HD, NH>(t, sc, lb + (j >> 1) * kKeys, row_valid, row_pos, a.scale_log2, lane, m, l, acc);
        __syncwarp();  // every lane has read tile j before its buffer takes tile j + 3
        if (j + 3 < n_t) issue(j + 3);
      }
    }
    // lanes meet in shared memory (each warp reuses its buffers); warp 0 merges 0..3
    LaneState<HD, NH>* st = reinterpret_cast<LaneState<HD, NH>*>(smem + warp * kRegion) + lane;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      st->m[h] = m[h];
      st->l[h] = l[h];
    }
#pragma unroll
    for (int j = 0; j < HD / 8; ++j)
#pragma unroll
      for (int c = 0; c < 2 * NH; ++c) st->acc[j][c] = acc[j][c];
    __syncthreads();
    if constexpr (FUSED) {
      // warps 0 and 4 fold the lanes of splits 0 and 1; warp 4 leaves its partial in its buffer
      if ((warp & 3) == 0 && split_live) {
        const int n_lanes = (kv_end - kv_begin + lane_len - 1) / lane_len;
        for (int w = 0; w < n_lanes; ++w) {
          const LaneState<HD, NH>* q =
              reinterpret_cast<const LaneState<HD, NH>*>(smem + (warp + w) * kRegion) + lane;
          lane_merge<HD, NH>(P, q->m, q->l, q->acc);
        }
        if (warp == 4) *(reinterpret_cast<LaneState<HD, NH>*>(smem + 4 * kRegion) + lane) = P;
      }
      __syncthreads();
      if (warp == 0)
        fused_split_merge<HD, NH>(a, P, reinterpret_cast<const LaneState<HD, NH>*>(smem + 4 * kRegion) + lane,
                                  row_valid, row_pos, row_tok, row_head, tq);
      return;
    }
    if (warp != 0) return;
    const int n_lanes = (kv_end - kv_begin + lane_len - 1) / lane_len;
    for (int w = 0; w < n_lanes; ++w) {
      const LaneState<HD, NH>* q = reinterpret_cast<const LaneState<HD, NH>*>(smem + w * kRegion) + lane;
      lane_merge<HD, NH>(P, q->m, q->l, q->acc);
    }
  } else {
    // ---- all warps share a two-stage ring; lanes are walked in order
    // bf16: two K+V tiles (the ring), then the running states.  KV8: one K+V
    // tile, the running states, then two staging areas (the ring).
    constexpr int kTiles = KV8 ? 1 : 2;
    LaneState<HD>* run = reinterpret_cast<LaneState<HD>*>(smem + kTiles * 2 * TILE_BYTES) + tid;
    uint8_t* stg0 = smem + kTiles * 2 * TILE_BYTES + 128 * sizeof(LaneState<HD>);
    *run = P;
    const int t_begin = kv_begin / kKeys;
    const int n_tiles = (kv_end - kv_begin + kKeys - 1) / kKeys;
    const int tiles_per_lane = lane_len / kKeys;
    if constexpr (KV8) load_tile8(t_begin * kKeys, stg0, tid, kThr128);
    else load_tile(t_begin * kKeys, smem, smem + TILE_BYTES, tid, kThr128);
    for (int t = 0; t < n_tiles; ++t) {
      const int stage = t & 1;
      uint8_t* sk = smem + (KV8 ? 0 : stage) * 2 * TILE_BYTES;
      if (t + 1 < n_tiles) {
        if constexpr (KV8) {
          load_tile8((t_begin + t + 1) * kKeys, stg0 + (stage ^ 1) * Kv8Stage<HD>::kBytes, tid, kThr128);
        } else {
          uint8_t* nk = smem + (stage ^ 1) * 2 * TILE_BYTES;
          load_tile((t_begin + t + 1) * kKeys, nk, nk + TILE_BYTES, tid, kThr128);
        }
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      if constexpr (KV8) {
        expand_tile8((t_begin + t) * kKeys, stg0 + stage * Kv8Stage<HD>::kBytes, sk, sk + TILE_BYTES, tid, kThr128);
        __syncthreads();
      }
      if (t > 0 && t % tiles_per_lane == 0) {  // lane boundary: fold the finished lane in
        LaneState<HD> r = *run;
        lane_merge<HD>(r, m, l, acc);
        *run = r;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int j = 0; j < HD / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
      }
      const uint8_t* stg_t = stg0 + stage * Kv8Stage<HD>::kBytes;
      attn_tile<HD>(smem_u32(sk), smem_u32(sk + TILE_BYTES), (t_begin + t) * kKeys, qf, row_valid, row_pos,
                    a.scale_log2, lane, m, l, acc, KV8 ? stage_ks(stg_t) : nullptr,
                    KV8 ? stage_ks(stg_t) + kKeys : nullptr);
      __syncthreads();
    }
    P = *run;
    lane_merge<HD>(P, m, l, acc);
  }
  write_partial<HD, NH>(a, P, row_valid, row_pos, row_tok, row_head, kv_begin, s, tq);
}

// ------------------------------------------------- tensor-memory prefill schedule
// PREFILL on the 5th-generation tensor cores, for bf16 caches: a CTA owns
// (piece, 128-row query tile, kv head, split); rows are the (token, q head of
// the group) pairs as above.  S = Q K^T (K = hd in 16-wide steps, ascending)
// and O += P V (K = 64 keys in 16-wide steps, ascending) accumulate in TMEM;
// tcgen05.mma and mma.sync give the same fp32 bits step for step, so each row
// gets exactly the arithmetic of the mma.sync schedules.  The eight softmax
// warps read S and O through the 16x256b TMEM shape, which gives a warp 16 rows
// in the mma.sync accumulator layout: the four threads of a quad are one row and
// thread q holds the keys 8j + 2q + {0, 1} of the tile, i.e. exactly the keys of
// the mma.sync fragment's quad sum s_q.  They repeat attn_update's operations in
// its order: scale and select-mask, the tile max (quad shuffles), alpha,
// P = exp2(v - m), s_q summed over its keys in order and the row sum formed as
// (s0 + s1) + (s2 + s3), l = l alpha + sum, O = O alpha (skipped when alpha is
// exactly 1, where it is the identity), P rounded to bf16; and at every lane
// boundary the finished lane folds into the running state (held in registers)
// with lane_merge's formula.
// A CTA walks up to kTcSplitsPerCta consecutive splits of its query tile, one
// after another (each split's partial is written when the next one starts), so
// the Q tile, TMEM and the page pipeline serve many tiles.
// The warp after the softmax warps streams the K and V pages by TMA (lane 0; the
// persistent decode kernel's tensor maps) into a ring; the next one owns TMEM and
// its lane 0 issues the MMAs, S of the next tile ahead of P V of this one.  V rows after
// the CTA's last query position are zeroed in shared memory before P V (TMA
// copies whole pages, and slots not yet written may hold anything); K rows
// there only feed scores that the select-mask replaces.
constexpr int kTcSplitsPerCta = 4;

template <int HD>
struct TcAttnLayout {
  static constexpr int kQ = 128 * HD * 2;           // HD/64 boxes of 128 rows x 128 bytes
  static constexpr int kPage = kKeys * HD * 2;      // one K or V page
  static constexpr int kStages = HD == 128 ? 3 : 4;
  static constexpr int kP = 128 * kKeys * 2;        // one P tile, 128 rows x 64 keys
  static constexpr int kOffKV = kQ;
  static constexpr int kOffP = kOffKV + kStages * 2 * kPage;
  static constexpr int kOffBar = kOffP + 2 * kP;
  static constexpr int kBytes = kOffBar + 256 + 1024;   // + barriers, + alignment slack
  static constexpr uint32_t kCols = 256;  // S0, S1 (64 each), O (HD); the lane accumulator R is in registers
  static constexpr uint32_t kColS = 0, kColO = 128;
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kThreads = 32 * kSoftmaxWarps + 64;  // + TMA warp, MMA warp
};

template <int HD>
__global__ void __launch_bounds__(TcAttnLayout<HD>::kThreads, 1)
    attention_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
  using Lay = TcAttnLayout<HD>;
  constexpr int NS = Lay::kStages;
  constexpr int KB = HD / 64;        // 64-dim boxes per row
  constexpr int kSM = Lay::kSoftmaxWarps * 32;
  constexpr int kWarpTma = Lay::kSoftmaxWarps, kWarpMma = Lay::kSoftmaxWarps + 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + Lay::kOffKV;  // stage st: K page at st * 2 * kPage, V page after it
  uint8_t* sP = smem + Lay::kOffP;
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* kv_empty = kv_full + NS;
  uint64_t* s_full = kv_empty + NS;   // [2] MMA -> softmax: S of a tile is in TMEM
  uint64_t* s_empty = s_full + 2;     // [2] softmax -> MMA: S read (16 warp arrivals)
  uint64_t* p_full = s_empty + 2;     // [2] softmax -> MMA: P written, O rescaled (16 warp arrivals)
  uint64_t* o_done = p_full + 2;      // MMA -> softmax: P V of a tile has completed
  uint64_t* q_full = o_done + 1;      // softmax -> MMA: Q tile loaded (kSM thread arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = blockIdx.y;
  const int kvh = blockIdx.z % a.Hkv;
  const int s0 = (blockIdx.z / a.Hkv) * kTcSplitsPerCta;  // first split of this CTA
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], Lay::kSoftmaxWarps);
      mbar_init(&p_full[i], Lay::kSoftmaxWarps);
    }
    mbar_init(o_done, 1);
    mbar_init(q_full, kSM);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, Lay::kCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // dependents may launch only once this CTA holds its TMEM columns
  pdl_trigger();
  pdl_wait();

  const int row0 = a.pm.row0[p];
  const int n_tok = a.pm.row0[p + 1] - row0;
  const int tok_per_tile = 128 / a.group;
  const int tok0 = blockIdx.x * tok_per_tile;
  const int pos_first = a.pm.pos0[p];
  // tiles of this CTA's splits in order: every split before the last live one is
  // whole (ntf tiles), so tile k is tile k % ntf of split s0 + k / ntf
  const int ntf = a.split / kKeys;
  int n_tiles = 0, max_pos = -1;
  if (tok0 < n_tok) {
    max_pos = pos_first + min(n_tok, tok0 + tok_per_tile) - 1;
    const int s_last = min(min(s0 + kTcSplitsPerCta, a.nsplit) - 1, max_pos / a.split);
    if (s_last >= s0) {
      const int kb = s_last * a.split;
      n_tiles = (s_last - s0) * ntf + (min(kb + a.split, max_pos + 1) - kb + kKeys - 1) / kKeys;
    }
  }
  const int tpl = (((a.split + 3) / 4 + kKeys - 1) / kKeys * kKeys) / kKeys;  // tiles per lane
  const int seq = a.pm.seq[p];
  const int32_t* bt = a.block_table + (int64_t)seq * a.max_blk;
  // first key of tile k (absolute position)
  auto tile_key0 = [&](int k) { return (s0 + k / ntf) * a.split + (k % ntf) * kKeys; };

  if (n_tiles > 0 && warp == kWarpTma) {
    if (lane == 0) {
      // ---------------- TMA producer: K and V pages of the split's tiles, in order
      const int rows_total = (int)(a.n_blocks * a.Hkv * kKeys);
      int t = 0;
      for (; t < n_tiles && !*abort_flag; ++t) {
        const int st = t % NS;
        if (t >= NS && !mbar_wait(&kv_empty[st], ((t / NS) - 1) & 1)) {
          report(a.status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const int blk_i = tile_key0(t) / kKeys;
        const int32_t blk = blk_i < a.max_blk ? bt[blk_i] : -1;
        int row = rows_total;  // past the end: the copy reads zeros
        if (blk >= 0 && blk < a.n_blocks) row = (int)((blk * a.Hkv + kvh) * kKeys);
        else report(a.status, DEV_BAD_INDEX);
        uint8_t* sk = sKV + st * 2 * Lay::kPage;
        mbar_arrive_expect_tx(&kv_full[st], 2 * Lay::kPage);
#pragma unroll
        for (int b = 0; b < KB; ++b) {
          tma_load_2d(sk + b * (kKeys * 128), &tmk, &kv_full[st], b * 64, row);
          tma_load_2d(sk + Lay::kPage + b * (kKeys * 128), &tmv, &kv_full[st], b * 64, row);
        }
      }
      // the copies this CTA started land before it can exit
      for (int i = 0; i < NS && i < t; ++i) {
        const int tt = t - 1 - i;
        mbar_wait(&kv_full[tt % NS], (tt / NS) & 1);
      }
    }
  } else if (n_tiles > 0 && warp == kWarpMma) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKeys);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD) | (1u << 16);  // V read MN-major
      bool ok = mbar_wait(q_full, 0);
      auto issue_s = [&](int j) -> bool {
        const int st = j % NS;
        if (!mbar_wait(&kv_full[st], (j / NS) & 1)) return false;
        if (j >= 2 && !mbar_wait(&s_empty[j & 1], ((j - 2) >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(sQ), ka = smem_u32(sKV + st * 2 * Lay::kPage);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * (128 * 128) + (k & 3) * 32, koff = (k >> 2) * (kKeys * 128) + (k & 3) * 32;
          tc_mma_bf16(tmem + Lay::kColS + (j & 1) * kKeys, sw128_kmajor_desc(qa + off),
                      sw128_kmajor_desc(ka + koff), idesc_s, k != 0 ? 1u : 0u);
        }
        tc_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int t = 0; ok && t < n_tiles && !*abort_flag; ++t) {
        if (t + 1 < n_tiles && !issue_s(t + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&p_full[t & 1], (t >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = t % NS;
        const uint32_t pa = smem_u32(sP + (t & 1) * Lay::kP), va = smem_u32(sKV + st * 2 * Lay::kPage + Lay::kPage);
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          tc_mma_bf16(tmem + Lay::kColO, sw128_kmajor_desc(pa + k * 32),
                      sw128_mnmajor_desc(va + k * 16 * 128, kKeys * 128, 1024), idesc_o, 1u);
        tc_commit(o_done);
        tc_commit(&kv_empty[st]);
      }
      if (!ok) {
        report(a.status, DEV_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (n_tiles > 0 && warp < Lay::kSoftmaxWarps) {
    // ---------------- softmax warps.  Warp w holds the 16 rows rb .. rb + 15, rb =
    // 32 (w % 4) + 16 (w / 4) (TMEM lanes; a warp reads only its lane quarter), in the
    // mma.sync accumulator layout that the 16x256b TMEM shape gives: thread (g, qd) =
    // (lane / 4, lane % 4) holds rows rb + g and rb + g + 8 and, of every 8-column group
    // of S, O and R, the columns 2 qd + {0, 1}.  So a row's keys 8j + 2qd + {0, 1} are this
    // thread's, the quad's four threads are the row, and the row max and sum are quad
    // shuffles, exactly as in the mma.sync schedules.
    const int g = lane >> 2, qd = lane & 3;
    const int rb = 32 * (warp & 3) + 16 * (warp >> 2);
    int r[2], row_tok[2], row_pos[2], row_head[2];
    bool row_valid[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      r[h] = rb + g + 8 * h;
      const int ti = tok0 + r[h] / a.group;
      row_valid[h] = ti < n_tok;
      row_tok[h] = row0 + ti;
      row_pos[h] = pos_first + ti;
      row_head[h] = kvh * a.group + (r[h] % a.group);
    }
    // the Q tile into the swizzled layout (zeros for rows past the piece), 16-byte
    // chunks spread over the softmax threads
    for (int i = tid; i < 128 * (HD / 8); i += kSM) {
      const int qrow = i / (HD / 8), ch = i % (HD / 8);
      const int ti = tok0 + qrow / a.group;
      const bool valid = ti < n_tok;
      const __nv_bfloat16* src =
          a.q + ((int64_t)(row0 + ti) * a.Hq + kvh * a.group + (qrow % a.group)) * HD + ch * 8;
      uint8_t* dst = sQ + (ch >> 3) * (128 * 128) + qrow * 128 + (((ch & 7) ^ (qrow & 7)) << 4);
      cp_async16(dst, valid ? src : a.q, valid);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async();
    mbar_arrive(q_full);

    const uint32_t tblk = tmem + ((uint32_t)rb << 16);
    const uint32_t tS = tblk + Lay::kColS, tO = tblk + Lay::kColO;
    // register i of a 16-register O group at column c0 is row (i >> 1) & 1, column
    // c0 + 8 (i >> 2) + 2 qd + (i & 1); the lane accumulator R holds the same elements,
    // R[c0 / 2 + i], in registers
    constexpr int NR = HD / 2;
    float R[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) R[i] = 0.f;
    auto zero_o = [&]() {
      uint32_t z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
      for (int c = 0; c < HD; c += 32) tmem_st_16x256b_x4(tO + c, z);
      tmem_st_wait();
    };
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float Rm[2] = {-INFINITY, -INFINITY}, Rl[2] = {0.f, 0.f};
    // R <- lane_merge(R, (m, l, O)) per row: R a + O b, or a copy into an empty R
    auto fold_lane = [&](const float (&mq)[2], const float (&lq)[2]) {
      bool has[2], copy[2];
      float M[2], fa[2], fb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        has[h] = mq[h] != -INFINITY;
        copy[h] = has[h] && Rm[h] == -INFINITY;
        M[h] = fmaxf(Rm[h], mq[h]);
        fa[h] = (Rm[h] == M[h]) ? 1.0f : exp2f(__fsub_rn(Rm[h], M[h]));
        fb[h] = (mq[h] == M[h]) ? 1.0f : exp2f(__fsub_rn(mq[h], M[h]));
      }
      if (__any_sync(0xffffffffu, has[0] || has[1])) {
#pragma unroll
        for (int c = 0; c < HD; c += 64) {  // two O groups per TMEM round trip
          uint32_t oo[2][16];
          tmem_ld_16x256b_x4(tO + c, oo[0]);
          tmem_ld_16x256b_x4(tO + c + 32, oo[1]);
          tmem_ld_wait();
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int h = (i >> 1) & 1, ri = (c + 32 * b) / 2 + i;
              const float rv = R[ri], ov = __uint_as_float(oo[b][i]);
              R[ri] = copy[h] ? ov : (has[h] ? __fadd_rn(__fmul_rn(rv, fa[h]), __fmul_rn(ov, fb[h])) : rv);
            }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (copy[h]) {
          Rm[h] = mq[h];
          Rl[h] = lq[h];
        } else if (has[h]) {
          Rl[h] = __fadd_rn(__fmul_rn(Rl[h], fa[h]), __fmul_rn(lq[h], fb[h]));
          Rm[h] = M[h];
        }
      }
    };
    // every decision that gates a warp-collective tcgen05.ld / st is taken for the
    // whole warp at once (a wait that gives up on any lane stops all of them)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool got = mbar_wait(bar, parity) && !*abort_flag;
      return __all_sync(0xffffffffu, got);
    };
    // the rows' partials (m, l, acc) of split s from R; every lane loads, rows that
    // have no key in the split store nothing
    auto write_partial = [&](int s) {
      bool store[2];
      int64_t pidx[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        store[h] = row_valid[h] && row_pos[h] >= s * a.split;
        pidx[h] = ((int64_t)row_tok[h] * a.Hq + row_head[h]) * a.nsplit + s;
      }
#pragma unroll
      for (int c = 0; c < HD; c += 32)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (store[h])
              *reinterpret_cast<float2*>(a.part_o + pidx[h] * HD + c + 8 * k + 2 * qd) =
                  make_float2(R[c / 2 + 4 * k + 2 * h], R[c / 2 + 4 * k + 2 * h + 1]);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (store[h] && qd == 0) *reinterpret_cast<float2*>(a.part_ml + pidx[h] * 2) = make_float2(Rm[h], Rl[h]);
    };
    zero_o();
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int key0 = tile_key0(t);
      const int tt = t % ntf;                                  // tile within its split
      const bool split_start = t > 0 && tt == 0;               // a new split: finish the previous one
      const bool lane_start = split_start || (tt > 0 && tt % tpl == 0);
      if (!warp_wait(&s_full[t & 1], (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // v[h][2j + e] is the score of key 8j + 2qd + e of the tile for row h
      float v[2][16];
      {
        uint32_t sa[16], sb[16];
        tmem_ld_16x256b_x4(tS + (t & 1) * kKeys, sa);
        tmem_ld_16x256b_x4(tS + (t & 1) * kKeys + 32, sb);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              v[h][2 * j + e] = __uint_as_float(sa[4 * j + 2 * h + e]);
              v[h][8 + 2 * j + e] = __uint_as_float(sb[4 * j + 2 * h + e]);
            }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[t & 1]);
      // a new lane starts from a fresh state; the finished one is folded into R
      // once its last P V has landed (below), so this tile's softmax runs while
      // the tensor core finishes the previous tile
      const float m_done[2] = {m[0], m[1]}, l_done[2] = {l[0], l[1]};
      if (lane_start) {
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
      }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // scale and mask (a tile wholly at or before the row's position needs no
        // mask), the tile max over the quad (the max of a set does not depend on
        // the order it is taken in)
        const bool open = row_valid[h] && key0 + kKeys - 1 <= row_pos[h];
        if (open) {
#pragma unroll
          for (int c = 0; c < 16; ++c) v[h][c] = __fmul_rn(v[h][c], a.scale_log2);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int key = key0 + 8 * (c >> 1) + 2 * qd + (c & 1);
            v[h][c] = (row_valid[h] && key <= row_pos[h]) ? __fmul_rn(v[h][c], a.scale_log2) : -INFINITY;
          }
        }
        float mx = v[h][0];
#pragma unroll
        for (int c = 1; c < 16; ++c) mx = fmaxf(mx, v[h][c]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m[h], mx);
        alpha[h] = (m_new == m[h]) ? 1.0f : exp2f(__fsub_rn(m[h], m_new));
        // P and this thread's quad sum s_qd over its keys in order (a score of an
        // open tile is never -inf, so the select is the identity there); the row
        // sum is (s0 + s1) + (s2 + s3)
        float sq = 0.f;
        if (open) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            v[h][c] = exp2_p(__fsub_rn(v[h][c], m_new));
            sq = __fadd_rn(sq, v[h][c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            v[h][c] = (v[h][c] == -INFINITY) ? 0.f : exp2_p(__fsub_rn(v[h][c], m_new));
            sq = __fadd_rn(sq, v[h][c]);
          }
        }
        const float s2 = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, 1));
        const float rs = __fadd_rn(s2, __shfl_xor_sync(0xffffffffu, s2, 2));
        l[h] = __fadd_rn(__fmul_rn(l[h], alpha[h]), rs);
        m[h] = m_new;
      }
      if (t > 0) {  // P V of the previous tile has landed in O
        if (!warp_wait(o_done, (t - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (lane_start) {
        fold_lane(m_done, l_done);
        if (split_start) {
          write_partial(s0 + t / ntf - 1);
          Rm[0] = Rm[1] = -INFINITY;  // the next fold copies into R
          Rl[0] = Rl[1] = 0.f;
        }
        zero_o();
      }
      // O = O alpha (identity where alpha == 1; O is +0 at a lane's first tile)
      if (t > 0 && !lane_start && __any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
        for (int c = 0; c < HD; c += 64) {  // two O groups per TMEM round trip
          uint32_t oo[2][16];
          tmem_ld_16x256b_x4(tO + c, oo[0]);
          tmem_ld_16x256b_x4(tO + c + 32, oo[1]);
          tmem_ld_wait();
#pragma unroll
          for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              oo[b][i] = __float_as_uint(__fmul_rn(__uint_as_float(oo[b][i]), alpha[(i >> 1) & 1]));
            tmem_st_16x256b_x4(tO + c + 32 * b, oo[b]);
          }
        }
        tmem_st_wait();
      }
      // the last tile may hold keys after the CTA's last position: zero those V rows
      const int st = t % NS;
      if (key0 + kKeys - 1 > max_pos) {
        if (!warp_wait(&kv_full[st], (t / NS) & 1)) {
          ok = false;
          break;
        }
        uint8_t* sv = sKV + st * 2 * Lay::kPage + Lay::kPage;
        for (int i = tid; i < kKeys * KB * 8; i += kSM) {  // (key, 16-byte chunk): whole rows, any chunk order
          const int key = i / (KB * 8), ch = i % (KB * 8);
          if (key0 + key > max_pos)
            *reinterpret_cast<uint4*>(sv + (ch >> 3) * (kKeys * 128) + key * 128 + ((ch & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // the rows' P in bf16: keys 8j + 2qd + {0, 1} are bytes 4qd .. 4qd + 3 of the
      // row's 16-byte chunk j in the swizzled P tile
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint8_t* prow = sP + (t & 1) * Lay::kP + r[h] * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint32_t*>(prow + ((j ^ (r[h] & 7)) << 4) + 4 * qd) =
              pack_bf16x2(v[h][2 * j], v[h][2 * j + 1]);
      }
      fence_proxy_async();
      tc_fence_before();
      // this warp's rows of P (and its share of the zeroed V rows) are written;
      // the MMA waits for all the softmax warps
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t & 1]);
    }
    if (ok && warp_wait(o_done, (n_tiles - 1) & 1)) {
      tc_fence_after();
      fold_lane(m, l);
      write_partial(s0 + (n_tiles - 1) / ntf);
    } else {
      report(a.status, DEV_TIMEOUT);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kCols);
  }
}

// ----------------------------------------------------------- decode schedule
// Persistent DECODE schedule, for query tiles of at most 16 rows over long
// contexts: the same per-row arithmetic as above, with the four lanes of a
// split computed in parallel by four warps and merged in lane order by warp 0.
// The kernel is
// persistent (one or two CTAs per SM walk the work items (piece, split, kv
// head) with a grid stride; each CTA first counts every piece's live splits
// into a prefix table in shared memory) and warp-specialised:
//   * warp 4 reads block-table entries and issues 128-byte-swizzled TMA copies
//     of each 64-key K and V page into a kDecSlots-deep ring per consumer warp,
//     running ahead across work items;
//   * warps 0..3 compute lane w of each item from ring w: scores from the K
//     page, then softmax and P*V from the V page, releasing each slot as soon
//     as it is read;
//   * at the end of an item warps 1..3 hand their lane state to warp 0 through
//     shared memory (named barriers 1 and 2), and warp 0 merges and writes the
//     split partial.
// TMA copies whole pages, so V rows after the item's last position (slots not
// yet written in the cache) are zeroed in shared memory before P*V; K rows
// there only feed scores that the select-mask replaces with -inf.
constexpr int kDecMaxPieces = 1024;      // larger decode calls take the per-CTA schedule (same bits)
constexpr int kDecPersistentSplits = 4;  // shorter contexts take the per-CTA schedule (same bits)

// KV8 (FP8 cache): eight loader warps replace the producer, two per consumer
// ring: warp 4 + w loads consumer w's K pages, warp 8 + w its V pages.  A
// loader walks the items as consumer w does and copies each of its pages' e4m3
// codes (64 rows x hd bytes, unswizzled) and 64 fp32 scales with TMA into its
// code slot, one page ahead; it expands the landed page a quarter at a time
// into its slot of the consumer's bf16 ring (the swizzled layout ldmatrix
// reads), rows and scales after the item's last position zero, and copies the
// next page into the code slot as soon as the last quarter and the scales are
// read.  The consumer runs the bf16 schedule on that page with the scales
// applied.  The consumers' warpgroup takes kConsumerRegs registers a thread and
// the two loader warpgroups kLoaderRegs (setmaxnreg), within the 168 a thread
// that 384 threads launch with (the host checks the compiled count).
template <int HD, bool KV8 = false, int NH = 2>
struct DecLayout {
  static constexpr int kThreads = KV8 ? 384 : 160;  // consumers, then producer (KV8: eight loaders)
  static constexpr int kLaunchRegs = 168;           // KV8: 65536 / 384, rounded down to a multiple of 8
  static constexpr int kConsumerRegs = 240, kLoaderRegs = 128;
  static_assert(!KV8 || 128 * kConsumerRegs + 256 * kLoaderRegs <= kThreads * kLaunchRegs, "register split");
  // bf16 ring depth per consumer warp: three slots at hd 128 (one CTA per SM);
  // two at hd 64 (two CTAs share an SM) and on an FP8 cache (two code slots
  // more per ring)
  static constexpr int kDecSlots = (HD == 64 || KV8) ? 2 : 3;
  static constexpr int kCodeSlots = 2;
  static constexpr int kTile = kKeys * HD * 2;                       // one bf16 K or V page
  static constexpr int kCodes = kKeys * HD;                          // one page of codes
  static constexpr int kCodeSlot = kCodes + kKeys * 4;               // codes, then scales
  static constexpr int kRing = 4 * kDecSlots * kTile;                // four bf16 rings
  static constexpr int kScales = kRing;                              // KV8: [4][kDecSlots][64] fp32
  static constexpr int kCodeRing = kScales + (KV8 ? 4 * kDecSlots * kKeys * 4 : 0);  // KV8: [4][2] code slots
  static constexpr int kStates = kCodeRing + (KV8 ? 4 * kCodeSlots * kCodeSlot : 0);  // lane states of warps 1..3
  static constexpr int kTable = kStates + 3 * 32 * (int)sizeof(LaneState<HD, NH>);  // int [kDecMaxPieces + 1]
  static constexpr int kBars = kTable + (kDecMaxPieces + 2) * 4;
  // full[4][S] (bf16: TMA -> consumer; KV8: code TMA -> loader, [4][2]), empty[4][S]
  // (consumer -> producer / loader), KV8 conv[4][S] (loader -> consumer)
  static constexpr int kNBars = (KV8 ? 3 : 2) * 4 * kDecSlots;
  static constexpr int kAbort = kBars + kNBars * 8;
  static constexpr int kBytes = kAbort + 16 + 1024;                  // + alignment slack
  static_assert(kBars % 8 == 0 && kCodeSlot % 128 == 0, "alignment");
  static_assert(!KV8 || kCodeSlots == kDecSlots, "one full barrier per code slot");
  static_assert(kBytes <= 232448, "decode schedule exceeds the shared-memory limit");
};

// Work items are (piece, split, kv head) with the split at or before the
// piece's last position, numbered piece by piece: item j belongs to the last
// piece p with first[p] <= j, and j - first[p] = split * Hkv + kv head.
struct DecItem {
  int p, s, kvh, n_tok, row0, pos_first, max_pos, kv_begin, kv_end, seq;
};

__device__ __forceinline__ DecItem dec_item(const AttnArgs& a, const int* first, int j, int P) {
  int lo = 0, hi = P - 1;  // first[lo] <= j < first[P]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (first[mid] <= j) lo = mid;
    else hi = mid - 1;
  }
  DecItem it;
  it.p = lo;
  const int r = j - first[lo];
  it.s = r / a.Hkv;
  it.kvh = r % a.Hkv;
  it.row0 = a.pm.row0[it.p];
  it.n_tok = a.pm.row0[it.p + 1] - it.row0;
  it.pos_first = a.pm.pos0[it.p];
  it.seq = a.pm.seq[it.p];
  it.max_pos = it.pos_first + it.n_tok - 1;
  it.kv_begin = it.s * a.split;
  it.kv_end = min(it.kv_begin + a.split, it.max_pos + 1);
  return it;
}

// Bounded mbarrier wait that also gives up once another warp has set *abort.
__device__ __forceinline__ bool dec_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(addr, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      report(status, DEV_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// KV8 loader step: a quarter of the codes of one page (64 rows x hd bytes), as
// this lane's uint4 chunks lane + 32 u of the quarter, and their expansion into
// the swizzled bf16 page of unscaled values, rows at or after nk zero.  One warp.
template <int HD>
struct DecCodes {
  static constexpr int C16 = HD / 16;              // 16-code chunks per key row
  static constexpr int kParts = 4;
  static constexpr int kPart = kKeys * C16 / (32 * kParts);  // chunks per lane and part
  uint4 raw[kPart];
  __device__ __forceinline__ void load(const uint8_t* codes, int lane, int part) {
#pragma unroll
    for (int u = 0; u < kPart; ++u)
      raw[u] = *reinterpret_cast<const uint4*>(codes + (lane + 32 * (part * kPart + u)) * 16);
  }
  __device__ __forceinline__ void expand(uint8_t* page, int nk, int lane, int part) const {
#pragma unroll
    for (int u = 0; u < kPart; ++u) {
      const int i = lane + 32 * (part * kPart + u), key = i / C16, c16 = i % C16;
      uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
      if (key < nk) {
        const uint2 b0 = e4m3x4_to_bf16x4(raw[u].x), b1 = e4m3x4_to_bf16x4(raw[u].y);
        const uint2 b2 = e4m3x4_to_bf16x4(raw[u].z), b3 = e4m3x4_to_bf16x4(raw[u].w);
        lo = make_uint4(b0.x, b0.y, b1.x, b1.y);
        hi = make_uint4(b2.x, b2.y, b3.x, b3.y);
      }
      *reinterpret_cast<uint4*>(page + kv_off<HD>(key, 2 * c16)) = lo;
      *reinterpret_cast<uint4*>(page + kv_off<HD>(key, 2 * c16 + 1)) = hi;
    }
  }
};

template <int HD, bool KV8, int NH>
__global__ void __launch_bounds__(DecLayout<HD, KV8, NH>::kThreads, (HD == 64 && !KV8) ? 2 : 1)
    attention_decode_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmks,
                            const __grid_constant__ CUtensorMap tmvs, int P) {
  using Lay = DecLayout<HD, KV8, NH>;
  constexpr int kDecSlots = Lay::kDecSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBars);  // [4][kDecSlots] TMA -> converter / consumer
  uint64_t* empty = full + 4 * kDecSlots;                           // [4][kDecSlots] consumer -> producer
  uint64_t* conv = empty + 4 * kDecSlots;                           // KV8: [4][kDecSlots] loader -> consumer
  uint64_t* ready = KV8 ? conv : full;                              // what a consumer waits for
  float* scl = reinterpret_cast<float*>(smem + Lay::kScales);       // KV8: [4][kDecSlots][64] page scales
  uint8_t* codes = smem + Lay::kCodeRing;                           // KV8: [4][2] code slots
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kAbort);
  int* first = reinterpret_cast<int*>(smem + Lay::kTable);          // [P + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 4 * kDecSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      if (KV8) mbar_init(&conv[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (tid == 128) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    if (KV8) {
      prefetch_tmap(&tmks);
      prefetch_tmap(&tmvs);
    }
  }
  pdl_trigger();
  pdl_wait();  // q, the cache pages and the piece positions come from preceding kernels
  // items per piece: splits 0 .. last position / split (at most nsplit) times Hkv
  for (int p = tid; p < P; p += blockDim.x) {
    const int n_tok = a.pm.row0[p + 1] - a.pm.row0[p];
    const int max_pos = a.pm.pos0[p] + n_tok - 1;
    first[p] = (n_tok > 0 && max_pos >= 0) ? min(a.nsplit, max_pos / a.split + 1) * a.Hkv : 0;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix sum, in order
    int run = 0;
    for (int base = 0; base < P; base += 32) {
      const int i = base + lane;
      const int v = i < P ? first[i] : 0;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      if (i < P) first[i] = run + inc - v;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) first[P] = run;
  }
  __syncthreads();
  const int n_items = first[P];
  const int lane_len = ((a.split + 3) / 4 + kKeys - 1) / kKeys * kKeys;
  const int tpl = lane_len / kKeys;  // tiles per lane
  if constexpr (KV8) {
    // warpgroup 0 consumes, warpgroups 1 and 2 load: the loaders give up their
    // registers first thing, before any of their warps can return
    if (warp < 4) reg_alloc_inc<Lay::kConsumerRegs>();
    else reg_alloc_dec<Lay::kLoaderRegs>();
  }

  if (!KV8 && warp == 4) {
    // ------------------------------------------------------------ producer
    int issued[4] = {0, 0, 0, 0};
    for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x) {
      const DecItem it = dec_item(a, first, item, P);
      const int32_t* bt = a.block_table + (int64_t)it.seq * a.max_blk;
      // tiles in (t, w) order: index i = 4 t + w
      for (int base = 0; base < 4 * tpl && !*abort_flag; base += 32) {
        const int i = base + lane;
        const int t = i >> 2, w = i & 3;
        const int lb = it.kv_begin + w * lane_len;
        const int le = min(lb + lane_len, it.kv_end);
        const int key0 = lb + t * kKeys;
        const bool need = i < 4 * tpl && key0 < le;
        int blk = -1;
        if (need) {
          blk = (key0 / kKeys < a.max_blk) ? bt[key0 / kKeys] : -1;
          if (blk < 0 || blk >= a.n_blocks) {
            report(a.status, DEV_BAD_INDEX);
            blk = -1;
          }
        }
        const unsigned need_mask = __ballot_sync(0xffffffffu, need);
        for (int j = 0; j < 32; ++j) {
          if (!((need_mask >> j) & 1u)) continue;
          const int bj = __shfl_sync(0xffffffffu, blk, j);
          const int wj = (base + j) & 3;
          int nok = 0;  // pages of this tile issued (K, then V)
          if (lane == 0) {
            for (int kv = 0; kv < 2; ++kv) {
              const int n = issued[wj] + kv;
              const int slot = wj * kDecSlots + n % kDecSlots;
              if (!dec_wait(&empty[slot], ((n / kDecSlots) & 1) ^ 1, abort_flag, a.status)) break;
              uint8_t* dst = smem + slot * Lay::kTile;
              if (bj >= 0) {
                mbar_arrive_expect_tx(&full[slot], Lay::kTile);
                const int y = (bj * a.Hkv + it.kvh) * kKeys;
#pragma unroll
                for (int bx = 0; bx < HD / 64; ++bx)
                  tma_load_2d(dst + bx * kKeys * 128, kv ? &tmv : &tmk, &full[slot], bx * 64, y);
              } else {
                mbar_arrive(&full[slot]);  // bad block (reported): the page is left as it was
              }
              ++nok;
            }
          }
          nok = __shfl_sync(0xffffffffu, nok, 0);
          issued[wj] += nok;
          if (nok < 2) break;
        }
      }
    }
    // let every copy this CTA started land before it can exit
    if (lane == 0) {
      for (int w = 0; w < 4; ++w)
        for (int i = 0; i < kDecSlots && i < issued[w]; ++i) {
          const int n = issued[w] - 1 - i;
          mbar_wait(&full[w * kDecSlots + n % kDecSlots], (n / kDecSlots) & 1);
        }
    }
    return;
  }

  if (KV8 && warp >= 4) {
    // ------------------------------------ loader of ring w, K or V pages (KV8)
    // objects in consumer w's order: items of this CTA, the ring's pages of each
    // (keys lb .. le); this warp takes the K (kv 0) or the V (kv 1) page of each.
    // With two bf16 slots per ring, consumer w's K pages always take slot 0 and
    // its V pages slot 1, so a loader owns one code slot and one bf16 slot.
    const int w = (warp - 4) & 3, kv = (warp - 4) >> 2;
    const int cs = w * kDecSlots + kv;
    int item = blockIdx.x, lb = 0, le = 0, key0 = 0, kv_end = 0, seq = 0, kvh = 0, blk_all = -1;
    bool more = false;
    auto enter = [&]() {  // the first item from `item` on with pages for this ring
      for (; item < n_items; item += gridDim.x) {
        const DecItem it = dec_item(a, first, item, P);
        lb = it.kv_begin + w * lane_len;
        le = min(lb + lane_len, it.kv_end);
        if (lb < le) {
          key0 = lb;
          kv_end = it.kv_end;
          seq = it.seq;
          kvh = it.kvh;
          // block-table entries of the first 32 pages, one per lane
          const int bi = lb / kKeys + lane;
          blk_all = (lb + lane * kKeys < le && bi < a.max_blk) ? a.block_table[(int64_t)seq * a.max_blk + bi] : -1;
          more = true;
          return;
        }
      }
      more = false;
    };
    auto advance = [&]() {
      key0 += kKeys;
      if (key0 >= le) {
        item += gridDim.x;
        enter();
      }
    };
    // the cursor's page, looked up before the slot is free (block-table entry, in
    // lane 0, and its keys at or before the item's last position); the code slot's
    // page is issued from these, so the lookups run while no codes are held
    int blk_next = -1, page_next = 0, nk_next = 0, nk_slot = 0;
    auto prepare = [&]() {  // whole warp
      nk_next = kv_end - key0;
      const int t = (key0 - lb) / kKeys;
      int blk = __shfl_sync(0xffffffffu, blk_all, t & 31);
      if (lane == 0) {
        if (t >= 32) {
          const int bi = key0 / kKeys;
          blk = bi < a.max_blk ? a.block_table[(int64_t)seq * a.max_blk + bi] : -1;
        }
        if (blk < 0 || blk >= a.n_blocks) {
          report(a.status, DEV_BAD_INDEX);
          blk = -1;
        }
        blk_next = blk;
        page_next = blk * a.Hkv + kvh;
      }
    };
    auto issue = [&]() {  // the prepared page into the code slot
      nk_slot = nk_next;
      if (lane == 0) {
        uint8_t* dst = codes + cs * Lay::kCodeSlot;
        if (blk_next >= 0) {
          mbar_arrive_expect_tx(&full[cs], Lay::kCodeSlot);
          tma_load_2d(dst, kv ? &tmv : &tmk, &full[cs], 0, page_next * kKeys);
          tma_load_2d(dst + Lay::kCodes, kv ? &tmvs : &tmks, &full[cs], 0, page_next);
        } else {
          mbar_arrive(&full[cs]);  // bad block (reported): the slot's old codes are expanded
        }
      }
    };
    int n_issued = 0, c = 0;
    enter();
    if (more) {
      prepare();
      issue();
      ++n_issued;
      advance();
      if (more) prepare();
    }
    DecCodes<HD> cd;
    uint8_t* bpage = smem + cs * Lay::kTile;
    for (; c < n_issued; ++c) {
      const int nk = nk_slot;
      if (!__all_sync(0xffffffffu, dec_wait(&full[cs], c & 1, abort_flag, a.status))) break;
      const uint8_t* src = codes + cs * Lay::kCodeSlot;
      cd.load(src, lane, 0);
      // bf16 slot: consumer w has released this loader's previous page
      if (!__all_sync(0xffffffffu, dec_wait(&empty[cs], (c & 1) ^ 1, abort_flag, a.status))) break;
      // all but the last part expanded straight from the slot; the last part and
      // the scales are read before the slot takes the next page
#pragma unroll 1
      for (int part = 0; part < DecCodes<HD>::kParts - 1; ++part) {
        cd.expand(bpage, nk, lane, part);
        cd.load(src, lane, part + 1);
      }
      const float* ssrc = reinterpret_cast<const float*>(src + Lay::kCodes);
      const float s0 = lane < nk ? ssrc[lane] : 0.f, s1 = lane + 32 < nk ? ssrc[lane + 32] : 0.f;
      fence_proxy_async();  // the reads above before the slot's next TMA copy
      __syncwarp();
      const bool issued = more;
      if (issued) {
        issue();
        ++n_issued;
      }
      cd.expand(bpage, nk, lane, DecCodes<HD>::kParts - 1);
      scl[cs * kKeys + lane] = s0;
      scl[cs * kKeys + lane + 32] = s1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv[cs]);
      if (issued) {
        advance();
        if (more) prepare();
      }
    }
    // every copy this warp started lands before it can exit
    if (lane == 0)
      for (int d = c; d < n_issued; ++d) mbar_wait(&full[cs], d & 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, tq = lane & 3;
  LaneState<HD, NH>* states = reinterpret_cast<LaneState<HD, NH>*>(smem + Lay::kStates);  // [3][32]
  int used = 0;  // objects taken from this warp's ring
  bool handed = false;
  DecItem nxt;
  if (blockIdx.x < n_items) nxt = dec_item(a, first, blockIdx.x, P);
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const DecItem it = nxt;
    // the next item's metadata loads overlap this item's pages
    if (item + (int)gridDim.x < n_items) nxt = dec_item(a, first, item + gridDim.x, P);
    int row_pos[2], row_tok[2], row_head[2];
    bool row_valid[2];
    const int tok_per_tile = 8 * NH / a.group;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // (row half 1 is empty at NH = 1)
      const int r = g + h * 8;
      const int ti = r / a.group;
      row_valid[h] = h < NH && ti < it.n_tok && ti < tok_per_tile;
      row_tok[h] = it.row0 + ti;
      row_pos[h] = it.pos_first + ti;
      row_head[h] = it.kvh * a.group + (r % a.group);
    }
    uint32_t qf[HD / 16][2 * NH];
    load_q_frags<HD, NH>(a, row_valid, row_tok, row_head, tq, qf);
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    float acc[HD / 8][2 * NH];
#pragma unroll
    for (int j = 0; j < HD / 8; ++j)
#pragma unroll
      for (int c = 0; c < 2 * NH; ++c) acc[j][c] = 0.f;

    const int lb = it.kv_begin + warp * lane_len;
    const int le = min(lb + lane_len, it.kv_end);
    for (int key0 = lb; key0 < le; key0 += kKeys) {
      float sc[8][2 * NH];
      const int n_keys = it.kv_end - key0;  // keys of this page at or before max_pos
      // K page
      int slot = warp * kDecSlots + used % kDecSlots;
      // decided for the whole warp: ldmatrix and mma.sync below are warp-collective
      bool ok = __all_sync(0xffffffffu, dec_wait(&ready[slot], (used / kDecSlots) & 1, abort_flag, a.status));
      if (ok) {
        attn_scores<HD, NH>(smem_u32(smem + slot * Lay::kTile), qf, lane, sc);
        if (KV8) {  // a score column times its key's K scale
          const float* ks = scl + slot * kKeys;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 kk = *reinterpret_cast<const float2*>(ks + j * 8 + tq * 2);
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              sc[j][h * 2] = __fmul_rn(sc[j][h * 2], kk.x);
              sc[j][h * 2 + 1] = __fmul_rn(sc[j][h * 2 + 1], kk.y);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++used;
      // V page
      slot = warp * kDecSlots + used % kDecSlots;
      ok = __all_sync(0xffffffffu, ok && dec_wait(&ready[slot], (used / kDecSlots) & 1, abort_flag, a.status));
      if (ok) {
        uint8_t* sv = smem + slot * Lay::kTile;
        if (!KV8 && n_keys < kKeys) {  // (the converter has zeroed an FP8 page's tail)
          for (int c = n_keys * (HD / 8) + lane; c < kKeys * (HD / 8); c += 32) {
            const int key = c / (HD / 8), ch = c % (HD / 8);
            *reinterpret_cast<uint4*>(sv + kv_off<HD>(key, ch)) = make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        attn_update<HD, NH>(smem_u32(sv), sc, key0, row_valid, row_pos, a.scale_log2, lane, m, l, acc,
                            KV8 ? scl + slot * kKeys : nullptr);
        if (!KV8) fence_proxy_async();  // generic writes above before the next TMA write of this slot
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++used;
    }

    // lanes meet: warps 1..3 hand over, warp 0 merges in lane order
    if (warp != 0) {
      if (handed) named_bar_sync(2, 128);  // warp 0 has read the previous item's states
      LaneState<HD, NH>* st = states + (warp - 1) * 32 + lane;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        st->m[h] = m[h];
        st->l[h] = l[h];
      }
#pragma unroll
      for (int j = 0; j < HD / 8; ++j)
#pragma unroll
        for (int c = 0; c < 2 * NH; ++c) st->acc[j][c] = acc[j][c];
      named_bar_arrive(1, 128);
      handed = true;
    } else {
      LaneState<HD, NH> Pm;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        Pm.m[h] = -INFINITY;
        Pm.l[h] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < HD / 8; ++j)
#pragma unroll
        for (int c = 0; c < 2 * NH; ++c) Pm.acc[j][c] = 0.f;
      lane_merge<HD, NH>(Pm, m, l, acc);
      named_bar_sync(1, 128);
#pragma unroll 1
      for (int w = 1; w < 4; ++w) {
        const LaneState<HD, NH>* q = states + (w - 1) * 32 + lane;
        lane_merge<HD, NH>(Pm, q->m, q->l, q->acc);
      }
      named_bar_arrive(2, 128);
      write_partial<HD, NH>(a, Pm, row_valid, row_pos, row_tok, row_head, it.kv_begin, it.s, tq);
    }
  }
  if (warp != 0 && handed) named_bar_sync(2, 128);  // pairs with warp 0's last hand-back
}

// Merge of the split partials in ascending split order (attn_merge.cuh).  One
// thread per output element (row, head, d), 128 per CTA; the split records are
// loaded in batches of kMergeBatch ahead of the in-order accumulation, so a row
// with many splits is bound by bandwidth rather than by one load latency per
// split.  q8 (optional): the output row is also quantised in 1 x 128 blocks (e4m3 codes
// q8 [T, Hq*hd], scales qs [T, Hq*hd / 128]); each CTA holds exactly one block.
// out may then be null.
// Split merge: one warp per 128 output columns of a row (one head at hd 128,
// two at hd 64), four columns per lane read as one 16-byte load per split.
// The lanes of a head load its split records (m_s, l_s) once, take M = max_s
// m_s, and hand each split's weight 2^(m_s - M) and l_s to every column by
// shuffles; each column then sums L and O over the splits in ascending order
// with the formula of merge_split_element, so its bits are unchanged.
constexpr int kMergeWarps = 4;
__global__ void __launch_bounds__(kMergeWarps * 32) attention_merge_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_ml, PieceMeta pm, int Hq, int hd, int nsplit,
    int split, __nv_bfloat16* __restrict__ out, uint8_t* __restrict__ q8, float* __restrict__ qs, int* status) {
  pdl_trigger();
  pdl_wait();
  const int p = blockIdx.y;
  const int i = blockIdx.x;
  const int row0 = pm.row0[p];
  if (i >= pm.row0[p + 1] - row0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.z * kMergeWarps + warp;  // 128-column block of the row
  const int width = Hq * hd;
  if (chunk * 128 >= width) return;
  const int G = hd / 4;                 // lanes per head (a power of two: 16 or 32)
  const int col = chunk * 128 + 4 * lane;
  const bool live = col < width;
  const int h = (live ? col : chunk * 128) / hd, d = col % hd;
  const int gl = lane % G;              // lane within its head's group
  const int64_t row = row0 + i;
  const int pos = pm.pos0[p] + i;
  const int ns = merge_split_count(pos, split, nsplit, status, chunk == 0 && lane == 0);
  const int64_t base = (row * Hq + h) * nsplit;
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + base;
  // M = max_s m_s (the max of a set does not depend on the order it is taken in)
  float M = -INFINITY;
  for (int s = gl; s < ns; s += G) M = fmaxf(M, ml[s].x);
  for (int o = G / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o, G));
  float L = 0.f, O[4] = {0.f, 0.f, 0.f, 0.f};
  const float4* po = reinterpret_cast<const float4*>(part_o + base * hd + d);
  for (int s0 = 0; s0 < ns; s0 += G) {
    // lane gl of the head holds split s0 + gl: its weight and l
    float wv = 0.f, lv = 0.f;
    if (s0 + gl < ns) {
      const float2 r = ml[s0 + gl];
      wv = merge_weight(r.x, M);
      lv = r.y;
    }
    const int nb = min(G, ns - s0);
    for (int k0 = 0; k0 < nb; k0 += 8) {
      float4 ov[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        ov[k] = (k0 + k < nb && live) ? po[(int64_t)(s0 + k0 + k) * (hd / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float w = __shfl_sync(0xffffffffu, wv, k0 + k, G);
        const float lk = __shfl_sync(0xffffffffu, lv, k0 + k, G);
        if (k0 + k < nb) {
          L = merge_term(L, lk, w);
          O[0] = merge_term(O[0], ov[k].x, w);
          O[1] = merge_term(O[1], ov[k].y, w);
          O[2] = merge_term(O[2], ov[k].z, w);
          O[3] = merge_term(O[3], ov[k].w, w);
        }
      }
    }
  }
  __nv_bfloat16 ob[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) ob[e] = f2bf(__fdiv_rn(O[e], L));
  if (out && live) {
    uint2 v;
    v.x = (uint32_t)__bfloat16_as_ushort(ob[0]) | ((uint32_t)__bfloat16_as_ushort(ob[1]) << 16);
    v.y = (uint32_t)__bfloat16_as_ushort(ob[2]) | ((uint32_t)__bfloat16_as_ushort(ob[3]) << 16);
    *reinterpret_cast<uint2*>(out + row * (int64_t)width + col) = v;
  }
  if (q8) {  // (Hq * hd is then a multiple of 128: every lane is live)
    float mx = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(bf2f(ob[e])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int ex = fp8_scale_exp(mx);
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) c |= (uint32_t)fp8_code(bf2f(ob[e]), ex) << (8 * e);
    *reinterpret_cast<uint32_t*>(q8 + row * (int64_t)width + col) = c;
    if (lane == 0) qs[row * (int64_t)(width / 128) + chunk] = ldexpf(1.f, ex);
  }
}

template <int HD, bool DECODE, bool KV8, bool FUSED = false>
constexpr int attn_smem_bytes() {
  // decode: one K+V tile per warp (+ one staging area per warp for KV8), four
  // warps or (FUSED) eight; prefill: a two-stage ring plus the running lane
  // state (KV8: one K+V tile, the running states and two staging areas)
  return DECODE ? (FUSED ? 8 : 4) * (kDecWarpTiles<KV8> * kKeys * HD * 2 + (KV8 ? Kv8Stage<HD>::kBytes : 0))
                : (KV8 ? 1 : 2) * 2 * kKeys * HD * 2 + 128 * (int)sizeof(LaneState<HD>) +
                      (KV8 ? 2 * Kv8Stage<HD>::kBytes : 0);
}

template <int HD, bool DECODE, bool KV8, bool FUSED = false, int NH = 2>
static bi_status launch_attention(const AttnArgs& args, dim3 grid, cudaStream_t st) {
  constexpr int smem = attn_smem_bytes<HD, DECODE, KV8, FUSED>();
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attention_kernel<HD, DECODE, KV8, FUSED, NH>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err != cudaSuccess)
    return fail(BI_ERR_CUDA, std::string("attention smem attribute: ") + cudaGetErrorString(attr_err));
  return launched(
      launch_pdl(attention_kernel<HD, DECODE, KV8, FUSED, NH>, grid, dim3(FUSED ? 256 : 128), smem, st, args),
      "attention_kernel");
}

// Persistent decode launch: as many CTAs as fit on the GPU at once (at most
// one per work item).  K and V are viewed as 2-D bf16 tensors [n_blocks * Hkv
// * 64 rows, hd] read in 64 x 64 boxes with 128-byte swizzle; an FP8 cache as
// code rows [n_blocks * Hkv * 64, hd bytes] read in 64-row boxes and scale rows
// [n_blocks * Hkv, 256 bytes] read one row per page, both unswizzled.
template <int HD, bool KV8, int NH>
static bi_status launch_attention_decode(const AttnArgs& args, int64_t P, cudaStream_t st) {
  constexpr int smem = DecLayout<HD, KV8, NH>::kBytes;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int per_sm = 1, launch_regs = 0;
  std::call_once(once, [] {
    attr_err =
        cudaFuncSetAttribute(attention_decode_kernel<HD, KV8, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr_err == cudaSuccess)
      attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attention_decode_kernel<HD, KV8, NH>,
                                                               DecLayout<HD, KV8, NH>::kThreads, smem);
    if (per_sm < 1) per_sm = 1;
    if (KV8 && attr_err == cudaSuccess) {
      cudaFuncAttributes fa{};
      attr_err = cudaFuncGetAttributes(&fa, attention_decode_kernel<HD, KV8, NH>);
      launch_regs = fa.numRegs;
    }
  });
  if (attr_err != cudaSuccess)
    return fail(BI_ERR_CUDA, std::string("attention decode attributes: ") + cudaGetErrorString(attr_err));
  // the warpgroups' register split must fit what the block launches with, or the
  // consumers' increase would never be granted
  if (KV8 && launch_regs < DecLayout<HD, KV8, NH>::kLaunchRegs)
    return fail(BI_ERR_CUDA, "attention decode (FP8): compiled with fewer registers than its warpgroup split needs");
  const uint64_t rows = (uint64_t)args.n_blocks * args.Hkv * kKeys;
  CUtensorMap tmk, tmv, tmks, tmvs;
  bool ok;
  if (KV8) {
    ok = encode_tmap_2d_u8(&tmk, args.k8, HD, rows, HD, HD, kKeys, false) &&
         encode_tmap_2d_u8(&tmv, args.v8, HD, rows, HD, HD, kKeys, false) &&
         encode_tmap_2d_u8(&tmks, args.ks, kKeys * 4, rows / kKeys, kKeys * 4, kKeys * 4, 1, false) &&
         encode_tmap_2d_u8(&tmvs, args.vs, kKeys * 4, rows / kKeys, kKeys * 4, kKeys * 4, 1, false);
  } else {
    ok = encode_tmap_2d_bf16(&tmk, args.k_cache, HD, rows, HD * 2, 64, kKeys, true) &&
         encode_tmap_2d_bf16(&tmv, args.v_cache, HD, rows, HD * 2, 64, kKeys, true);
    tmks = tmk;
    tmvs = tmv;
  }
  if (!ok) return fail(BI_ERR_CUDA, "attention decode: cuTensorMapEncodeTiled failed for the K/V cache");
  const int64_t grid = std::min<int64_t>(P * args.Hkv * args.nsplit, (int64_t)num_sms() * per_sm);
  return launched(launch_pdl(attention_decode_kernel<HD, KV8, NH>, dim3((unsigned)grid), dim3(DecLayout<HD, KV8, NH>::kThreads),
                             smem, st, args, tmk,
                             tmv, tmks, tmvs, (int)P),
                  "attention_decode_kernel");
}

// Tensor-memory prefill launch: K and V viewed as the persistent decode kernel
// views them (2-D bf16 [n_blocks * Hkv * 64, hd], 64 x 64 boxes, 128-byte swizzle).
template <int HD>
static bi_status launch_attention_tc(const AttnArgs& args, dim3 grid, cudaStream_t st) {
  constexpr int smem = TcAttnLayout<HD>::kBytes;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attention_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err != cudaSuccess)
    return fail(BI_ERR_CUDA, std::string("attention prefill attributes: ") + cudaGetErrorString(attr_err));
  const uint64_t rows = (uint64_t)args.n_blocks * args.Hkv * kKeys;
  CUtensorMap tmk, tmv;
  if (!encode_tmap_2d_bf16(&tmk, args.k_cache, HD, rows, HD * 2, 64, kKeys, true) ||
      !encode_tmap_2d_bf16(&tmv, args.v_cache, HD, rows, HD * 2, 64, kKeys, true))
    return fail(BI_ERR_CUDA, "attention prefill: cuTensorMapEncodeTiled failed for the K/V cache");
  return launched(launch_pdl(attention_tc_kernel<HD>, grid, dim3(TcAttnLayout<HD>::kThreads), smem, st, args, tmk,
                             tmv),
                  "attention_tc_kernel");
}

// Positions per split: the fixed kv_split, or (BI_FAST) a size chosen from the
// batch so that the decode grid fills the GPU (flash-decoding heuristic).
static int choose_split(int mode, int kv_split, int64_t P, int64_t max_q_len, int Hkv, int group, int64_t max_ctx) {
  if (mode != BI_FAST || max_q_len * group > kRows) return kv_split;
  const int64_t qtiles = 1;
  const int64_t ctas = P * Hkv * qtiles;
  const int64_t want = std::max<int64_t>(1, cdiv(2 * (int64_t)num_sms(), std::max<int64_t>(ctas, 1)));
  int64_t sz = cdiv(std::max<int64_t>(max_ctx, 1), want);
  sz = std::max<int64_t>(64, cdiv(sz, 64) * 64);
  return (int)std::min<int64_t>(sz, kv_split);
}

static int64_t n_splits(int64_t max_ctx, int split) { return std::max<int64_t>(1, cdiv(max_ctx, split)); }

}  // namespace bi

extern "C" {

bi_status bi_rope_table(float* rope_table, int64_t max_pos, int hd, double theta, void* stream) {
  using namespace bi;
  BI_REQUIRE(rope_table, "null table");
  BI_REQUIRE(max_pos > 0 && hd > 0 && hd % 2 == 0, "bad shape");
  const int64_t total = max_pos * (hd / 2);
  const int blocks = (int)std::min<int64_t>(cdiv(total, 256), 4096);
  return launched(launch_pdl(rope_table_kernel, dim3(blocks), dim3(256), 0, as_stream(stream), rope_table, max_pos, hd,
                             theta),
                  "bi_rope_table");
}

bi_status bi_rope_kv_write(const void* qkv, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                           const float* rope_table, int64_t max_pos, const int32_t* block_table,
                           int64_t max_blocks_per_seq, int64_t n_blocks, void* q_out, void* k_cache, void* v_cache,
                           void* stream) {
  using namespace bi;
  BI_REQUIRE(T >= 0 && P >= 0, "bad shape");
  if (T == 0 || P == 0) return BI_OK;
  BI_REQUIRE(qkv && piece_seq && piece_row0 && piece_pos0 && rope_table && block_table && q_out && k_cache && v_cache,
             "null pointer");
  BI_REQUIRE(Hq > 0 && Hkv > 0 && Hq % Hkv == 0 && hd > 0 && hd % 2 == 0, "bad heads");
  BI_REQUIRE(max_q_len > 0 && max_q_len <= 65535 && P <= 65535, "bad max_q_len / P");
  BI_REQUIRE(max_blocks_per_seq > 0 && n_blocks > 0, "bad cache shape");
  PieceMeta pm{piece_seq, piece_row0, piece_pos0};
  dim3 grid((unsigned)max_q_len, (unsigned)P);
  return launched(launch_pdl(rope_kv_write_kernel, grid, dim3(128), 0, as_stream(stream),
                             static_cast<const __nv_bfloat16*>(qkv), pm, Hq, Hkv, hd, rope_table, max_pos, block_table,
                             max_blocks_per_seq, n_blocks, static_cast<__nv_bfloat16*>(q_out),
                             static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache),
                             device_status_ptr()),
                  "bi_rope_kv_write");
}

size_t bi_attention_workspace_size(int64_t max_T, int Hq, int hd, int64_t max_ctx, int kv_split) {
  if (max_T <= 0 || Hq <= 0 || hd <= 0 || max_ctx <= 0 || kv_split < 64) return 0;
  // BI_FAST may shrink the split down to 64 positions for decode-sized calls;
  // size for the invariant split and for 64 and take the larger.
  const int64_t ns = std::max(bi::n_splits(max_ctx, kv_split), std::min<int64_t>(bi::n_splits(max_ctx, 64),
                                                                                   bi::n_splits(max_ctx, kv_split) * 8));
  const size_t per = (size_t)max_T * Hq * ns;
  return per * hd * sizeof(float) + per * 2 * sizeof(float) + 256;
}

}  // extern "C"

namespace bi {

// Shared body of bi_attention (bf16 cache) and bi_attention_fp8 (k8 != null).
static bi_status attention_impl(const void* q, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                                const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                                const void* k_cache, const void* v_cache, const void* k8, const void* v8,
                                const float* ks, const float* vs, const int32_t* block_table,
                                int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx, int kv_split,
                                float scale, void* workspace, size_t ws_bytes, void* out, void* out_q,
                                float* out_scale, int mode, void* stream) {
  BI_REQUIRE(T >= 0 && P >= 0, "bad shape");
  if (T == 0 || P == 0) return BI_OK;
  const bool kv8 = k8 != nullptr;
  BI_REQUIRE(q && piece_seq && piece_row0 && piece_pos0 && block_table && workspace, "null pointer");
  BI_REQUIRE(kv8 ? (v8 && ks && vs) : (k_cache && v_cache), "null cache pointer");
  BI_REQUIRE(out || out_q, "null output");
  BI_REQUIRE(!out_q == !out_scale, "out_q and out_scale go together");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  BI_REQUIRE_SHAPE(hd == 64 || hd == 128, "head_dim must be 64 or 128");
  BI_REQUIRE(Hq > 0 && Hkv > 0 && Hq % Hkv == 0, "Hq must be a multiple of Hkv");
  BI_REQUIRE_SHAPE(!out_q || (Hq * hd) % 128 == 0, "quantised output needs Hq*hd to be a multiple of 128");
  const int group = Hq / Hkv;
  BI_REQUIRE_SHAPE(kRows % group == 0, "64 must be a multiple of Hq/Hkv");
  BI_REQUIRE(kv_split >= 64 && kv_split % 64 == 0, "kv_split must be a positive multiple of 64");
  BI_REQUIRE(max_ctx > 0 && max_q_len > 0, "bad max_ctx / max_q_len");
  BI_REQUIRE(max_blocks_per_seq > 0 && n_blocks > 0 && n_blocks * Hkv * 64 < (int64_t(1) << 32),
             "bad cache shape (max_blocks_per_seq, n_blocks)");
  BI_REQUIRE(aligned16(q) && aligned16(workspace) && (!out || aligned16(out)), "pointers must be 16-byte aligned");
  BI_REQUIRE(kv8 ? (aligned16(k8) && aligned16(v8) && aligned16(ks) && aligned16(vs))
                 : (aligned16(k_cache) && aligned16(v_cache)),
             "cache pointers must be 16-byte aligned");
  const int split = choose_split(mode, kv_split, P, max_q_len, Hkv, group, max_ctx);
  const int64_t ns = n_splits(max_ctx, split);
  const size_t per = (size_t)T * Hq * ns;
  const size_t need = per * hd * sizeof(float) + per * 2 * sizeof(float);
  BI_REQUIRE(ws_bytes >= need, "attention workspace too small (bi_attention_workspace_size)");
  float* part_o = static_cast<float*>(workspace);
  float* part_ml = part_o + per * hd;
  const int64_t qtiles = cdiv(max_q_len * group, kRows);
  BI_REQUIRE(qtiles <= 0x7fffffff && P <= 65535 && Hkv * ns <= 65535, "grid too large");
  AttnArgs args;
  args.q = static_cast<const __nv_bfloat16*>(q);
  args.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  args.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  args.k8 = static_cast<const uint8_t*>(k8);
  args.v8 = static_cast<const uint8_t*>(v8);
  args.ks = ks;
  args.vs = vs;
  args.block_table = block_table;
  args.part_o = part_o;
  args.part_ml = part_ml;
  args.status = device_status_ptr();
  args.pm = PieceMeta{piece_seq, piece_row0, piece_pos0};
  args.max_blk = max_blocks_per_seq;
  args.n_blocks = n_blocks;
  args.Hq = Hq;
  args.Hkv = Hkv;
  args.group = group;
  args.nsplit = (int)ns;
  args.split = split;
  args.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = as_stream(stream);
  // Four schedules with the same per-row arithmetic (so the same bits):
  // query tiles of at most 16 rows (decode steps) take the lane-parallel
  // schedule, persistent with TMA page streaming once contexts span more than
  // kDecPersistentSplits splits (and the call has at most kDecMaxPieces
  // sequences), one CTA per (sequence, kv head, split) otherwise; bigger query
  // tiles take the tensor-memory prefill schedule (bf16 caches) or the
  // mma.sync row-parallel one (FP8 caches).
  const bool decode = max_q_len * group <= 16;
  // decode tiles of at most 8 query rows (GQA group x tokens) keep one row half
  // of the 16-row MMA tiles: the same bits, half the softmax and state work
  const bool half = max_q_len * group <= 8;
  args.out = static_cast<__nv_bfloat16*>(out);
  if (decode && ns <= 2 && hd == 64 && out && !out_q) {
    // short contexts: both splits in one CTA, merged there (no partials, no merge kernel)
    dim3 grid((unsigned)cdiv(max_q_len * group, 16), (unsigned)P, (unsigned)Hkv);
    if (half)
      return kv8 ? launch_attention<64, true, true, true, 1>(args, grid, st)
                 : launch_attention<64, true, false, true, 1>(args, grid, st);
    return kv8 ? launch_attention<64, true, true, true>(args, grid, st)
               : launch_attention<64, true, false, true>(args, grid, st);
  }
  if (decode && ns > kDecPersistentSplits && P <= kDecMaxPieces) {
    BI_REQUIRE(P * Hkv * ns < (int64_t(1) << 31), "too many attention work items");
    // tiles of at most 8 query rows (GQA group x tokens) keep one row half
    const bool half = max_q_len * group <= 8;
    if (kv8 && half)
      BI_TRY(hd == 64 ? launch_attention_decode<64, true, 1>(args, P, st)
                      : launch_attention_decode<128, true, 1>(args, P, st));
    else if (kv8)
      BI_TRY(hd == 64 ? launch_attention_decode<64, true, 2>(args, P, st)
                      : launch_attention_decode<128, true, 2>(args, P, st));
    else if (half)
      BI_TRY(hd == 64 ? launch_attention_decode<64, false, 1>(args, P, st)
                      : launch_attention_decode<128, false, 1>(args, P, st));
    else
      BI_TRY(hd == 64 ? launch_attention_decode<64, false, 2>(args, P, st)
                      : launch_attention_decode<128, false, 2>(args, P, st));
  } else if (decode) {
    dim3 grid((unsigned)cdiv(max_q_len * group, 16), (unsigned)P, (unsigned)(Hkv * ns));
    if (kv8 && half)
      BI_TRY(hd == 64 ? launch_attention<64, true, true, false, 1>(args, grid, st)
                      : launch_attention<128, true, true, false, 1>(args, grid, st));
    else if (kv8)
      BI_TRY(hd == 64 ? launch_attention<64, true, true>(args, grid, st)
                      : launch_attention<128, true, true>(args, grid, st));
    else if (half)
      BI_TRY(hd == 64 ? launch_attention<64, true, false, false, 1>(args, grid, st)
                      : launch_attention<128, true, false, false, 1>(args, grid, st));
    else
      BI_TRY(hd == 64 ? launch_attention<64, true, false>(args, grid, st)
                      : launch_attention<128, true, false>(args, grid, st));
  } else if (!kv8 && n_blocks * Hkv * kKeys < (int64_t(1) << 31)) {
    // bf16 cache: 128-row query tiles on the tensor cores (TMA page coordinates are 32-bit)
    dim3 grid((unsigned)cdiv(max_q_len * group, 128), (unsigned)P, (unsigned)(Hkv * cdiv(ns, kTcSplitsPerCta)));
    BI_TRY(hd == 64 ? launch_attention_tc<64>(args, grid, st) : launch_attention_tc<128>(args, grid, st));
  } else {
    dim3 grid((unsigned)qtiles, (unsigned)P, (unsigned)(Hkv * ns));
    if (kv8)
      BI_TRY(hd == 64 ? launch_attention<64, false, true>(args, grid, st)
                      : launch_attention<128, false, true>(args, grid, st));
    else
      BI_TRY(hd == 64 ? launch_attention<64, false, false>(args, grid, st)
                      : launch_attention<128, false, false>(args, grid, st));
  }
  dim3 mgrid((unsigned)max_q_len, (unsigned)P, (unsigned)cdiv(cdiv(Hq * hd, 128), kMergeWarps));
  return launched(launch_pdl(attention_merge_kernel, mgrid, dim3(kMergeWarps * 32), 0, st, (const float*)part_o,
                             (const float*)part_ml, args.pm, Hq, hd, (int)ns, split, static_cast<__nv_bfloat16*>(out),
                             static_cast<uint8_t*>(out_q), out_scale, args.status),
                  "attention_merge_kernel");
}

}  // namespace bi

extern "C" {

bi_status bi_attention(const void* q, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                       const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx, int kv_split, float scale,
                       void* workspace, size_t ws_bytes, void* out, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(out || T == 0 || P == 0, "null pointer");
  BI_REQUIRE((k_cache && v_cache) || T == 0 || P == 0, "null pointer");
  return attention_impl(q, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, k_cache, v_cache,
                        nullptr, nullptr, nullptr, nullptr, block_table, max_blocks_per_seq, n_blocks, max_ctx,
                        kv_split, scale, workspace, ws_bytes, out, nullptr, nullptr, mode, stream);
}

bi_status bi_attention_fp8(const void* q, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                           const void* k_cache8, const void* v_cache8, const float* k_scale, const float* v_scale,
                           const int32_t* block_table, int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx,
                           int kv_split, float scale, void* workspace, size_t ws_bytes, void* out, void* out_q,
                           float* out_scale, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE((k_cache8 && v_cache8 && k_scale && v_scale) || T == 0 || P == 0, "null pointer");
  return attention_impl(q, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, nullptr, nullptr,
                        k_cache8, v_cache8, k_scale, v_scale, block_table, max_blocks_per_seq, n_blocks, max_ctx,
                        kv_split, scale, workspace, ws_bytes, out, out_q, out_scale, mode, stream);
}

}  // extern "C"

// ------------------------------------------------- attention, library scratch
// For callers that cannot hand the library a workspace: the split partials go
// to a fixed array that lives in this module on every device that loads it.
namespace bi {

constexpr size_t kAttnStaticScratchBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_attn_static_scratch[kAttnStaticScratchBytes];

// Device address of the array in the current context: looked up on a device's
// first call and again whenever the context has changed since (a reset device,
// or a context the caller made), never reused across contexts.
static bi_status attn_static_scratch_addr(void** out) {
  static ModuleAddressCache cache;
  if (!module_symbol_address(&g_attn_static_scratch, out, &cache))
    return fail(BI_ERR_CUDA, "bi_attention_static_scratch: cudaGetSymbolAddress of the scratch array failed");
  return BI_OK;
}

// Bytes of split partials a call needs, T * Hq * ns * (hd + 2) * 4, or false
// when that product does not fit in 64 bits (so huge sizes cannot wrap around
// to a small one).
static bool attn_partials_bytes(int64_t T, int Hq, int64_t ns, int hd, uint64_t* need) {
  uint64_t b = (uint64_t)(hd + 2) * sizeof(float);
  const uint64_t factors[3] = {(uint64_t)Hq, (uint64_t)ns, (uint64_t)T};
  for (uint64_t f : factors)
    if (__builtin_mul_overflow(b, f, &b)) return false;
  *need = b;
  return true;
}

}  // namespace bi

extern "C" bi_status bi_attention_static_scratch(const void* q, int64_t T, const int32_t* piece_seq,
                                                 const int32_t* piece_row0, const int32_t* piece_pos0, int64_t P,
                                                 int64_t max_q_len, int Hq, int Hkv, int hd, const void* k_cache,
                                                 const void* v_cache, const int32_t* block_table,
                                                 int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx,
                                                 int kv_split, float scale, void* out, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(T >= 0 && P >= 0, "bad shape");
  if (T == 0 || P == 0) return BI_OK;
  BI_REQUIRE(Hq > 0 && Hkv > 0 && Hq % Hkv == 0, "Hq must be a multiple of Hkv");
  BI_REQUIRE(hd > 0 && kv_split >= 64 && kv_split % 64 == 0 && max_ctx > 0 && max_q_len > 0,
             "bad head_dim / kv_split / max_ctx / max_q_len");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  // the partials this call needs, computed the way bi_attention sizes them
  const int split = choose_split(mode, kv_split, P, max_q_len, Hkv, Hq / Hkv, max_ctx);
  const int64_t ns = n_splits(max_ctx, split);
  uint64_t need = 0;
  const bool exact = attn_partials_bytes(T, Hq, ns, hd, &need);
  if (!exact || need > kAttnStaticScratchBytes)
    return fail(BI_ERR_INVALID_ARG,
                "bi_attention_static_scratch: this call needs " +
                    (exact ? std::to_string(need) : std::string("more than 2^64")) +
                    " bytes of split partials (T " + std::to_string(T) + " x Hq " + std::to_string(Hq) + " x splits " +
                    std::to_string(ns) + " x (hd + 2) x 4) but the static scratch array holds " +
                    std::to_string(kAttnStaticScratchBytes) + " bytes; use bi_attention with a caller workspace");
  void* scratch = nullptr;
  BI_TRY(attn_static_scratch_addr(&scratch));
  return bi_attention(q, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, k_cache, v_cache,
                      block_table, max_blocks_per_seq, n_blocks, max_ctx, kv_split, scale, scratch,
                      kAttnStaticScratchBytes, out, mode, stream);
}
