// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 "Dense GEMM: keep
// FP8, one accumulation order for every M": the inference engine's M-dependent
// kernel switch is removed so a request's row never changes with the batch.
// Here the invariant path runs ONE kernel for every M: a 128 x BN x 64 CTA
// tile (BN fixed by the weight's (N, K) and the epilogue), K consumed in
// ascending 16-wide tcgen05.mma steps into a single fp32 TMEM accumulator, no
// split-K.  A row's bits therefore depend only on that row of A and on W.
//
// §4.4 "Expert GEMM: two layouts, same row result": the grouped variant maps
// each 128-row tile to one expert; row results do not depend on the layout.
//
// CTA = 4 warps.  Warp 0 lane 0 issues TMA loads into a STAGES-deep ring
// (full/empty mbarriers), warp 1 lane 0 issues tcgen05.mma and commits each
// stage back to its empty barrier, then all four warps drain TMEM (warp w owns
// TMEM lanes 32w..32w+31 = tile rows) through the epilogue.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "norm.cuh"

namespace bi {

enum EpiKind : int {
  EPI_BF16 = 0,
  EPI_F32 = 1,
  EPI_SWIGLU = 2,
  EPI_PARTIAL = 3,
  EPI_PARTIAL_SWIGLU = 4,
  EPI_LSE = 5,
  EPI_ROPE = 6
};

// Operands of the QKV epilogue that applies RoPE and writes K/V into the paged cache.
struct RopeKvArgs {
  const int32_t* row_seq;   // [M] sequence of each row
  const int32_t* row_pos;   // [M] absolute position of each row
  const float* table;       // [max_pos, hd]: cos | sin
  const int32_t* block_table;
  __nv_bfloat16* q_out;     // [M, Hq, hd]
  __nv_bfloat16* k_cache;   // [n_blocks, Hkv, 64, hd] (one layer)
  __nv_bfloat16* v_cache;
  int64_t max_pos, max_blk, n_blocks;
  int Hq, Hkv, hd;
};

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;

// TMA ring depth per tile width (about 190-220 KB of stages): deep enough that
// a decode-size K range of a small weight is in flight at once, all of it
// requested before the dependency wait.  It never changes results.
template <int BN>
struct GemmSmem {
  static constexpr int kStages = BN == 16 ? 12 : (BN == 32 ? 11 : (BN == 64 ? 9 : (BN == 128 ? 5 : 4)));
  static constexpr int kBTileBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes;
  static constexpr int kBytes = 1024 + kStages * kStageBytes + 256;
};

// The fused log-softmax at 64 and 128 columns keeps two staging buffers of a
// 16-row tile ([16][BN + 4] fp32 each) for tiles of at most 16 rows.
template <int BN, int EPI>
struct LseStage {
  static constexpr bool kOn = EPI == 5 && (BN == 64 || BN == 128);  // EPI_LSE
  static constexpr int kFloats = 16 * (BN + 4);
  static constexpr int kBytes = kOn ? 2 * kFloats * 4 : 0;
};
template <int BN, int EPI>
constexpr int gemm_tc_smem() {
  return GemmSmem<BN>::kBytes + LseStage<BN, EPI>::kBytes;
}

struct GemmArgs {
  void* C;
  float* partial;           // split-K partials [splits, M, ldp]
  const int32_t* tile_expert;
  int* status;
  int M, K, ldc;            // ldc = output columns
  int n_out;                // valid output columns (N, or F for SwiGLU)
  int w_rows_per_expert;    // rows of W per expert (grouped); 0 for dense
  int up_offset;            // SwiGLU: row offset of the up half inside one expert's W
  int k_blocks_per_split;
  int ldp;                  // partial row length
  const int32_t* ids;       // EPI_LSE: target id of each row (NULL = greedy)
  TileLse* lse;             // EPI_LSE: [M, n_tiles] tile partials
  int n_tiles;              // EPI_LSE: vocab tiles per row
  int m_tiles, n_tiles_grid, splits;  // tile space walked by the persistent CTAs
  int a_box_rows;                     // rows of A one TMA copy brings in (128, or M rounded up to 8 when M < 128)
  int group_m;                        // M-tiles per rasterisation group
  RopeKvArgs rope;                    // EPI_ROPE only
  // decode-size schedule with the RMSNorm folded in: A = norm(nx (+ nres_in)) * ngamma
  const __nv_bfloat16* nx;
  const __nv_bfloat16* nres_in;
  __nv_bfloat16* nres_out;
  const __nv_bfloat16* ngamma;
  float neps;
};

// Online (max, sum-exp, argmax) over 4 consecutive logits, in column order.
__device__ __forceinline__ void tile_lse_step4(float& m, float& s, float& best, int& idx, const uint32_t* r,
                                               int col) {
  const float x0 = __uint_as_float(r[0]), x1 = __uint_as_float(r[1]);
  const float x2 = __uint_as_float(r[2]), x3 = __uint_as_float(r[3]);
  const float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  if (mx > m) {
    s = (m == -INFINITY) ? 0.f : __fmul_rn(s, expf(__fsub_rn(m, mx)));
    m = mx;
  }
  s = __fadd_rn(s, expf(__fsub_rn(x0, m)));
  s = __fadd_rn(s, expf(__fsub_rn(x1, m)));
  s = __fadd_rn(s, expf(__fsub_rn(x2, m)));
  s = __fadd_rn(s, expf(__fsub_rn(x3, m)));
  if (x0 > best) { best = x0; idx = col; }
  if (x1 > best) { best = x1; idx = col + 1; }
  if (x2 > best) { best = x2; idx = col + 2; }
  if (x3 > best) { best = x3; idx = col + 3; }
}

// The same (max, sum-exp, argmax) record of one tile row, with the row's BN
// logits staged in shared memory and shared by 8 threads (16-row tiles: 128
// threads).  Each thread takes BN/8 consecutive columns.  The running max after
// each 4-column group is a prefix max (order-free), so every exponential and
// every rescale factor of the column-order recurrence is computed in parallel;
// only the fp32 fold of s is sequential, carried from chunk to chunk by
// shuffles, with the recurrence's operations in its order (s reset to 0 when the
// running max was -inf, s * expf(m - mx) when a group raises it, then its four
// terms added in column order).  The argmax of a later chunk replaces that of an
// earlier one only when strictly greater, as the sequential scan does.  So the
// record equals tile_lse_step4's over the row, bit for bit.
constexpr int kLseSmallRows = 16;
template <int BN>
__device__ __forceinline__ void lse_small_tile_row(const GemmArgs& args, const float* stg, int m_tile, int n_tile,
                                                   int u, bool do_store) {
  constexpr int CPC = BN / 8;  // columns per chunk
  constexpr int G = CPC / 4;   // 4-column groups per chunk
  const int r = u >> 3, k = u & 7;
  const int row = m_tile * kBM + r;
  const bool row_ok = row < args.M;
  const int n0 = n_tile * BN, c0 = n0 + k * CPC;
  float x[CPC];
#pragma unroll
  for (int i = 0; i < CPC; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(stg + r * (BN + 4) + k * CPC + i);
    x[i] = v.x;
    x[i + 1] = v.y;
    x[i + 2] = v.z;
    x[i + 3] = v.w;
  }
  bool gv[G];
  float gm[G];
  float cm = -INFINITY;  // this chunk's max over its groups
#pragma unroll
  for (int g = 0; g < G; ++g) {
    gv[g] = c0 + 4 * g < args.n_out;
    gm[g] = fmaxf(fmaxf(x[4 * g], x[4 * g + 1]), fmaxf(x[4 * g + 2], x[4 * g + 3]));
    if (gv[g]) cm = fmaxf(cm, gm[g]);
  }
  // the running max entering this chunk: max over the row's earlier chunks
  float incl = cm;
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) {
    const float v = __shfl_up_sync(0xffffffffu, incl, d, 8);
    if (k >= d) incl = fmaxf(incl, v);
  }
  float m = __shfl_up_sync(0xffffffffu, incl, 1, 8);
  if (k == 0) m = -INFINITY;
  // per group: does it raise the max, from -inf, the rescale factor, the terms
  bool up[G], from_inf[G];
  float rs[G], e[CPC];
  float best = -INFINITY;
  int idx = 0x7fffffff;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    up[g] = false;
    from_inf[g] = false;
    rs[g] = 1.f;
    if (!gv[g]) continue;
    if (gm[g] > m) {
      up[g] = true;
      from_inf[g] = m == -INFINITY;
      if (!from_inf[g]) rs[g] = expf(__fsub_rn(m, gm[g]));
      m = gm[g];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[4 * g + i] = expf(__fsub_rn(x[4 * g + i], m));
      if (x[4 * g + i] > best) {
        best = x[4 * g + i];
        idx = c0 + 4 * g + i;
      }
    }
  }
  // the fold of s, chunk after chunk
  float s_out = 0.f;
#pragma unroll 1
  for (int step = 0; step < 8; ++step) {
    const float s_in = __shfl_up_sync(0xffffffffu, s_out, 1, 8);
    if (k == step) {
      float s = k == 0 ? 0.f : s_in;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (!gv[g]) continue;
        if (up[g]) s = from_inf[g] ? 0.f : __fmul_rn(s, rs[g]);
#pragma unroll
        for (int i = 0; i < 4; ++i) s = __fadd_rn(s, e[4 * g + i]);
      }
      s_out = s;
    }
  }
  // argmax over the chunks in order: a later chunk wins only when strictly greater
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) {
    const float vb = __shfl_up_sync(0xffffffffu, best, d, 8);
    const int vi = __shfl_up_sync(0xffffffffu, idx, d, 8);
    if (k >= d && !(best > vb)) {
      best = vb;
      idx = vi;
    }
  }
  // the target's logit, from the chunk that holds it
  const int tgt = (row_ok && args.ids) ? args.ids[row] : -1;
  const int off = tgt - n0;
  float xt = __int_as_float(0x7fc00000);
  if (off >= 0 && off < BN && off / CPC == k) {
#pragma unroll
    for (int i = 0; i < CPC; ++i)
      if (i == off - k * CPC) xt = x[i];
  }
  const int owner = (off >= 0 && off < BN) ? off / CPC : 7;
  const float xt_row = __shfl_sync(0xffffffffu, xt, (threadIdx.x & 24) + owner);
  if (k == 7 && do_store && row_ok) {
    TileLse t;
    t.m = incl;
    t.s = s_out;
    t.best = best;
    t.xt = xt_row;
    t.idx = idx;
    t.pad[0] = t.pad[1] = t.pad[2] = 0;
    args.lse[(size_t)row * args.n_tiles + n_tile] = t;
  }
}

__device__ __forceinline__ float silu_f(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }

// Per-element epilogue arithmetic, shared by every GEMM schedule.
// SwiGLU: silu(bf16(gate)) * bf16(up) in fp32, from the fp32 accumulators.
__device__ __forceinline__ float swiglu_elem(float g, float u) {
  return __fmul_rn(silu_f(bf2f(f2bf(g))), bf2f(f2bf(u)));
}
// RoPE rotate-half of the pair (x1, x2) = bf16 of the accumulators (j, j + hd/2).
__device__ __forceinline__ void rope_pair(float x1, float x2, float c, float s, float& o1, float& o2) {
  const float v1 = bf2f(f2bf(x1)), v2 = bf2f(f2bf(x2));
  o1 = __fsub_rn(__fmul_rn(v1, c), __fmul_rn(v2, s));
  o2 = __fadd_rn(__fmul_rn(v2, c), __fmul_rn(v1, s));
}

// CW consecutive accumulator columns of this warp's 32 TMEM lanes (CW = 16 or 32).
template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32) tmem_ld_32x32b_x32(taddr, r);
  else tmem_ld_32x32b_x16(taddr, r);
}

// Epilogue of one 128 x BN accumulator tile: this warp drains TMEM lanes
// 32q..32q+31 (tile rows) from column base t_row and writes its rows.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& args, uint32_t t_row, int row, bool row_ok,
                                              bool do_store, int n_tile, int split) {
  if constexpr (EPI == EPI_SWIGLU || EPI == EPI_PARTIAL_SWIGLU) {
    const int j0 = n_tile * (BN / 2);
    constexpr int CW = BN / 2 < 32 ? BN / 2 : 32;
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += CW) {
      uint32_t g[CW], u[CW];
      tmem_ld_cols<CW>(t_row + c, g);
      tmem_ld_cols<CW>(t_row + BN / 2 + c, u);
      tmem_ld_wait();
      if (!(do_store && row_ok)) continue;
      if (EPI == EPI_SWIGLU) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.C) + (size_t)row * args.ldc;
#pragma unroll
        for (int q = 0; q < CW / 8; ++q) {
          const int col = j0 + c + q * 8;
          if (col >= args.n_out) break;
          uint4 v;
          uint32_t* pv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float a2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = q * 8 + e * 2 + h;
              a2[h] = swiglu_elem(__uint_as_float(g[i]), __uint_as_float(u[i]));
            }
            pv[e] = pack_bf16x2(a2[0], a2[1]);
          }
          *reinterpret_cast<uint4*>(out + col) = v;
        }
      } else {
        float* pg = args.partial + ((size_t)split * args.M + row) * args.ldp;
        float* pu = pg + args.n_out;
#pragma unroll
        for (int q = 0; q < CW / 4; ++q) {
          const int col = j0 + c + q * 4;
          if (col >= args.n_out) break;
          *reinterpret_cast<float4*>(pg + col) =
              make_float4(__uint_as_float(g[q * 4]), __uint_as_float(g[q * 4 + 1]), __uint_as_float(g[q * 4 + 2]),
                          __uint_as_float(g[q * 4 + 3]));
          *reinterpret_cast<float4*>(pu + col) =
              make_float4(__uint_as_float(u[q * 4]), __uint_as_float(u[q * 4 + 1]), __uint_as_float(u[q * 4 + 2]),
                          __uint_as_float(u[q * 4 + 3]));
        }
      }
    }
  } else if constexpr (EPI == EPI_ROPE) {
    // q/k heads: rotate-half pairs (j, j + hd/2) of bf16(acc) in fp32, rounded
    // to bf16; q to q_out, k and v into the paged cache at the row's position.
    const RopeKvArgs& ra = args.rope;
    const int hd = ra.hd, half = hd / 2;
    const int n0 = n_tile * BN;
    bool ok = do_store && row_ok;
    int64_t pos = 0, blk = -1;
    if (ok) {
      const int seq = ra.row_seq[row];
      pos = ra.row_pos[row];
      if (pos < 0 || pos >= ra.max_pos) {
        report(args.status, DEV_BAD_INDEX);
        ok = false;
      } else {
        const int32_t b = (pos / 64 < ra.max_blk) ? ra.block_table[(int64_t)seq * ra.max_blk + pos / 64] : -1;
        if (b >= 0 && b < ra.n_blocks) blk = b;
        else report(args.status, DEV_BAD_INDEX);
      }
    }
    const int slot = (int)(pos % 64);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int n = n0 + c;
      if (n >= args.n_out) break;  // a last tile past the final head
      const int h = n / hd, j0 = n % hd;
      if (h < ra.Hq + ra.Hkv) {
        if (j0 >= half) continue;  // done together with its partner chunk
        uint32_t x1[32], x2[32];
        tmem_ld_32x32b_x32(t_row + c, x1);
        tmem_ld_32x32b_x32(t_row + c + half, x2);
        tmem_ld_wait();
        if (!ok) continue;
        __nv_bfloat16* dst;
        if (h < ra.Hq) dst = ra.q_out + ((int64_t)row * ra.Hq + h) * hd;
        else if (blk >= 0) dst = ra.k_cache + (((int64_t)blk * ra.Hkv + (h - ra.Hq)) * 64 + slot) * hd;
        else continue;
        // the row's cos and sin runs as 16-byte loads (a thread is a row: one line per lane)
        const float4* c4 = reinterpret_cast<const float4*>(ra.table + pos * hd + j0);
        const float4* s4 = reinterpret_cast<const float4*>(ra.table + pos * hd + half + j0);
        uint32_t o1[16], o2[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 cv = c4[i / 4], sv = s4[i / 4];
          const float cc[4] = {cv.x, cv.y, cv.z, cv.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
          float a1[4], a2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            rope_pair(__uint_as_float(x1[i + e]), __uint_as_float(x2[i + e]), cc[e], ss[e], a1[e], a2[e]);
          o1[i / 2] = pack_bf16x2(a1[0], a1[1]);
          o1[i / 2 + 1] = pack_bf16x2(a1[2], a1[3]);
          o2[i / 2] = pack_bf16x2(a2[0], a2[1]);
          o2[i / 2 + 1] = pack_bf16x2(a2[2], a2[3]);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          reinterpret_cast<uint4*>(dst + j0)[v] = make_uint4(o1[4 * v], o1[4 * v + 1], o1[4 * v + 2], o1[4 * v + 3]);
          reinterpret_cast<uint4*>(dst + j0 + half)[v] =
              make_uint4(o2[4 * v], o2[4 * v + 1], o2[4 * v + 2], o2[4 * v + 3]);
        }
      } else {
        uint32_t x[32];
        tmem_ld_32x32b_x32(t_row + c, x);
        tmem_ld_wait();
        if (!ok || blk < 0) continue;
        __nv_bfloat16* dst =
            ra.v_cache + (((int64_t)blk * ra.Hkv + (h - ra.Hq - ra.Hkv)) * 64 + slot) * hd + j0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(x[8 * v + 0]), __uint_as_float(x[8 * v + 1]));
          w.y = pack_bf16x2(__uint_as_float(x[8 * v + 2]), __uint_as_float(x[8 * v + 3]));
          w.z = pack_bf16x2(__uint_as_float(x[8 * v + 4]), __uint_as_float(x[8 * v + 5]));
          w.w = pack_bf16x2(__uint_as_float(x[8 * v + 6]), __uint_as_float(x[8 * v + 7]));
          reinterpret_cast<uint4*>(dst)[v] = w;
        }
      }
    }
  } else if constexpr (EPI == EPI_LSE) {
    static_assert(EPI != EPI_LSE || BN >= 64, "the fused log-softmax keeps 64+ wide vocab tiles");
    // fp32 logits of this row's BN columns, visited in column order
    const int n0 = n_tile * BN;
    const int tgt = (row_ok && args.ids) ? args.ids[row] : -1;
    float m = -INFINITY, s = 0.f, best = -INFINITY, xt = __int_as_float(0x7fc00000);
    int idx = 0x7fffffff;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c, r);
      tmem_ld_wait();
      if (!(do_store && row_ok)) continue;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int col = n0 + c + q * 4;
        if (col < args.n_out) tile_lse_step4(m, s, best, idx, r + q * 4, col);
      }
      const int off = tgt - (n0 + c);
      if (off >= 0 && off < 32) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i == off) xt = __uint_as_float(r[i]);
      }
    }
    if (do_store && row_ok) {
      TileLse t;
      t.m = m;
      t.s = s;
      t.best = best;
      t.xt = xt;
      t.idx = idx;
      t.pad[0] = t.pad[1] = t.pad[2] = 0;
      args.lse[(size_t)row * args.n_tiles + n_tile] = t;
    }
  } else {
    const int n0 = n_tile * BN;
    constexpr int CW = BN < 32 ? BN : 32;
#pragma unroll 1
    for (int c = 0; c < BN; c += CW) {
      uint32_t r[CW];
      tmem_ld_cols<CW>(t_row + c, r);
      tmem_ld_wait();
      if (!(do_store && row_ok)) continue;
      if (EPI == EPI_BF16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.C) + (size_t)row * args.ldc;
#pragma unroll
        for (int q = 0; q < CW / 8; ++q) {
          const int col = n0 + c + q * 8;
          if (col >= args.n_out) break;
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(r[q * 8 + 0]), __uint_as_float(r[q * 8 + 1]));
          v.y = pack_bf16x2(__uint_as_float(r[q * 8 + 2]), __uint_as_float(r[q * 8 + 3]));
          v.z = pack_bf16x2(__uint_as_float(r[q * 8 + 4]), __uint_as_float(r[q * 8 + 5]));
          v.w = pack_bf16x2(__uint_as_float(r[q * 8 + 6]), __uint_as_float(r[q * 8 + 7]));
          *reinterpret_cast<uint4*>(out + col) = v;
        }
      } else {
        float* out = (EPI == EPI_F32) ? static_cast<float*>(args.C) + (size_t)row * args.ldc
                                      : args.partial + ((size_t)split * args.M + row) * args.ldp;
#pragma unroll
        for (int q = 0; q < CW / 4; ++q) {
          const int col = n0 + c + q * 4;
          if (col >= args.n_out) break;
          *reinterpret_cast<float4*>(out + col) =
              make_float4(__uint_as_float(r[q * 4]), __uint_as_float(r[q * 4 + 1]), __uint_as_float(r[q * 4 + 2]),
                          __uint_as_float(r[q * 4 + 3]));
        }
      }
    }
  }
}

// Persistent warp-specialized kernel: one CTA per SM walks its tiles
// (t = blockIdx.x, blockIdx.x + gridDim.x, ...).  Warp 0 lane 0 = TMA producer,
// warp 1 = TMEM owner and (lane 0) MMA issuer, warps 2..5 = epilogue.  The fp32
// accumulator is double-buffered in TMEM so the epilogue of tile i overlaps
// the mainloop of tile i+1.  Each tile's MMAs, K order and epilogue are the
// same as for a lone tile: the schedule never changes results.
struct TileCoord {
  int m_tile, n_tile, split;
};

// Grouped rasterisation: group_m M-tiles at a time, N-tiles within the group,
// so that concurrently running tiles share their A and W tiles in L2.  Dense
// calls take 16; expert GEMMs take 1 (an M-tile's N-tiles in a row, M-tiles in
// order), so that the few M-tiles of one expert run together and fetch each of
// its weight tiles from DRAM once, whatever the expert boundaries.
constexpr int kGroupM = 16;
__device__ __forceinline__ TileCoord tile_coord(int t, int m_tiles, int n_tiles, int group_m) {
  TileCoord c;
  const int per_split = m_tiles * n_tiles;
  c.split = t / per_split;
  t -= c.split * per_split;
  const int per_group = group_m * n_tiles;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int gm = min(group_m, m_tiles - g * group_m);
  c.n_tile = r / gm;
  c.m_tile = g * group_m + (r - c.n_tile * gm);
  return c;
}

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                                                         const __grid_constant__ CUtensorMap tmB,
                                                         const __grid_constant__ CUtensorMap tmB2,
                                                         const GemmArgs args) {
  using S = GemmSmem<BN>;
  constexpr int kStages = S::kStages;
  constexpr bool kSwiglu = (EPI == EPI_SWIGLU || EPI == EPI_PARTIAL_SWIGLU);
  constexpr uint32_t kTmemCols = 2 * BN;  // two accumulator buffers
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * S::kBTileBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;   // [2] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;     // [2] epilogue -> MMA (4 warp arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* lse_ready = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // [2] LseStage: a 16-row tile is staged
  float* lse_stage = reinterpret_cast<float*>(sB + kStages * S::kBTileBytes + 256);  // LseStage only
  static_assert((2 * kStages + 4) * 8 + 8 + 16 <= 256, "barrier area");

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = args.m_tiles, n_tiles = args.n_tiles_grid;
  const int total = m_tiles * n_tiles * args.splits;
  const int nk = args.k_blocks_per_split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
      if (LseStage<BN, EPI>::kOn) mbar_init(&lse_ready[b], 1);
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
    if (kSwiglu) prefetch_tmap(&tmB2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // expert of an M-tile (grouped GEMM); -1 tiles are skipped by every role alike
  auto tile_expert = [&](int m_tile) { return args.tile_expert ? args.tile_expert[m_tile] : 0; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      auto load_w = [&](int expert, int n_tile, int kc, int s) {
        const int wbase = expert * args.w_rows_per_expert;
        if (kSwiglu) {
          const int j0 = n_tile * (BN / 2);
          tma_load_2d(sB + s * S::kBTileBytes, &tmB, &full[s], kc, wbase + j0);
          tma_load_2d(sB + s * S::kBTileBytes + (BN / 2) * kBK * 2, &tmB2, &full[s], kc,
                      wbase + args.up_offset + j0);
        } else {
          tma_load_2d(sB + s * S::kBTileBytes, &tmB, &full[s], kc, wbase + n_tile * BN);
        }
      };
      // bytes of one stage: the A rows the copy brings (a decode-size A leaves the
      // tile's other rows as they are; MMA rows never mix and rows >= M are
      // never stored) plus the W tile
      const uint32_t stage_bytes = (uint32_t)args.a_box_rows * kBK * 2 + S::kBTileBytes;
      int kb_total = 0;  // ring position across tiles
      bool first = true;
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, m_tiles, n_tiles, args.group_m);
        int expert = 0;
        int pre = 0;
        if (first && !args.tile_expert) {
          // weights never come from the preceding kernel: start fetching them
          // while it finishes; A is read only after the dependency wait
          pre = nk < kStages ? nk : kStages;
          for (int kb = 0; kb < pre; ++kb) {
            mbar_arrive_expect_tx(&full[kb], stage_bytes);
            load_w(0, tc.n_tile, (tc.split * nk + kb) * kBK, kb);
          }
        }
        if (first) pdl_wait();
        first = false;
        if (args.tile_expert) {
          expert = tile_expert(tc.m_tile);
          if (expert < 0) continue;
        }
        for (int kb = 0; kb < pre; ++kb)
          tma_load_2d(sA + kb * kATileBytes, &tmA, &full[kb], (tc.split * nk + kb) * kBK, tc.m_tile * kBM);
        kb_total += pre;
        for (int kb = pre; kb < nk; ++kb, ++kb_total) {
          const int s = kb_total % kStages;
          const uint32_t ph = (kb_total / kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1) || *abort_flag) {
            report(args.status, DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          const int kc = (tc.split * nk + kb) * kBK;
          tma_load_2d(sA + s * kATileBytes, &tmA, &full[s], kc, tc.m_tile * kBM);
          load_w(expert, tc.n_tile, kc, s);
        }
      }
      if (first) pdl_wait();  // no tile for this CTA: still order after the predecessor
      // let the last copies this CTA started land before it can exit
      for (int i = 0; i < kStages && i < kb_total; ++i) {
        const int kb = kb_total - 1 - i;
        mbar_wait(&full[kb % kStages], (kb / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      pdl_wait();
      int kb_total = 0, local = 0;
      for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, m_tiles, n_tiles, args.group_m);
        if (args.tile_expert && tile_expert(tc.m_tile) < 0) continue;
        const int b = local & 1;
        const uint32_t bph = (local >> 1) & 1;
        if (!mbar_wait(&acc_empty[b], bph ^ 1)) {
          report(args.status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + b * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++kb_total) {
          const int s = kb_total % kStages;
          const uint32_t ph = (kb_total / kStages) & 1;
          if (!mbar_wait(&full[s], ph) || *abort_flag) {
            report(args.status, DEV_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + s * kATileBytes);
          const uint32_t b_addr = smem_u32(sB + s * S::kBTileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            tc_mma_bf16(d, sw128_kmajor_desc(a_addr + k * 32), sw128_kmajor_desc(b_addr + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[b]);  // fires once this tile's MMAs have completed
        ++local;
        if (!ok) break;
      }
    }
  } else {
    // ---------------- epilogue warps 2..5: TMEM lane quarter q = warp % 4
    const int q = warp & 3;
    int local = 0;
    pdl_wait();
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, m_tiles, n_tiles, args.group_m);
      if (args.tile_expert && tile_expert(tc.m_tile) < 0) continue;
      const int b = local & 1;
      const uint32_t bph = (local >> 1) & 1;
      // decided for the whole warp: the TMEM loads below are warp-collective
      const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[b], bph));
      tc_fence_after();
      if (!acc_ok) {
        report(args.status, DEV_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      const int row = tc.m_tile * kBM + q * 32 + lane;
      bool small = false;
      if constexpr (LseStage<BN, EPI>::kOn) {
        small = args.M - tc.m_tile * kBM <= kLseSmallRows;
        if (small) {
          // a tile of at most 16 rows: TMEM lanes 0..15 staged by warp q = 0, then all
          // four epilogue warps (8 threads per row) form the rows' records
          float* stg = lse_stage + b * LseStage<BN, EPI>::kFloats;
          if (q == 0) {
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(tmem_base + b * BN + c, r);
              tmem_ld_wait();
              if (lane < kLseSmallRows) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                  *reinterpret_cast<float4*>(stg + lane * (BN + 4) + c + i) =
                      make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                                  __uint_as_float(r[i + 3]));
              }
            }
          }
          // the other warps wait for the staged rows (bounded; a stage buffer is
          // rewritten only after every epilogue warp has released its accumulator)
          bool staged = true;
          if (q == 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&lse_ready[b]);
          } else {
            staged = __all_sync(0xffffffffu, mbar_wait(&lse_ready[b], bph));
            if (!staged) {
              report(args.status, DEV_TIMEOUT);
              *abort_flag = 1;
            }
          }
          if (staged)
            lse_small_tile_row<BN>(args, stg, tc.m_tile, tc.n_tile, (warp - 2) * 32 + lane, !*abort_flag);
        }
      }
      if (!small) {
        epilogue_tile<BN, EPI>(args, tmem_base + b * BN + ((uint32_t)(q * 32) << 16), row, row < args.M,
                               !*abort_flag, tc.n_tile, tc.split);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++local;
      if (*abort_flag) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ decode-size rows
// Calls with M <= 16 rows (a decode step) of a dense weight.  One CTA per
// TN-wide output tile; MMA warp w accumulates the 16 x 8 slice of the tile's W
// rows 8w..8w+7 over the whole K in ascending 16-wide mma.sync steps
// (m16n8k16, fp32 accumulator starting at -0, the identity of the first add),
// while four loader warps stream the operands into shared memory.
// Each step is the same 16-term bf16 tensor-core dot product added to the
// accumulator as one tcgen05.mma K-step, which gives the same fp32 bits; the
// epilogue applies the same per-element formulas.  So every element equals
// the tcgen05 kernel's bit for bit (the row-invariance tests compare rows on
// both sides of M = 16).  What changes is the schedule for a tile of 16 rows:
// no TMEM, no stage ring, the whole W slice requested (cp.async) before the
// dependency wait, A after it, both consumed in 256-column K chunks as they
// land.  (Per-row bulk copies cost about 70 cycles each in the copy engine,
// more than these 16-row tiles' data takes through cp.async.)
constexpr int kRowsM = 16;
constexpr int kRowsKC = 256;
constexpr int kRowsMaxK = 4096;
constexpr size_t kRowsMaxSmem = 220 * 1024;

__host__ __device__ constexpr int rows_stride(int K) { return K * 2 + 16; }  // bytes; ldmatrix rows hit distinct banks
// barriers | A rows | W rows | staged accumulators [16][TN + 4]
__host__ constexpr size_t rows_smem_bytes(int K, int TN) {
  return 256 + (size_t)(kRowsM + TN) * rows_stride(K) + (size_t)kRowsM * (TN + 4) * 4;
}

constexpr int kRowsLoadWarps = 4;
template <int TN>
constexpr int rows_threads() { return (TN / 8 + kRowsLoadWarps) * 32; }

// The normalised A rows of a fused-norm call, into the padded shared rows sA:
// warp w of nw takes rows w, w + nw, ... (< M), lane l the 16-byte vectors
// l + 32 j (j < NJ) of a row.  K = 256 NJ, so each of the norm kernels' K/8
// threads owns exactly one vector and their warps are the j's: the sum of
// squares per vector, the xor butterfly per j and the j sums added in order
// are the norm kernels' operations (norm.cuh).  With write_res, x + res_in
// goes to res_out.  RB rows' loads are in flight together.
template <int NJ>
__device__ __forceinline__ void rows_norm(const GemmArgs& args, uint8_t* sA, int stride, int M, int w, int nw,
                                          int lane, bool write_res) {
  constexpr int RB = NJ >= 8 ? 1 : 2;
  const int K = args.K;
  const uint4* gam = reinterpret_cast<const uint4*>(args.ngamma);
  for (int r0 = w; r0 < M; r0 += RB * nw) {
    uint4 a[RB][NJ], h[RB][NJ];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const int r = r0 + b * nw;
      if (r >= M) continue;
      const uint4* xr = reinterpret_cast<const uint4*>(args.nx + (int64_t)r * K);
      const uint4* hr = args.nres_in ? reinterpret_cast<const uint4*>(args.nres_in + (int64_t)r * K) : nullptr;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        a[b][j] = xr[lane + 32 * j];
        if (args.nres_in) h[b][j] = hr[lane + 32 * j];
      }
    }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const int r = r0 + b * nw;
      if (r >= M) continue;
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (args.nres_in) {
          a[b][j] = norm_residual_add(a[b][j], h[b][j]);
          if (write_res) reinterpret_cast<uint4*>(args.nres_out + (int64_t)r * K)[lane + 32 * j] = a[b][j];
        }
        t += norm_warp_sum(norm_ss_vec(a[b][j], 0.f));
      }
      const float inv = norm_inv(t, K, args.neps);
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        *reinterpret_cast<uint4*>(sA + r * stride + (lane + 32 * j) * 16) = norm_apply(a[b][j], gam[lane + 32 * j], inv);
    }
  }
}

template <int EPI, int TN, int NJ = 0>
__global__ void __launch_bounds__(rows_threads<TN>()) gemm_rows_kernel(const __nv_bfloat16* __restrict__ A,
                                                                       const __nv_bfloat16* __restrict__ W,
                                                                       const GemmArgs args) {
  constexpr bool kSwiglu = EPI == EPI_SWIGLU;
  constexpr int kTS = TN + 4;  // staged accumulator row (floats)
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw);
  const int K = args.K, M = args.M, stride = rows_stride(K);
  uint8_t* sA = smem_raw + 256;
  uint8_t* sW = sA + kRowsM * stride;
  float* sT = reinterpret_cast<float*>(sW + TN * stride);
  const int nch = (K + kRowsKC - 1) / kRowsKC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  pdl_trigger();

  // global W row of tile row r (SwiGLU: gate rows, then the matching up rows), -1 past the weight
  auto w_row = [&](int r) -> int64_t {
    if (kSwiglu) {
      const int j = tile * (TN / 2) + (r % (TN / 2));
      if (j >= args.n_out) return -1;
      return r < TN / 2 ? j : (int64_t)args.n_out + j;
    }
    const int n = tile * TN + r;
    return n < args.n_out ? n : -1;
  };
  auto chunk_cols = [&](int c) { return min(kRowsKC, K - c * kRowsKC); };

  constexpr int kMmaWarps = TN / 8, kLoaders = kRowsLoadWarps * 32;
  if (threadIdx.x == 0) {
    // every loader arrives once per chunk when its copies have landed
    for (int c = 0; c < nch; ++c) mbar_init(&bar[c], kLoaders);
    fence_barrier_init();
  }
  __syncthreads();
  if (warp >= kMmaWarps) {
    // loader warps: warp lw copies rows lw, lw + 4, ... in 16-byte cp.async
    // pieces, lane by lane along the row.  The weights never come from the
    // preceding kernel and are in flight before the dependency wait; A follows
    // it chunk by chunk, each chunk's barrier completing once every loader's
    // copies up to it have landed.  Rows past the weight or past M are not
    // copied: MMA rows never mix, and those rows are never stored.
    // (One piece per lane per row and chunk, the row loop unrolled: a loop with
    // run-time bounds around each copy costs more issue slots than the copies.)
    const int lw = warp - kMmaWarps;
    for (int c = 0; c < nch; ++c) {
      const bool on = lane * 8 < chunk_cols(c);
      const int k = c * kRowsKC + lane * 8;
#pragma unroll 4
      for (int rr = 0; rr < TN / kRowsLoadWarps; ++rr) {
        const int r = lw + rr * kRowsLoadWarps;
        const int64_t gr = w_row(r);
        if (on && gr >= 0) cp_async16(sW + r * stride + k * 2, W + gr * K + k, true);
      }
    }
    pdl_wait();
    if constexpr (NJ == 0) {
      for (int c = 0; c < nch; ++c) {
        const bool on = lane * 8 < chunk_cols(c);
        const int k = c * kRowsKC + lane * 8;
#pragma unroll
        for (int rr = 0; rr < kRowsM / kRowsLoadWarps; ++rr) {
          const int r = lw + rr * kRowsLoadWarps;
          if (on && r < M) cp_async16(sA + r * stride + k * 2, A + (int64_t)r * K + k, true);
        }
        cp_async_mbar_arrive(&bar[c]);
      }
    } else {
      for (int c = 0; c < nch; ++c) cp_async_mbar_arrive(&bar[c]);  // the W copies only
    }
  } else {
    pdl_wait();  // the outputs below are written only after the preceding kernel is done
  }
  if constexpr (NJ != 0) {
    // every warp normalises its share of the rows (whole rows: the MMA starts
    // once all are written); CTA 0 also writes the new residual rows
    rows_norm<NJ>(args, sA, stride, M, warp, blockDim.x >> 5, lane, tile == 0);
    __syncthreads();
  }

  // MMA warps 0 .. TN/8-1 start on each chunk as soon as it has landed
  float d[4] = {-0.f, -0.f, -0.f, -0.f};
  bool ok = true;
  const uint32_t a_lane = smem_u32(sA) + (lane & 15) * stride + (lane >> 4) * 16;
  const uint32_t w_lane = smem_u32(sW) + (warp * 8 + (lane & 7)) * stride + (lane >> 3) * 16;
  for (int c = 0; c < nch && ok && warp < kMmaWarps; ++c) {
    // decided for the whole warp: ldmatrix and mma.sync below are warp-collective
    if (!__all_sync(0xffffffffu, mbar_wait(&bar[c], 0))) {
      ok = false;
      break;
    }
    const int k_end = c * kRowsKC + chunk_cols(c);
#pragma unroll 2
    for (int k = c * kRowsKC; k < k_end; k += 32) {
      uint32_t a0[4], a1[4], b0, b1, b2, b3;
      ldsm_x4(a_lane + k * 2, a0[0], a0[1], a0[2], a0[3]);
      ldsm_x4(a_lane + k * 2 + 32, a1[0], a1[1], a1[2], a1[3]);
      ldsm_x4(w_lane + k * 2, b0, b1, b2, b3);
      mma_bf16_16816(d, a0, b0, b1);
      mma_bf16_16816(d, a1, b2, b3);
    }
  }
  if (!ok) report(args.status, DEV_TIMEOUT);
  cp_async_wait<0>();  // this thread's copies have landed before it can leave
  ok = __syncthreads_and(ok);
  if (!ok) return;

  const int g = lane >> 2, t2 = 2 * (lane & 3);
  if constexpr (EPI == EPI_BF16 || EPI == EPI_F32) {
    const int col = tile * TN + warp * 8 + t2;
    if (warp < kMmaWarps && col < args.n_out) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = g + 8 * h;
        if (row >= M) continue;
        if (EPI == EPI_BF16)
          *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(args.C) + (size_t)row * args.ldc + col) =
              pack_bf16x2(d[2 * h], d[2 * h + 1]);
        else
          *reinterpret_cast<float2*>(static_cast<float*>(args.C) + (size_t)row * args.ldc + col) =
              make_float2(d[2 * h], d[2 * h + 1]);
      }
    }
  } else {
    // stage the 16 x TN accumulators, then apply the pairwise epilogue
    if (warp < kMmaWarps) {
      sT[g * kTS + warp * 8 + t2] = d[0];
      sT[g * kTS + warp * 8 + t2 + 1] = d[1];
      sT[(g + 8) * kTS + warp * 8 + t2] = d[2];
      sT[(g + 8) * kTS + warp * 8 + t2 + 1] = d[3];
    }
    __syncthreads();
    if constexpr (kSwiglu) {
      constexpr int H = TN / 2;
      const int j0 = tile * H;
      for (int i = threadIdx.x; i < kRowsM * H; i += blockDim.x) {
        const int row = i / H, j = i % H;
        if (row >= M || j0 + j >= args.n_out) continue;
        static_cast<__nv_bfloat16*>(args.C)[(size_t)row * args.ldc + j0 + j] =
            f2bf(swiglu_elem(sT[row * kTS + j], sT[row * kTS + H + j]));
      }
    } else if constexpr (EPI == EPI_ROPE) {
      // the tile is head `tile`: q and k heads rotate-half, v heads copied; rows as the tcgen05 epilogue
      const RopeKvArgs& ra = args.rope;
      constexpr int half = TN / 2;
      const int h = tile;
      for (int i = threadIdx.x; i < kRowsM * half; i += blockDim.x) {
        const int row = i / half, j = i % half;
        if (row >= M) continue;
        const int seq = ra.row_seq[row];
        const int64_t pos = ra.row_pos[row];
        if (pos < 0 || pos >= ra.max_pos) {
          if (j == 0) report(args.status, DEV_BAD_INDEX);
          continue;
        }
        int64_t blk = -1;
        const int32_t b = (pos / 64 < ra.max_blk) ? ra.block_table[(int64_t)seq * ra.max_blk + pos / 64] : -1;
        if (b >= 0 && b < ra.n_blocks) blk = b;
        else if (j == 0) report(args.status, DEV_BAD_INDEX);
        const int slot = (int)(pos % 64);
        const float x1 = sT[row * kTS + j], x2 = sT[row * kTS + half + j];
        __nv_bfloat16* dst;
        if (h < ra.Hq + ra.Hkv) {
          if (h < ra.Hq) dst = ra.q_out + ((int64_t)row * ra.Hq + h) * TN;
          else if (blk >= 0) dst = ra.k_cache + ((blk * ra.Hkv + (h - ra.Hq)) * 64 + slot) * TN;
          else continue;
          const float* cs = ra.table + pos * TN;
          float o1, o2;
          rope_pair(x1, x2, cs[j], cs[half + j], o1, o2);
          dst[j] = f2bf(o1);
          dst[half + j] = f2bf(o2);
        } else {
          if (blk < 0) continue;
          dst = ra.v_cache + ((blk * ra.Hkv + (h - ra.Hq - ra.Hkv)) * 64 + slot) * TN;
          dst[j] = f2bf(x1);
          dst[half + j] = f2bf(x2);
        }
      }
    }
  }
}

// Split-K reduction of the non-invariant path: sums partials in split order.
template <int EPI>
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int M, int n_out, int ldp,
                                     void* C) {
  pdl_trigger();
  pdl_wait();
  const int64_t total = (int64_t)M * n_out;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / n_out;
    const int n = (int)(i % n_out);
    float a = 0.f, b = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float* p = part + ((int64_t)s * M + m) * ldp;
      a += p[n];
      if (EPI == EPI_SWIGLU) b += p[n_out + n];
    }
    if (EPI == EPI_BF16) {
      static_cast<__nv_bfloat16*>(C)[i] = f2bf(a);
    } else if (EPI == EPI_F32) {
      static_cast<float*>(C)[i] = a;
    } else {
      const float gb = bf2f(f2bf(a)), ub = bf2f(f2bf(b));
      static_cast<__nv_bfloat16*>(C)[i] = f2bf(__fmul_rn(silu_f(gb), ub));
    }
  }
}

// ------------------------------------------------------------------ host side
template <int BN, int EPI>
static bi_status launch_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const GemmArgs& args,
                           dim3 grid, cudaStream_t st) {
  constexpr int smem = gemm_tc_smem<BN, EPI>();
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err != cudaSuccess) return fail(BI_ERR_CUDA, std::string("gemm smem attribute: ") + cudaGetErrorString(attr_err));
  return launched(launch_pdl(gemm_tc_kernel<BN, EPI>, grid, dim3(192), smem, st, a, b, b2, args), "gemm_tc_kernel");
}

template <int EPI>
static bi_status dispatch_bn(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                             const GemmArgs& args, dim3 grid, cudaStream_t st) {
  switch (bn) {
    case 16:
      if constexpr (EPI != EPI_LSE && EPI != EPI_ROPE && EPI != EPI_SWIGLU && EPI != EPI_PARTIAL_SWIGLU)
        return launch_tc<16, EPI>(a, b, b2, args, grid, st);
      break;
    case 32:
      if constexpr (EPI != EPI_LSE && EPI != EPI_ROPE) return launch_tc<32, EPI>(a, b, b2, args, grid, st);
      break;
    case 64: return launch_tc<64, EPI>(a, b, b2, args, grid, st);
    case 128: return launch_tc<128, EPI>(a, b, b2, args, grid, st);
    case 256: return launch_tc<256, EPI>(a, b, b2, args, grid, st);
  }
  return fail(BI_ERR_UNSUPPORTED_SHAPE, "gemm: bad tile width");
}

static bi_status dispatch_epi(int epi, int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                              const GemmArgs& args, dim3 grid, cudaStream_t st) {
  switch (epi) {
    case EPI_BF16: return dispatch_bn<EPI_BF16>(bn, a, b, b2, args, grid, st);
    case EPI_F32: return dispatch_bn<EPI_F32>(bn, a, b, b2, args, grid, st);
    case EPI_SWIGLU: return dispatch_bn<EPI_SWIGLU>(bn, a, b, b2, args, grid, st);
    case EPI_PARTIAL: return dispatch_bn<EPI_PARTIAL>(bn, a, b, b2, args, grid, st);
    case EPI_PARTIAL_SWIGLU: return dispatch_bn<EPI_PARTIAL_SWIGLU>(bn, a, b, b2, args, grid, st);
    case EPI_LSE: return dispatch_bn<EPI_LSE>(bn, a, b, b2, args, grid, st);
    case EPI_ROPE: return dispatch_bn<EPI_ROPE>(bn, a, b, b2, args, grid, st);
  }
  return fail(BI_ERR_UNSUPPORTED_SHAPE, "gemm: bad epilogue");
}

// Accumulator tile width for a weight: a function of its shape (N, K, number of
// experts) and of the epilogue only, never of M.  Dense weights under 1M
// elements take 16-wide tiles, and SwiGLU weights under 2M elements 32-wide
// ones (16 gate and 16 up columns), so that a decode-size call spreads a small
// weight over many CTAs and each CTA's slice of it is in flight before the
// dependency wait; other weights under 2M elements 64; then 128, and weights of 16M+ elements, 32K+ rows, or
// expert weights of 256+ rows 256, where the tensor pipe rather than shared
// memory bandwidth bounds a prefill-size call.  The fused log-softmax keeps
// 64+ and the fused RoPE whole heads (both raised by the caller).
static int tile_n_for(int64_t n_rows_w, int64_t K, bool swiglu, int64_t E = 1) {
  const int64_t elems = n_rows_w * K;
  if (E == 1 && !swiglu && elems < (int64_t(1) << 20)) return 16;
  if (E == 1 && swiglu && elems < (int64_t(1) << 21)) return 32;
  if (elems < (int64_t(1) << 21)) return 64;
  if (E > 1 && n_rows_w >= 256) return 256;  // expert weights: a layer's experts together are large
  if (elems < (int64_t(1) << 24) && n_rows_w < 32768) return 128;
  return 256;
}

// Tile width of a decode-size call (17..128 rows) of a dense weight without the
// fused log-softmax or RoPE: an element's bits do not depend on the tile width
// (only the log-softmax records do, and RoPE needs whole heads), so the width
// that minimises the bytes the busiest CTA reads (its tiles x (the call's A
// rows + its W slice)) is taken, spreading a large weight over the GPU.
static int decode_tile_n(int64_t M, int64_t n_rows_w, int64_t K, bool swiglu, int bn_weight) {
  const int64_t n_out = swiglu ? n_rows_w / 2 : n_rows_w;
  const int64_t a_rows = std::max<int64_t>(8, cdiv(M, 8) * 8);
  int best = bn_weight;
  double best_bytes = 0.0;
  for (int bn : {256, 128, 64, 32, 16}) {
    if (swiglu && bn < 32) continue;
    const int64_t tiles = cdiv(n_out, swiglu ? bn / 2 : bn);
    const int64_t per_cta = cdiv(tiles, (int64_t)num_sms());
    const double bytes = (double)per_cta * (double)(a_rows + bn) * (double)K * 2.0;
    if (best_bytes == 0.0 || bytes < best_bytes) {
      best = bn;
      best_bytes = bytes;
    }
  }
  return best;
}

// Tile width of a call of more than 128 rows on a weight whose own width is
// below 256 (the width that spreads the weight over the GPU at decode size).
// Bits do not depend on the width, so a prefill pass takes the width that
// minimises the bytes its busiest CTA reads over all its tiles (tiles x (128 A
// rows + the W slice)): 16- or 32-wide tiles would re-read the A rows once per 16
// or 32 columns, and at thousands of rows 256-wide tiles carry twice the MMA work
// per staged byte of 128-wide ones.  min_bn: SwiGLU pairs need 32, RoPE whole
// heads (and a width that divides N).
static int wide_tile_n(int64_t M, int64_t n_rows_w, bool swiglu, int min_bn, bool divides, int bn_weight) {
  const int64_t n_out = swiglu ? n_rows_w / 2 : n_rows_w;
  const int64_t m_tiles = cdiv(M, kBM);
  int best = bn_weight;
  double best_bytes = 0.0;
  for (int bn : {256, 128, 64, 32, 16}) {
    if (bn < min_bn || (divides && (n_out % bn || bn % min_bn))) continue;
    const int64_t tiles = m_tiles * cdiv(n_out, swiglu ? bn / 2 : bn);
    const int64_t per_cta = cdiv(tiles, (int64_t)num_sms());
    const double bytes = (double)per_cta * (double)(kBM + bn);
    if (best_bytes == 0.0 || bytes < best_bytes) {
      best = bn;
      best_bytes = bytes;
    }
  }
  return best;
}

// Non-invariant choices (BI_FAST): tile width and split count chosen from M.
static void fast_plan(int64_t M, int64_t n_rows_w, int64_t K, bool swiglu, int* bn, int* splits) {
  *bn = tile_n_for(n_rows_w, K, swiglu);
  *splits = 1;
  if (M > 128) return;
  *bn = std::min(*bn, 64);
  const int64_t n_cols = swiglu ? n_rows_w / 2 : n_rows_w;
  const int64_t tiles = cdiv(n_cols, swiglu ? *bn / 2 : *bn);
  const int64_t kblocks = K / kBK;
  int64_t s = cdiv((int64_t)num_sms(), tiles);
  s = std::min<int64_t>(s, kblocks / 2 > 0 ? kblocks / 2 : 1);
  while (s > 1 && kblocks % s) --s;
  *splits = (int)std::max<int64_t>(s, 1);
}

struct GemmCall {
  const void* A;
  int64_t M, K;
  const void* W;
  int64_t n_rows_w;        // rows of W per expert (2F for SwiGLU)
  int64_t E;               // number of experts (1 = dense)
  const int32_t* tile_expert;
  void* C;
  int c_dtype, epilogue, mode;
  void* ws;
  size_t ws_bytes;
  const int32_t* ids = nullptr;  // fused log-softmax: targets (NULL = greedy)
  TileLse* lse = nullptr;        // fused log-softmax: tile partials (non-NULL selects it)
  const RopeKvArgs* rope = nullptr;  // fused RoPE + paged KV write (non-NULL selects it)
  const NormIn* norm = nullptr;      // RMSNorm in front (A unused; non-NULL selects it)
};

template <int EPI, int TN, int NJ = 0>
static bi_status launch_rows(const void* A, const void* W, const GemmArgs& args, int n_tiles, size_t smem,
                             cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_rows_kernel<EPI, TN, NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kRowsMaxSmem);
  });
  if (attr_err != cudaSuccess)
    return fail(BI_ERR_CUDA, std::string("gemm rows smem attribute: ") + cudaGetErrorString(attr_err));
  return launched(launch_pdl(gemm_rows_kernel<EPI, TN, NJ>, dim3(n_tiles), dim3(rows_threads<TN>()), smem, st,
                             static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(W), args),
                  "gemm_rows_kernel");
}

// Output columns per CTA of the decode-size schedule (never changes results):
// 16 (SwiGLU: 16 gate + 16 up), whole heads for the fused RoPE.
static int rows_tile(const GemmCall& g, bool swiglu) {
  if (g.rope) return g.rope->hd;
  return swiglu ? 32 : 16;
}

// The decode-size schedule takes dense calls of at most 16 rows of a weight
// under 4M elements (a decoder layer's projections; larger weights, such as a
// vocabulary head, stream faster through the tcgen05 kernel's TMA ring) whose
// W slice and rows fit shared memory, in either mode (BI_FAST has nothing
// faster for them); the fused log-softmax stays on the tcgen05 kernel.
static bool rows_path(const GemmCall& g, int64_t n_out, bool swiglu) {
  if (g.M < 1 || g.M > kRowsM || g.E != 1 || g.tile_expert || g.lse) return false;
  if (g.n_rows_w * g.K >= (int64_t(1) << 22)) return false;
  if (g.K % 64 || g.K > kRowsMaxK || n_out % 8) return false;
  if ((reinterpret_cast<uintptr_t>(g.A) | reinterpret_cast<uintptr_t>(g.W)) & 15) return false;
  if (g.rope && ((g.rope->hd != 64 && g.rope->hd != 128) || g.n_rows_w % g.rope->hd)) return false;
  return rows_smem_bytes((int)g.K, rows_tile(g, swiglu)) <= kRowsMaxSmem;
}

// The RMSNorm folds into the decode-size schedule for the SwiGLU and fused-RoPE
// (head_dim 64) epilogues when K is 512, 1024 or 2048 (norm_nj = K / 256).
static int norm_nj(const GemmCall& g, bool swiglu) {
  if (!(swiglu || (g.rope && g.rope->hd == 64))) return 0;
  return (g.K == 512 || g.K == 1024 || g.K == 2048) ? (int)(g.K / 256) : 0;
}

template <int EPI, int TN>
static bi_status launch_rows_nj(int nj, const GemmCall& g, const GemmArgs& args, int n_tiles, size_t smem,
                                cudaStream_t st) {
  switch (nj) {
    case 2: return launch_rows<EPI, TN, 2>(g.A, g.W, args, n_tiles, smem, st);
    case 4: return launch_rows<EPI, TN, 4>(g.A, g.W, args, n_tiles, smem, st);
    case 8: return launch_rows<EPI, TN, 8>(g.A, g.W, args, n_tiles, smem, st);
  }
  return fail(BI_ERR_UNSUPPORTED_SHAPE, "gemm: norm width");
}

static bi_status run_rows(const GemmCall& g, int64_t n_out, bool swiglu, cudaStream_t st) {
  GemmArgs args = {};
  const int nj = g.norm ? norm_nj(g, swiglu) : 0;
  if (nj) {
    args.nx = static_cast<const __nv_bfloat16*>(g.norm->x);
    args.nres_in = static_cast<const __nv_bfloat16*>(g.norm->res_in);
    args.nres_out = static_cast<__nv_bfloat16*>(g.norm->res_out);
    args.ngamma = static_cast<const __nv_bfloat16*>(g.norm->gamma);
    args.neps = g.norm->eps;
  }
  args.C = g.C;
  args.status = device_status_ptr();
  args.M = (int)g.M;
  args.K = (int)g.K;
  args.ldc = (int)n_out;
  args.n_out = (int)n_out;
  const int tn = rows_tile(g, swiglu);
  const size_t smem = rows_smem_bytes((int)g.K, tn);
  if (g.rope) {
    args.rope = *g.rope;
    const int heads = (int)(g.n_rows_w / tn);
    if (nj) return launch_rows_nj<EPI_ROPE, 64>(nj, g, args, heads, smem, st);
    return tn == 64 ? launch_rows<EPI_ROPE, 64>(g.A, g.W, args, heads, smem, st)
                    : launch_rows<EPI_ROPE, 128>(g.A, g.W, args, heads, smem, st);
  }
  const int n_tiles = (int)cdiv(n_out, 16);
  if (swiglu) {
    if (nj) return launch_rows_nj<EPI_SWIGLU, 32>(nj, g, args, n_tiles, smem, st);
    return launch_rows<EPI_SWIGLU, 32>(g.A, g.W, args, n_tiles, smem, st);
  }
  return g.c_dtype == BI_DTYPE_FP32 ? launch_rows<EPI_F32, 16>(g.A, g.W, args, n_tiles, smem, st)
                                    : launch_rows<EPI_BF16, 16>(g.A, g.W, args, n_tiles, smem, st);
}

static size_t partial_bytes(int64_t M, int64_t n_rows_w, int splits) {
  return splits > 1 ? (size_t)splits * M * n_rows_w * sizeof(float) : 0;
}

static bi_status run_gemm(const GemmCall& g, cudaStream_t st) {
  const bool swiglu = g.epilogue == BI_EPI_SWIGLU;
  const int64_t n_out = swiglu ? g.n_rows_w / 2 : g.n_rows_w;
  if (g.norm) {
    if (rows_path(g, n_out, swiglu) && norm_nj(g, swiglu)) return run_rows(g, n_out, swiglu, st);
    // the norm as its own kernel, then the GEMM of its rows
    const NormIn& n = *g.norm;
    BI_TRY(rmsnorm_rows_to(n.x, n.res_in, n.res_out, n.gamma, n.y, g.M, g.K, n.eps, nullptr, st));
    GemmCall plain = g;
    plain.norm = nullptr;
    plain.A = n.y;
    return run_gemm(plain, st);
  }
  if (rows_path(g, n_out, swiglu)) return run_rows(g, n_out, swiglu, st);
  int bn = tile_n_for(g.n_rows_w, g.K, swiglu, g.E), splits = 1;
  if (g.mode == BI_FAST && g.E == 1) {
    fast_plan(g.M, g.n_rows_w, g.K, swiglu, &bn, &splits);
    if (g.lse || g.rope) splits = 1;  // fused epilogues keep whole K per tile; FAST narrows the tiles instead
  }
  if (!g.lse && !g.rope && g.E == 1 && !g.tile_expert && g.M <= kBM && splits == 1)
    bn = decode_tile_n(g.M, g.n_rows_w, g.K, swiglu, bn);
  if (!g.lse && g.E == 1 && !g.tile_expert && g.M > kBM && splits == 1 && bn < 256)
    bn = wide_tile_n(g.M, g.n_rows_w, swiglu, g.rope ? g.rope->hd : (swiglu ? 32 : 16), g.rope != nullptr, bn);
  if (g.lse && bn < 64) bn = 64;  // the fused log-softmax records are per 64+ vocab columns
  if (g.rope) {
    // a tile must hold whole heads so that rotate-half pairs meet in one thread
    while (bn < g.rope->hd) bn *= 2;
    if (bn % g.rope->hd) return fail(BI_ERR_UNSUPPORTED_SHAPE, "QKV tile width must be a multiple of head_dim");
  }
  const int64_t kblocks = g.K / kBK;

  CUtensorMap ta, tb, tb2;
  // a dense call with M < 128 copies only its M rows (rounded up to 8) of A per stage
  const int a_box_rows = (g.M < kBM && g.E == 1 && !g.tile_expert) ? (int)std::max<int64_t>(8, cdiv(g.M, 8) * 8)
                                                                    : kBM;
  if (!encode_tmap_2d_bf16(&ta, g.A, g.K, g.M, g.K * 2, kBK, (uint32_t)a_box_rows, true))
    return fail(BI_ERR_CUDA, "gemm: TMA descriptor for A failed");
  const uint32_t box_b = swiglu ? bn / 2 : bn;
  if (g.E == 1 && swiglu) {
    const char* w = static_cast<const char*>(g.W);
    if (!encode_tmap_2d_bf16(&tb, w, g.K, n_out, g.K * 2, kBK, box_b, true) ||
        !encode_tmap_2d_bf16(&tb2, w + n_out * g.K * 2, g.K, n_out, g.K * 2, kBK, box_b, true))
      return fail(BI_ERR_CUDA, "gemm: TMA descriptor for W failed");
  } else {
    if (!encode_tmap_2d_bf16(&tb, g.W, g.K, g.n_rows_w * g.E, g.K * 2, kBK, box_b, true))
      return fail(BI_ERR_CUDA, "gemm: TMA descriptor for W failed");
    tb2 = tb;
  }

  GemmArgs args;
  args.C = g.C;
  args.partial = nullptr;
  args.tile_expert = g.tile_expert;
  args.status = device_status_ptr();
  args.M = (int)g.M;
  args.K = (int)g.K;
  args.ldc = (int)n_out;
  args.n_out = (int)n_out;
  args.w_rows_per_expert = g.E > 1 || g.tile_expert ? (int)g.n_rows_w : 0;
  args.up_offset = (g.E == 1 && !g.tile_expert) ? 0 : (int)n_out;
  args.k_blocks_per_split = (int)(kblocks / splits);
  args.ldp = (int)g.n_rows_w;
  args.ids = g.ids;
  args.lse = g.lse;
  if (g.rope) args.rope = *g.rope;

  const int64_t n_tiles = swiglu ? cdiv(n_out, bn / 2) : cdiv(n_out, bn);
  args.n_tiles = (int)n_tiles;
  args.m_tiles = (int)cdiv(g.M, kBM);
  args.n_tiles_grid = (int)n_tiles;
  args.splits = splits;
  args.a_box_rows = a_box_rows;
  args.group_m = g.tile_expert ? 1 : kGroupM;
  const int64_t tiles = (int64_t)args.m_tiles * n_tiles * splits;
  BI_REQUIRE_SHAPE(tiles < (1ll << 31), "too many tiles");
  dim3 grid((unsigned)std::min<int64_t>(tiles, num_sms()));
  int epi;
  if (g.lse) {
    if (splits != 1) return fail(BI_ERR_INVALID_ARG, "fused log-softmax cannot run split-K");
    epi = EPI_LSE;
  } else if (g.rope) {
    epi = EPI_ROPE;
  } else if (splits > 1) {
    if (g.ws_bytes < partial_bytes(g.M, g.n_rows_w, splits) || !g.ws)
      return fail(BI_ERR_INVALID_ARG, "bi_gemm: BI_FAST split-K needs workspace (bi_gemm_workspace_size)");
    args.partial = static_cast<float*>(g.ws);
    epi = swiglu ? EPI_PARTIAL_SWIGLU : EPI_PARTIAL;
  } else {
    epi = swiglu ? EPI_SWIGLU : (g.c_dtype == BI_DTYPE_FP32 ? EPI_F32 : EPI_BF16);
  }
  BI_TRY(dispatch_epi(epi, bn, ta, tb, tb2, args, grid, st));
  if (splits > 1) {
    const int64_t total = g.M * n_out;
    const int blocks = (int)std::min<int64_t>(cdiv(total, 256), 4 * (int64_t)num_sms());
    auto* kern = swiglu ? splitk_reduce_kernel<EPI_SWIGLU>
                        : (g.c_dtype == BI_DTYPE_FP32 ? splitk_reduce_kernel<EPI_F32> : splitk_reduce_kernel<EPI_BF16>);
    BI_TRY(launched(launch_pdl(kern, dim3(blocks), dim3(256), 0, st, (const float*)args.partial, splits, (int)g.M,
                               (int)n_out, (int)g.n_rows_w, g.C),
                    "splitk_reduce_kernel"));
  }
  return BI_OK;
}

}  // namespace bi

extern "C" {

int bi_gemm_tile_n(int64_t N, int64_t K, int epilogue) { return bi::tile_n_for(N, K, epilogue == BI_EPI_SWIGLU); }

size_t bi_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int epilogue, int mode) {
  if (mode != BI_FAST || M <= 0 || K % bi::kBK) return 0;
  int bn, splits;
  bi::fast_plan(M, N, K, epilogue == BI_EPI_SWIGLU, &bn, &splits);
  return bi::partial_bytes(M, N, splits);
}

bi_status bi_gemm(const void* A, int64_t M, int64_t K, const void* W, int64_t N, void* C, int c_dtype, int epilogue,
                  int mode, void* workspace, size_t ws_bytes, void* stream) {
  using namespace bi;
  BI_REQUIRE(M >= 0 && N > 0 && K > 0, "bad shape");
  if (M == 0) return BI_OK;
  BI_REQUIRE(A && W && C, "null pointer");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  BI_REQUIRE(epilogue == BI_EPI_NONE || epilogue == BI_EPI_SWIGLU, "bad epilogue");
  BI_REQUIRE(c_dtype == BI_DTYPE_BF16 || c_dtype == BI_DTYPE_FP32, "bad c_dtype");
  BI_REQUIRE(epilogue != BI_EPI_SWIGLU || c_dtype == BI_DTYPE_BF16, "SwiGLU output is bf16");
  BI_REQUIRE(aligned16(A) && aligned16(W) && aligned16(C), "pointers must be 16-byte aligned");
  BI_REQUIRE_SHAPE(K % 64 == 0, "K must be a multiple of 64");
  BI_REQUIRE_SHAPE(N % 8 == 0, "N must be a multiple of 8");
  BI_REQUIRE_SHAPE(epilogue != BI_EPI_SWIGLU || (N % 16 == 0), "SwiGLU needs N = 2F with F % 8 == 0");
  BI_REQUIRE_SHAPE(M < (1ll << 31) && N < (1ll << 31) && K < (1ll << 31), "shape too large");
  GemmCall g{A, M, K, W, N, 1, nullptr, C, c_dtype, epilogue, mode, workspace, ws_bytes};
  return run_gemm(g, as_stream(stream));
}

bi_status bi_grouped_gemm(const void* A, int64_t M_rows, int64_t K, const void* W, int64_t E, int64_t N,
                          const int32_t* tile_expert, void* C, int c_dtype, int epilogue, void* stream) {
  using namespace bi;
  BI_REQUIRE(M_rows >= 0 && N > 0 && K > 0 && E > 0, "bad shape");
  if (M_rows == 0) return BI_OK;
  BI_REQUIRE(A && W && C && tile_expert, "null pointer");
  BI_REQUIRE(M_rows % 128 == 0, "M_rows must be a multiple of 128");
  BI_REQUIRE(epilogue == BI_EPI_NONE || epilogue == BI_EPI_SWIGLU, "bad epilogue");
  BI_REQUIRE(c_dtype == BI_DTYPE_BF16 || c_dtype == BI_DTYPE_FP32, "bad c_dtype");
  BI_REQUIRE(epilogue != BI_EPI_SWIGLU || c_dtype == BI_DTYPE_BF16, "SwiGLU output is bf16");
  BI_REQUIRE(aligned16(A) && aligned16(W) && aligned16(C), "pointers must be 16-byte aligned");
  BI_REQUIRE_SHAPE(K % 64 == 0, "K must be a multiple of 64");
  const bool swiglu = epilogue == BI_EPI_SWIGLU;
  const int bn = tile_n_for(N, K, swiglu, E);
  BI_REQUIRE_SHAPE(swiglu ? (N / 2) % (bn / 2) == 0 : N % bn == 0,
                   "grouped GEMM needs the per-expert N to be a multiple of the tile width");
  BI_REQUIRE_SHAPE(M_rows < (1ll << 31) && N * E < (1ll << 31), "shape too large");
  GemmCall g{A, M_rows, K, W, N, E, tile_expert, C, c_dtype, epilogue, BI_INVARIANT, nullptr, 0};
  return run_gemm(g, as_stream(stream));
}

}  // extern "C"

// ----------------------------------------------- fused lm_head + log-softmax
namespace bi {

// Vocab tile width of the fused head: the invariant width of the weight, or
// (BI_FAST, at most 128 rows) the narrow width that spreads the vocab over more CTAs.
static int lm_head_tile_n(int64_t T, int64_t V, int64_t K, int mode) {
  int bn = tile_n_for(V, K, false), splits = 1;
  if (mode == BI_FAST) fast_plan(T, V, K, false, &bn, &splits);
  return std::max(bn, 64);  // the records are per 64+ vocab columns (as run_gemm raises it)
}

size_t lm_head_partial_bytes(int64_t T, int64_t V, int64_t K, int mode) {
  if (T <= 0 || V <= 0) return 0;
  return (size_t)T * cdiv(V, lm_head_tile_n(T, V, K, mode)) * sizeof(TileLse);
}

bi_status lm_head_logprob_to(const void* X, int64_t T, int64_t K, const void* W, int64_t V, const int32_t* ids,
                             float* logprob_out, int32_t* argmax_out, const int32_t* dst, int mode, void* workspace,
                             size_t ws_bytes, void* stream) {
  BI_REQUIRE(T >= 0 && V > 0 && K > 0, "bad shape");
  if (T == 0) return BI_OK;
  BI_REQUIRE(X && W && logprob_out && workspace, "null pointer");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  BI_REQUIRE(aligned16(X) && aligned16(W) && aligned16(workspace), "pointers must be 16-byte aligned");
  BI_REQUIRE_SHAPE(K % 64 == 0, "K must be a multiple of 64");
  BI_REQUIRE_SHAPE(V % 8 == 0, "V must be a multiple of 8");
  BI_REQUIRE_SHAPE(T < (1ll << 31) && V < (1ll << 31), "shape too large");
  BI_REQUIRE(ws_bytes >= lm_head_partial_bytes(T, V, K, mode), "workspace too small (bi_lm_head_logprob_workspace_size)");
  const int bn = lm_head_tile_n(T, V, K, mode);
  GemmCall g{X, T, K, W, V, 1, nullptr, nullptr, BI_DTYPE_FP32, BI_EPI_NONE, mode, nullptr, 0};
  g.ids = ids;
  g.lse = static_cast<TileLse*>(workspace);
  BI_TRY(run_gemm(g, as_stream(stream)));
  return lse_tiles_merge(g.lse, T, (int)cdiv(V, bn), bn, ids, logprob_out, argmax_out, dst, stream);
}

}  // namespace bi

extern "C" {

size_t bi_lm_head_logprob_workspace_size(int64_t T, int64_t V, int64_t K, int mode) {
  return bi::lm_head_partial_bytes(T, V, K, mode);
}

bi_status bi_lm_head_logprob(const void* X, int64_t T, int64_t K, const void* W, int64_t V, const int32_t* ids,
                             float* logprob_out, int32_t* argmax_out, int mode, void* workspace, size_t ws_bytes,
                             void* stream) {
  return bi::lm_head_logprob_to(X, T, K, W, V, ids, logprob_out, argmax_out, nullptr, mode, workspace, ws_bytes,
                                stream);
}

}  // extern "C"

// ------------------------------------------- fused QKV + RoPE + paged KV write
namespace bi {

bi_status gemm_qkv_rope(const void* A, int64_t M, int64_t K, const void* W, int64_t N, const int32_t* row_seq,
                        const int32_t* row_pos, const float* rope_table, int64_t max_pos, const int32_t* block_table,
                        int64_t max_blk, int64_t n_blocks, void* q_out, void* k_cache, void* v_cache, int Hq, int Hkv,
                        int hd, int mode, void* stream) {
  BI_REQUIRE(M >= 0 && K > 0 && N > 0, "bad shape");
  if (M == 0) return BI_OK;
  BI_REQUIRE(A && W && row_seq && row_pos && rope_table && block_table && q_out && k_cache && v_cache, "null pointer");
  BI_REQUIRE(N == (int64_t)(Hq + 2 * Hkv) * hd, "N must be (Hq + 2 Hkv) * head_dim");
  BI_REQUIRE_SHAPE(hd == 64 || hd == 128, "head_dim must be 64 or 128");
  BI_REQUIRE_SHAPE(K % 64 == 0, "K must be a multiple of 64");
  BI_REQUIRE(aligned16(A) && aligned16(W) && aligned16(q_out) && aligned16(k_cache) && aligned16(v_cache) &&
                 aligned16(rope_table),
             "pointers must be 16-byte aligned");
  RopeKvArgs ra{row_seq, row_pos, rope_table, block_table, static_cast<__nv_bfloat16*>(q_out),
                static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), max_pos, max_blk,
                n_blocks, Hq, Hkv, hd};
  GemmCall g{A, M, K, W, N, 1, nullptr, q_out, BI_DTYPE_BF16, BI_EPI_NONE, mode, nullptr, 0};
  g.rope = &ra;
  return run_gemm(g, as_stream(stream));
}

static bi_status check_norm(const NormIn& n, int64_t K) {
  BI_REQUIRE(n.x && n.gamma && n.y, "null pointer");
  BI_REQUIRE(!n.res_in == !n.res_out, "res_in and res_out go together");
  BI_REQUIRE(!n.res_in || n.res_in != n.res_out, "res_out must be another buffer than res_in");
  BI_REQUIRE(aligned16(n.x) && aligned16(n.gamma) && aligned16(n.y) &&
                 (!n.res_in || (aligned16(n.res_in) && aligned16(n.res_out))),
             "pointers must be 16-byte aligned");
  BI_REQUIRE(n.eps > 0.f, "eps must be positive");
  BI_REQUIRE_SHAPE(K <= 16384, "K must be at most 16384 for the norm");
  return BI_OK;
}

bi_status gemm_norm(const NormIn& norm, int64_t M, int64_t K, const void* W, int64_t N, void* C, int epilogue,
                    int mode, void* workspace, size_t ws_bytes, void* stream) {
  BI_REQUIRE(M >= 0 && K > 0 && N > 0, "bad shape");
  if (M == 0) return BI_OK;
  BI_REQUIRE(W && C, "null pointer");
  BI_REQUIRE(epilogue == BI_EPI_NONE || epilogue == BI_EPI_SWIGLU, "bad epilogue");
  BI_REQUIRE_SHAPE(K % 64 == 0 && (epilogue != BI_EPI_SWIGLU || N % 2 == 0), "bad GEMM shape");
  BI_REQUIRE(aligned16(W) && aligned16(C), "pointers must be 16-byte aligned");
  BI_TRY(check_norm(norm, K));
  GemmCall g{nullptr, M, K, W, N, 1, nullptr, C, BI_DTYPE_BF16, epilogue, mode, workspace, ws_bytes};
  g.norm = &norm;
  return run_gemm(g, as_stream(stream));
}

bi_status gemm_qkv_rope_norm(const NormIn& norm, int64_t M, int64_t K, const void* W, int64_t N,
                             const int32_t* row_seq, const int32_t* row_pos, const float* rope_table, int64_t max_pos,
                             const int32_t* block_table, int64_t max_blk, int64_t n_blocks, void* q_out,
                             void* k_cache, void* v_cache, int Hq, int Hkv, int hd, int mode, void* stream) {
  BI_REQUIRE(M >= 0 && K > 0 && N > 0, "bad shape");
  if (M == 0) return BI_OK;
  BI_REQUIRE(W && row_seq && row_pos && rope_table && block_table && q_out && k_cache && v_cache, "null pointer");
  BI_REQUIRE(N == (int64_t)(Hq + 2 * Hkv) * hd, "N must be (Hq + 2 Hkv) * head_dim");
  BI_REQUIRE_SHAPE(hd == 64 || hd == 128, "head_dim must be 64 or 128");
  BI_REQUIRE_SHAPE(K % 64 == 0, "K must be a multiple of 64");
  BI_REQUIRE(aligned16(W) && aligned16(q_out) && aligned16(k_cache) && aligned16(v_cache) &&
                 aligned16(rope_table),
             "pointers must be 16-byte aligned");
  BI_TRY(check_norm(norm, K));
  RopeKvArgs ra{row_seq, row_pos, rope_table, block_table, static_cast<__nv_bfloat16*>(q_out),
                static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), max_pos, max_blk,
                n_blocks, Hq, Hkv, hd};
  GemmCall g{nullptr, M, K, W, N, 1, nullptr, q_out, BI_DTYPE_BF16, BI_EPI_NONE, mode, nullptr, 0};
  g.rope = &ra;
  g.norm = &norm;
  return run_gemm(g, as_stream(stream));
}

}  // namespace bi

extern "C" bi_status bi_qkv_rope_kv_write(const void* x, int64_t T, int64_t K, const void* wqkv, int Hq, int Hkv,
                                          int hd, const int32_t* row_seq, const int32_t* row_pos,
                                          const float* rope_table, int64_t max_pos, const int32_t* block_table,
                                          int64_t max_blocks_per_seq, int64_t n_blocks, void* q_out, void* k_cache,
                                          void* v_cache, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(Hq > 0 && Hkv > 0 && Hq % Hkv == 0, "bad heads");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  BI_REQUIRE(max_pos > 0 && max_blocks_per_seq > 0 && n_blocks > 0, "bad table / cache shape");
  return gemm_qkv_rope(x, T, K, wqkv, (int64_t)(Hq + 2 * Hkv) * hd, row_seq, row_pos, rope_table, max_pos,
                       block_table, max_blocks_per_seq, n_blocks, q_out, k_cache, v_cache, Hq, Hkv, hd, mode, stream);
}
