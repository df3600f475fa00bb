// FP8 KV cache: one quantising write path and one dequantise-and-gather read
// path shared by prefill, decode and the training recompute.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §4.2 ("FP8 KV cache: keep
// FP8 storage, unify the read path"): the cache is stored in FP8; decode gives
// up its own FP8-reading kernel and goes through prefill's path: dequantise and
// gather the KV it needs into a bf16 workspace sized by model limits, then run
// the same attention.  Training writes a private cache the same way, so K and
// V make the same FP8 round trip.
//
// Readings: e4m3 codes with one power-of-two scale per (token, kv head) vector
// of hd values, for K and for V separately (the smallest power of two s with
// 448 s >= amax, 1 for an all-zero vector); round to nearest even, saturating.
// A code times its scale is exact in bf16, so everything after the gather is
// the bf16 attention unchanged.
#include <cuda_fp8.h>

#include <string>

#include "common.cuh"
#include "fp8.cuh"

namespace bi {

struct KvPieces {
  const int32_t* seq;
  const int32_t* row0;
  const int32_t* pos0;
};

// One warp per (token, kv head, K or V): hd values -> codes and a scale in the token's page slot.
__global__ void __launch_bounds__(256) kv_fp8_write_kernel(const __nv_bfloat16* __restrict__ k,
                                                           const __nv_bfloat16* __restrict__ v, KvPieces pm,
                                                           int64_t max_q_len, int Hkv, int hd,
                                                           const int32_t* __restrict__ block_table, int64_t max_blk,
                                                           int64_t n_blocks, uint8_t* __restrict__ k8,
                                                           uint8_t* __restrict__ v8, float* __restrict__ ks,
                                                           float* __restrict__ vs, int* status) {
  pdl_trigger();
  pdl_wait();
  const int p = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);  // (token in piece, kv head, K|V)
  const int i = item / (2 * Hkv), kh = (item / 2) % Hkv, which = item & 1;
  const int row0 = pm.row0[p];
  if (i >= max_q_len || i >= pm.row0[p + 1] - row0) return;
  const int64_t row = row0 + i, pos = (int64_t)pm.pos0[p] + i;
  const int seq = pm.seq[p];
  const int32_t blk = (pos >= 0 && pos / 64 < max_blk) ? block_table[(int64_t)seq * max_blk + pos / 64] : -1;
  if (blk < 0 || blk >= n_blocks) {
    if (lane == 0) report(status, DEV_BAD_INDEX);
    return;
  }
  const __nv_bfloat16* src = (which ? v : k) + (row * Hkv + kh) * hd;
  const int per = hd / 32;  // 2 or 4 values per lane
  float x[4];
  float m = 0.f;
  for (int u = 0; u < per; ++u) {
    x[u] = bf2f(src[lane * per + u]);
    m = fmaxf(m, fabsf(x[u]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int e = fp8_scale_exp(m);
  const int64_t slot = ((int64_t)blk * Hkv + kh) * 64 + pos % 64;
  uint8_t* dst = (which ? v8 : k8) + slot * hd;
  for (int u = 0; u < per; ++u)
    dst[lane * per + u] = (uint8_t)fp8_code(x[u], e);
  if (lane == 0) (which ? vs : ks)[slot] = ldexpf(1.f, e);
}

// One CTA per (piece, logical page): every kv head's K and V page dequantised
// into the workspace page piece * max_blk + page; the workspace block table row
// of the piece lists them (-1 past the piece's last position).
__global__ void __launch_bounds__(256) kv_fp8_gather_kernel(const uint8_t* __restrict__ k8,
                                                            const uint8_t* __restrict__ v8,
                                                            const float* __restrict__ ks,
                                                            const float* __restrict__ vs, int64_t n_blocks,
                                                            KvPieces pm, int Hkv, int hd,
                                                            const int32_t* __restrict__ block_table, int64_t max_blk,
                                                            int64_t ws_blk, __nv_bfloat16* __restrict__ kw,
                                                            __nv_bfloat16* __restrict__ vw, int32_t* __restrict__ wbt,
                                                            int* status) {
  pdl_trigger();
  pdl_wait();
  const int p = blockIdx.y;
  const int64_t l = blockIdx.x;
  const int n_tok = pm.row0[p + 1] - pm.row0[p];
  const int64_t ctx = (int64_t)pm.pos0[p] + n_tok;  // positions 0 .. ctx-1 are read
  const int64_t wpage = (int64_t)p * ws_blk + l;
  const bool live = n_tok > 0 && l * 64 < ctx && l < max_blk;
  if (threadIdx.x == 0) wbt[(int64_t)p * ws_blk + l] = live ? (int32_t)wpage : -1;
  if (!live) return;
  const int32_t blk = block_table[(int64_t)pm.seq[p] * max_blk + l];
  if (blk < 0 || blk >= n_blocks) {
    if (threadIdx.x == 0) report(status, DEV_BAD_INDEX);
    return;
  }
  const int64_t n = (int64_t)Hkv * 64 * hd;  // one page of one of K / V
  // 16 codes (one 16-byte load, one row: hd is a multiple of 16) per thread and step
  for (int64_t e = (int64_t)threadIdx.x * 16; e < 2 * n; e += 16 * blockDim.x) {
    const int which = e >= n;
    const int64_t off = which ? e - n : e;
    const int64_t slot = off / hd;  // (kv head, slot in page)
    const uint8_t* src = (which ? v8 : k8) + (int64_t)blk * n + off;
    const float sc = (which ? vs : ks)[(int64_t)blk * Hkv * 64 + slot];
    const uint4 raw = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t packed[8];
#pragma unroll
    for (int u = 0; u < 16; u += 2) {
      float f[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t code = (w[(u + t) >> 2] >> (8 * ((u + t) & 3))) & 0xffu;
        const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
        // code x power-of-two scale is exact, so the bf16 rounding is exact too
        f[t] = __fmul_rn(__half2float(__half(hr)), sc);
      }
      packed[u / 2] = pack_bf16x2(f[0], f[1]);
    }
    uint4* dst = reinterpret_cast<uint4*>((which ? vw : kw) + wpage * n + off);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}

}  // namespace bi

extern "C" {

bi_status bi_kv_fp8_write(const void* k, const void* v, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                          const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hkv, int hd,
                          const int32_t* block_table, int64_t max_blocks_per_seq, int64_t n_blocks, void* k_cache8,
                          void* v_cache8, float* k_scale, float* v_scale, void* stream) {
  using namespace bi;
  BI_REQUIRE(T >= 0 && P >= 0, "bad shape");
  if (T == 0 || P == 0) return BI_OK;
  BI_REQUIRE(k && v && piece_seq && piece_row0 && piece_pos0 && block_table && k_cache8 && v_cache8 && k_scale &&
                 v_scale,
             "null pointer");
  BI_REQUIRE_SHAPE(hd == 64 || hd == 128, "head_dim must be 64 or 128");
  BI_REQUIRE(Hkv > 0 && max_q_len > 0 && P <= 65535 && max_blocks_per_seq > 0 && n_blocks > 0, "bad arguments");
  const int64_t items = max_q_len * Hkv * 2;
  BI_REQUIRE(cdiv(items, 8) <= 0x7fffffff, "too many rows");
  return launched(launch_pdl(kv_fp8_write_kernel, dim3((unsigned)cdiv(items, 8), (unsigned)P), dim3(256), 0,
                             as_stream(stream), static_cast<const __nv_bfloat16*>(k),
                             static_cast<const __nv_bfloat16*>(v), KvPieces{piece_seq, piece_row0, piece_pos0},
                             max_q_len, Hkv, hd, block_table, max_blocks_per_seq, n_blocks,
                             static_cast<uint8_t*>(k_cache8), static_cast<uint8_t*>(v_cache8), k_scale, v_scale,
                             device_status_ptr()),
                  "bi_kv_fp8_write");
}

}  // extern "C"

namespace bi {
// Gather into workspace pages p * ws_blk + l (ws_blk >= the pages any piece needs).
bi_status kv_fp8_gather_to(const void* k_cache8, const void* v_cache8, const float* k_scale, const float* v_scale,
                           int64_t n_blocks, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int Hkv, int hd, const int32_t* block_table,
                           int64_t max_blocks_per_seq, int64_t ws_blk, void* k_ws, void* v_ws, int32_t* ws_block_table,
                           cudaStream_t st) {
  if (P == 0) return BI_OK;
  BI_REQUIRE(P <= 65535 && ws_blk > 0 && ws_blk <= 0x7fffffff, "bad pieces / workspace pages");
  return launched(launch_pdl(kv_fp8_gather_kernel, dim3((unsigned)ws_blk, (unsigned)P), dim3(256), 0, st,
                             static_cast<const uint8_t*>(k_cache8), static_cast<const uint8_t*>(v_cache8), k_scale,
                             v_scale, n_blocks, KvPieces{piece_seq, piece_row0, piece_pos0}, Hkv, hd, block_table,
                             max_blocks_per_seq, ws_blk, static_cast<__nv_bfloat16*>(k_ws),
                             static_cast<__nv_bfloat16*>(v_ws), ws_block_table, device_status_ptr()),
                  "bi_kv_fp8_gather");
}
}  // namespace bi

extern "C" {

bi_status bi_kv_fp8_gather(const void* k_cache8, const void* v_cache8, const float* k_scale, const float* v_scale,
                           int64_t n_blocks, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int Hkv, int hd, const int32_t* block_table,
                           int64_t max_blocks_per_seq, void* k_ws, void* v_ws, int32_t* ws_block_table,
                           void* stream) {
  using namespace bi;
  BI_REQUIRE(P >= 0, "bad shape");
  if (P == 0) return BI_OK;
  BI_REQUIRE(k_cache8 && v_cache8 && k_scale && v_scale && piece_seq && piece_row0 && piece_pos0 && block_table &&
                 k_ws && v_ws && ws_block_table,
             "null pointer");
  BI_REQUIRE_SHAPE(hd == 64 || hd == 128, "head_dim must be 64 or 128");
  BI_REQUIRE(Hkv > 0 && P <= 65535 && max_blocks_per_seq > 0 && max_blocks_per_seq <= 0x7fffffff && n_blocks > 0,
             "bad arguments");
  BI_REQUIRE(aligned16(k_ws) && aligned16(v_ws) && aligned16(k_cache8) && aligned16(v_cache8),
             "workspace and cache pages must be 16-byte aligned");
  return kv_fp8_gather_to(k_cache8, v_cache8, k_scale, v_scale, n_blocks, piece_seq, piece_row0, piece_pos0, P, Hkv,
                          hd, block_table, max_blocks_per_seq, max_blocks_per_seq, k_ws, v_ws, ws_block_table,
                          as_stream(stream));
}

}  // extern "C"
