// Model drivers: chunked packed prefill (rollout prompts, training recompute) and decode.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §3.1 (training forward
// calls the inference kernels: "inference kernels define the values") and §2
// (phase consistency: a token gets the same result in prefill and in decode).
// Both drivers below run one layer stack, `run_pass`, over a set of rows; the
// only difference between prefill and decode is how the rows' metadata is
// produced.  §4.6 (CUDA Graph): the decode step reads nothing back to the host
// and its workspace is sized by limits, so it can be captured and replayed.
#include <algorithm>
#include <cmath>
#include <vector>

#include "common.cuh"

struct bi_model {
  bi_model_config cfg;
  const void* embed;
  const void* final_norm;
  const void* lm_head;
  float* rope_table;
  std::vector<bi_layer_weights> layers;
  void* dump = nullptr;       // optional per-layer residual dump (bf16 [n_layers + 2, dump_rows, d])
  int64_t dump_rows = 0;
};

namespace bi {

constexpr int kMaxPiecesPerPass = 128;

struct PassMeta {
  int n_pieces, n_rows, n_logit;
  int seq[kMaxPiecesPerPass];
  int row0[kMaxPiecesPerPass + 1];
  int pos0[kMaxPiecesPerPass];
  int tok0[kMaxPiecesPerPass];
  int lfirst[kMaxPiecesPerPass];
  int loff[kMaxPiecesPerPass + 1];
};

struct DevMeta {
  int32_t* piece_seq;
  int32_t* piece_row0;
  int32_t* piece_pos0;
  int32_t* ids;        // token id of every pass row
  int32_t* logit_src;  // pass row of each logit row
  int32_t* logit_dst;  // call row of each logit row
  int32_t* logit_tgt;  // target id of each logit row (or -1)
  int32_t* row_seq;    // sequence of every pass row
  int32_t* row_pos;    // absolute position of every pass row
};

__global__ void pass_meta_kernel(const PassMeta pm, const int32_t* __restrict__ tokens,
                                 const int32_t* __restrict__ targets, DevMeta dm) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x == 0) {
    for (int p = threadIdx.x; p < pm.n_pieces; p += blockDim.x) {
      dm.piece_seq[p] = pm.seq[p];
      dm.piece_row0[p] = pm.row0[p];
      dm.piece_pos0[p] = pm.pos0[p];
    }
    if (threadIdx.x == 0) dm.piece_row0[pm.n_pieces] = pm.row0[pm.n_pieces];
  }
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= pm.n_rows) return;
  int lo = 0, hi = pm.n_pieces - 1;  // last piece with row0 <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (pm.row0[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int p = lo;
  const int i = r - pm.row0[p];
  const int tok = pm.tok0[p] + i;
  dm.ids[r] = tokens[tok];
  dm.row_seq[r] = pm.seq[p];
  dm.row_pos[r] = pm.pos0[p] + i;
  if (i >= pm.lfirst[p]) {
    const int j = pm.loff[p] + (i - pm.lfirst[p]);
    dm.logit_src[j] = r;
    dm.logit_dst[j] = tok;
    dm.logit_tgt[j] = targets ? targets[tok] : -1;
  }
}

// Decode step metadata (one piece per sequence, one row each) fused with the
// embedding gather of that row.
__global__ void decode_embed_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ pos, int B,
                                    DevMeta dm, const __nv_bfloat16* __restrict__ table, int64_t V, int64_t d,
                                    __nv_bfloat16* __restrict__ h, int* status) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int32_t id = tokens[b];
  if (threadIdx.x == 0) {
    if (b == 0) dm.piece_row0[B] = B;
    dm.piece_seq[b] = b;
    dm.piece_row0[b] = b;
    dm.piece_pos0[b] = pos[b];
    dm.ids[b] = id;
    dm.row_seq[b] = b;
    dm.row_pos[b] = pos[b];
    dm.logit_src[b] = b;
    dm.logit_dst[b] = b;
    dm.logit_tgt[b] = -1;
  }
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) report(status, DEV_BAD_INDEX);
  const uint4* src = reinterpret_cast<const uint4*>(table + (int64_t)(ok ? id : 0) * d);
  uint4* dst = reinterpret_cast<uint4*>(h + (int64_t)b * d);
  for (int64_t v = threadIdx.x; v < d / 8; v += blockDim.x) dst[v] = ok ? src[v] : make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------- workspace plan
// Passes of at most this many rows (decode steps) fold each RMSNorm into the
// GEMM after it (gemm_norm, gemm_qkv_rope_norm), which writes the new residual
// rows to the other of two buffers; longer passes run the norm kernel in place.
constexpr int64_t kFoldRows = 16;
struct FwdLayout {
  size_t piece_seq, piece_row0, piece_pos0, ids, logit_src, logit_dst, logit_tgt, row_seq, row_pos;
  size_t h, h2, x, q, ao, tmp, act, attn_ws, xsel, logits, gemm_ws;
  size_t attn_ws_bytes, gemm_ws_bytes, lp_ws_bytes;
  // fp8 only: bf16 qkv and gate/up outputs, activation codes and scales
  size_t qkv, g13, qa, sa;
  size_t total;
};

static FwdLayout plan_layout(const bi_model_config& c, int64_t Tm, int64_t Pm, int64_t max_ctx, int64_t Rm, int mode) {
  FwdLayout L{};
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t r = off;
    off += (n + 255) / 256 * 256;
    return r;
  };
  const int64_t nqkv = (c.n_heads_q + 2 * c.n_heads_kv) * c.head_dim;
  const int64_t hq = c.n_heads_q * c.head_dim;
  L.piece_seq = take(Pm * 4);
  L.piece_row0 = take((Pm + 1) * 4);
  L.piece_pos0 = take(Pm * 4);
  L.ids = take(Tm * 4);
  L.logit_src = take(std::max(Tm, Rm) * 4);
  L.logit_dst = take(std::max(Tm, Rm) * 4);
  L.logit_tgt = take(std::max(Tm, Rm) * 4);
  L.row_seq = take(Tm * 4);
  L.row_pos = take(Tm * 4);
  L.h = take(Tm * c.d * 2);
  // passes of at most kFoldRows rows alternate the residual stream between h and h2
  L.h2 = take(std::min<int64_t>(Tm, kFoldRows) * c.d * 2);
  L.x = take(Tm * c.d * 2);

  L.q = take(Tm * hq * 2);
  L.ao = take(Tm * hq * 2);
  L.tmp = take(Tm * c.d * 2);
  L.act = take(Tm * c.ffn * 2);
  L.attn_ws_bytes = bi_attention_workspace_size(Tm, (int)c.n_heads_q, (int)c.head_dim, max_ctx, (int)c.kv_split);
  L.attn_ws = take(L.attn_ws_bytes);
  L.xsel = take(Rm * c.d * 2);
  // fused lm_head + log-softmax: per-(row, vocab tile) records, no logits
  const size_t head_bytes = std::max(lm_head_partial_bytes(Rm, c.vocab, c.d, mode),
                                     lm_head_partial_bytes(std::min<int64_t>(Rm, 128), c.vocab, c.d, mode));
  L.logits = take(head_bytes);
  L.lp_ws_bytes = head_bytes;
  size_t g = 0;
  if (mode == BI_FAST) {
    const int64_t m = std::min<int64_t>(std::max(Tm, Rm), 128);
    g = std::max(g, bi_gemm_workspace_size(m, nqkv, c.d, BI_EPI_NONE, mode));
    g = std::max(g, bi_gemm_workspace_size(m, c.d, hq, BI_EPI_NONE, mode));
    g = std::max(g, bi_gemm_workspace_size(m, 2 * c.ffn, c.d, BI_EPI_SWIGLU, mode));
    g = std::max(g, bi_gemm_workspace_size(m, c.d, c.ffn, BI_EPI_NONE, mode));
  }
  L.gemm_ws_bytes = g;
  L.gemm_ws = take(g);
  if (c.fp8) {
    const int64_t kmax = std::max(std::max(c.d, hq), c.ffn);
    L.qkv = take(Tm * nqkv * 2);
    L.g13 = take(Tm * 2 * c.ffn * 2);
    L.qa = take(Tm * kmax);
    L.sa = take(Tm * (kmax / 128) * 4);
  }
  L.total = off + 256;
  return L;
}

template <typename T>
static T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

struct PassShape {
  int64_t rows, pieces, max_q_len, max_ctx, n_logit;
  bool embedded;  // the embedding rows are already in the residual buffer
};

// One layer pass of a prefill call: the pieces it holds and its shape.
struct PassPlan {
  PassMeta pm;
  PassShape ps;
};

// The pass schedule of a prefill call (host only).  Pieces in chunk-major order
// (every sequence's chunk 0, then chunk 1, ...), each at most `chunk` rows;
// passes take pieces in that order up to max_tokens rows and Pm pieces; a piece
// larger than a whole pass is split.  logit_from (or NULL: every row) gives each
// sequence's first row with logits.
static std::vector<PassPlan> plan_prefill(const int64_t* cu_seqlens, const int64_t* start_pos,
                                          const int64_t* logit_from, int64_t B, int64_t chunk, int64_t max_tokens,
                                          int64_t Pm) {
  struct Piece { int64_t seq, start, len; };
  std::vector<Piece> pieces;
  int64_t max_len = 0;
  for (int64_t b = 0; b < B; ++b) max_len = std::max(max_len, cu_seqlens[b + 1] - cu_seqlens[b]);
  for (int64_t c0 = 0; c0 < max_len; c0 += chunk)
    for (int64_t b = 0; b < B; ++b) {
      const int64_t n = cu_seqlens[b + 1] - cu_seqlens[b];
      if (c0 < n) pieces.push_back({b, c0, std::min(chunk, n - c0)});
    }
  std::vector<PassPlan> plan;
  size_t i = 0;
  while (i < pieces.size()) {
    PassMeta pm{};
    PassShape ps{};
    int64_t rows = 0, nlog = 0;
    int np = 0;
    while (i < pieces.size() && np < Pm) {
      const Piece& pc = pieces[i];
      int64_t len = pc.len;
      if (rows + len > max_tokens) {
        if (rows > 0) break;
        len = max_tokens;  // a single piece larger than the pass limit: split it
      }
      const int64_t lf_call = logit_from ? logit_from[pc.seq] : 0;
      const int64_t lfirst = std::min(std::max<int64_t>(lf_call - pc.start, 0), len);
      pm.seq[np] = (int)pc.seq;
      pm.row0[np] = (int)rows;
      pm.pos0[np] = (int)(start_pos[pc.seq] + pc.start);
      pm.tok0[np] = (int)(cu_seqlens[pc.seq] + pc.start);
      pm.lfirst[np] = (int)lfirst;
      pm.loff[np] = (int)nlog;
      nlog += len - lfirst;
      rows += len;
      ps.max_q_len = std::max(ps.max_q_len, len);
      ps.max_ctx = std::max(ps.max_ctx, start_pos[pc.seq] + pc.start + len);
      ++np;
      if (len < pieces[i].len) {
        pieces[i].start += len;
        pieces[i].len -= len;
      } else {
        ++i;
      }
    }
    pm.n_pieces = np;
    pm.n_rows = (int)rows;
    pm.n_logit = (int)nlog;
    pm.row0[np] = (int)rows;
    pm.loff[np] = (int)nlog;
    ps.rows = rows;
    ps.pieces = np;
    ps.n_logit = nlog;
    plan.push_back({pm, ps});
  }
  return plan;
}

// The layer stack over the rows of one pass (identical for prefill and decode).
static bi_status run_pass(bi_model* m, void* ws, const FwdLayout& L, const PassShape& ps, int64_t Rm,
                          const int32_t* block_table, int64_t max_blk, void* k_cache, void* v_cache,
                          int64_t n_blocks, bool greedy, float* logprob_out, int32_t* sampled_out, int mode,
                          void* stream) {
  const bi_model_config& c = m->cfg;
  const int64_t T = ps.rows;
  const int64_t nqkv = (c.n_heads_q + 2 * c.n_heads_kv) * c.head_dim;
  const int64_t hq = c.n_heads_q * c.head_dim;
  const int Hq = (int)c.n_heads_q, Hkv = (int)c.n_heads_kv, hd = (int)c.head_dim;
  const float scale = 1.0f / std::sqrt((float)c.head_dim);
  auto* piece_seq = at<int32_t>(ws, L.piece_seq);
  auto* piece_row0 = at<int32_t>(ws, L.piece_row0);
  auto* piece_pos0 = at<int32_t>(ws, L.piece_pos0);
  void* h = at<void>(ws, L.h);
  void* x = at<void>(ws, L.x);

  void* q = at<void>(ws, L.q);
  void* ao = at<void>(ws, L.ao);
  void* tmp = at<void>(ws, L.tmp);
  void* act = at<void>(ws, L.act);
  void* gws = L.gemm_ws_bytes ? at<void>(ws, L.gemm_ws) : nullptr;
  // bf16: [n_blocks, Hkv, 64, hd] per layer; fp8: codes [n_blocks, Hkv, 64, hd] then fp32 scales [n_blocks, Hkv, 64]
  const size_t layer_cache = (size_t)n_blocks * Hkv * 64 * (c.fp8 ? hd + 4 : hd * 2);
  const size_t layer_codes = (size_t)n_blocks * Hkv * 64 * hd;
  const cudaStream_t cst = as_stream(stream);

  const bool dumping = m->dump && T <= m->dump_rows;
  const size_t slot_bytes = (size_t)m->dump_rows * c.d * 2;
  auto dump_slot = [&](int64_t l) { return static_cast<uint8_t*>(m->dump) + l * slot_bytes; };
  auto dump_copy = [&](int64_t l, const void* src) -> bi_status {
    if (!dumping) return BI_OK;
    cudaMemcpyAsync(dump_slot(l), src, (size_t)T * c.d * 2, cudaMemcpyDeviceToDevice, as_stream(stream));
    return check_launch("dump copy");
  };

  if (!ps.embedded) BI_TRY(bi_embed(at<int32_t>(ws, L.ids), T, m->embed, c.vocab, c.d, h, stream));
  BI_TRY(dump_copy(0, h));
  // bf16 passes of at most kFoldRows rows (decode steps) fold each norm into
  // the next GEMM; the residual stream then alternates between h and h2 (res
  // is the current one), every row keeping the norm kernel's arithmetic
  const bool fold = !c.fp8 && !dumping && T <= kFoldRows;
  void* res = h;
  void* h2 = at<void>(ws, L.h2);
  auto other = [&](void* r) { return r == h ? h2 : h; };
  if (c.fp8)
    BI_TRY(rmsnorm_fp8_rows(h, nullptr, m->layers[0].attn_norm, nullptr, at<uint8_t>(ws, L.qa), at<float>(ws, L.sa),
                            T, c.d, c.eps, stream));
  else if (!fold)
    BI_TRY(bi_rmsnorm(h, nullptr, m->layers[0].attn_norm, x, T, c.d, c.eps, mode, stream));
  for (int64_t li = 0; li < c.n_layers; ++li) {
    const bi_layer_weights& lw = m->layers[li];
    void* kc = static_cast<uint8_t*>(k_cache) + li * layer_cache;
    void* vc = static_cast<uint8_t*>(v_cache) + li * layer_cache;
    if (c.fp8) {
      // block-FP8 W8A8 layer; K and V make the FP8 round trip through the one read path.
      // qa/sa hold the quantised input rows of the next GEMM (written by the
      // preceding norm, or by the quantiser / SwiGLU in front of it).
      auto* qa = at<uint8_t>(ws, L.qa);
      auto* sa = at<float>(ws, L.sa);
      void* qkv = at<void>(ws, L.qkv);
      float* ks = reinterpret_cast<float*>(static_cast<uint8_t*>(kc) + layer_codes);
      float* vs = reinterpret_cast<float*>(static_cast<uint8_t*>(vc) + layer_codes);
      BI_TRY(bi_gemm_fp8(qa, sa, T, c.d, lw.wqkv8, lw.wqkv_s, nqkv, qkv, BI_DTYPE_BF16, mode, stream));
      BI_TRY(rope_kv_write_fp8(qkv, T, at<int32_t>(ws, L.row_seq), at<int32_t>(ws, L.row_pos), Hq, Hkv, hd,
                               m->rope_table, c.max_pos, block_table, max_blk, n_blocks, q, kc, ks, vc, vs, cst));
      // attention reads the FP8 pages directly (bit-equal to gather + bf16 attention)
      // and its split merge writes the quantised output rows for the O projection
      BI_TRY(bi_attention_fp8(q, T, piece_seq, piece_row0, piece_pos0, ps.pieces, ps.max_q_len, Hq, Hkv, hd, kc, vc,
                              ks, vs, block_table, max_blk, n_blocks, ps.max_ctx, (int)c.kv_split, scale,
                              at<void>(ws, L.attn_ws), L.attn_ws_bytes, nullptr, qa, sa, mode, stream));
      BI_TRY(bi_gemm_fp8(qa, sa, T, hq, lw.wo8, lw.wo_s, c.d, tmp, BI_DTYPE_BF16, mode, stream));
      BI_TRY(rmsnorm_fp8_rows(tmp, h, lw.ffn_norm, nullptr, qa, sa, T, c.d, c.eps, stream));
      BI_TRY(bi_gemm_fp8(qa, sa, T, c.d, lw.w138, lw.w13_s, 2 * c.ffn, at<void>(ws, L.g13), BI_DTYPE_BF16, mode,
                         stream));
      BI_TRY(swiglu_fp8(at<void>(ws, L.g13), T, c.ffn, qa, sa, cst));
      BI_TRY(bi_gemm_fp8(qa, sa, T, c.ffn, lw.w28, lw.w2_s, c.d, tmp, BI_DTYPE_BF16, mode, stream));
      if (li + 1 < c.n_layers) {
        BI_TRY(rmsnorm_fp8_rows(tmp, h, m->layers[li + 1].attn_norm, nullptr, qa, sa, T, c.d, c.eps, stream));
        BI_TRY(dump_copy(li + 1, h));
      }
      continue;
    }
    // QKV projection with RoPE and the paged K/V write fused into its epilogue
    if (fold) {
      // the layer's input norm: of the embeddings (layer 0), else of the last down projection + residual
      const NormIn n = li == 0 ? NormIn{h, nullptr, nullptr, lw.attn_norm, c.eps, x}
                               : NormIn{tmp, res, other(res), lw.attn_norm, c.eps, x};
      if (li > 0) res = other(res);
      BI_TRY(gemm_qkv_rope_norm(n, T, c.d, lw.wqkv, nqkv, at<int32_t>(ws, L.row_seq), at<int32_t>(ws, L.row_pos),
                                m->rope_table, c.max_pos, block_table, max_blk, n_blocks, q, kc, vc, Hq, Hkv, hd,
                                mode, stream));
    } else {
      BI_TRY(gemm_qkv_rope(x, T, c.d, lw.wqkv, nqkv, at<int32_t>(ws, L.row_seq), at<int32_t>(ws, L.row_pos),
                           m->rope_table, c.max_pos, block_table, max_blk, n_blocks, q, kc, vc, Hq, Hkv, hd, mode,
                           stream));
    }
    BI_TRY(bi_attention(q, T, piece_seq, piece_row0, piece_pos0, ps.pieces, ps.max_q_len, Hq, Hkv, hd, kc, vc,
                        block_table, max_blk, n_blocks, ps.max_ctx, (int)c.kv_split, scale, at<void>(ws, L.attn_ws),
                        L.attn_ws_bytes, ao, mode, stream));
    BI_TRY(bi_gemm(ao, T, hq, lw.wo, c.d, tmp, BI_DTYPE_BF16, BI_EPI_NONE, mode, gws, L.gemm_ws_bytes, stream));
    if (fold) {
      const NormIn n{tmp, res, other(res), lw.ffn_norm, c.eps, x};
      res = other(res);
      BI_TRY(gemm_norm(n, T, c.d, lw.w13, 2 * c.ffn, act, BI_EPI_SWIGLU, mode, gws, L.gemm_ws_bytes, stream));
    } else {
      BI_TRY(bi_rmsnorm(tmp, h, lw.ffn_norm, x, T, c.d, c.eps, mode, stream));
      BI_TRY(bi_gemm(x, T, c.d, lw.w13, 2 * c.ffn, act, BI_DTYPE_BF16, BI_EPI_SWIGLU, mode, gws, L.gemm_ws_bytes,
                     stream));
    }
    BI_TRY(bi_gemm(act, T, c.ffn, lw.w2, c.d, tmp, BI_DTYPE_BF16, BI_EPI_NONE, mode, gws, L.gemm_ws_bytes, stream));
    if (li + 1 < c.n_layers && !fold) {
      BI_TRY(bi_rmsnorm(tmp, h, m->layers[li + 1].attn_norm, x, T, c.d, c.eps, mode, stream));
      BI_TRY(dump_copy(li + 1, h));
    }
  }
  if (dumping) {
    // residual after the last layer and the final-norm output of every row
    BI_TRY(dump_copy(c.n_layers, h));
    BI_TRY(bi_rmsnorm(tmp, dump_slot(c.n_layers), m->final_norm, dump_slot(c.n_layers + 1), T, c.d, c.eps, mode,
                      stream));
  }
  // final residual add + norm only on the rows whose logits are wanted
  const cudaStream_t st = as_stream(stream);
  for (int64_t r0 = 0; r0 < ps.n_logit; r0 += Rm) {
    const int64_t R = std::min(Rm, ps.n_logit - r0);
    const int32_t* src = at<int32_t>(ws, L.logit_src) + r0;
    void* xsel = at<void>(ws, L.xsel);
    // rows src[j] of (down-proj out + residual) -> final norm -> compact row j
    BI_TRY(rmsnorm_rows(tmp, res, m->final_norm, xsel, R, c.d, c.eps, src, stream));
    // lm_head + log-softmax + gather fused; results land at the call's row index
    const int32_t* tgt = greedy ? nullptr : at<int32_t>(ws, L.logit_tgt) + r0;
    BI_TRY(lm_head_logprob_to(xsel, R, c.d, m->lm_head, c.vocab, tgt, logprob_out, sampled_out,
                              at<int32_t>(ws, L.logit_dst) + r0, mode, at<void>(ws, L.logits), L.lp_ws_bytes, stream));
  }
  (void)st;
  return BI_OK;
}

static bi_status validate_cfg(const bi_model_config* c) {
  BI_REQUIRE(c, "null config");
  BI_REQUIRE(c->n_layers > 0 && c->d > 0 && c->n_heads_q > 0 && c->n_heads_kv > 0 && c->head_dim > 0 && c->ffn > 0 &&
                 c->vocab > 0 && c->max_pos > 0,
             "non-positive config field");
  BI_REQUIRE(c->n_heads_q % c->n_heads_kv == 0, "n_heads_q must be a multiple of n_heads_kv");
  BI_REQUIRE_SHAPE(c->kv_block == 64, "kv_block must be 64");
  BI_REQUIRE(c->kv_split >= 64 && c->kv_split % 64 == 0, "kv_split must be a positive multiple of 64");
  BI_REQUIRE_SHAPE(c->head_dim == 64 || c->head_dim == 128, "head_dim must be 64 or 128");
  BI_REQUIRE_SHAPE(c->d % 64 == 0 && c->ffn % 64 == 0 && (c->n_heads_q * c->head_dim) % 64 == 0,
                   "d, ffn and Hq*hd must be multiples of 64");
  BI_REQUIRE_SHAPE(c->vocab % 8 == 0, "vocab must be a multiple of 8");
  BI_REQUIRE_SHAPE(64 % (c->n_heads_q / c->n_heads_kv) == 0, "Hq/Hkv must divide 64");
  BI_REQUIRE(c->eps > 0.f, "eps must be positive");
  BI_REQUIRE(c->fp8 == 0 || c->fp8 == 1, "fp8 must be 0 or 1");
  if (c->fp8)
    BI_REQUIRE_SHAPE(c->d % 128 == 0 && c->ffn % 128 == 0 && (c->n_heads_q * c->head_dim) % 128 == 0 &&
                         ((c->n_heads_q + 2 * c->n_heads_kv) * c->head_dim) % 128 == 0,
                     "fp8 needs d, ffn, Hq*hd and (Hq + 2 Hkv)*hd multiples of 128");
  return BI_OK;
}

}  // namespace bi

extern "C" {

bi_status bi_model_create(const bi_model_config* cfg, const bi_weights* w, void* stream, bi_model** out) {
  using namespace bi;
  BI_TRY(validate_cfg(cfg));
  BI_REQUIRE(w && out && w->embed && w->final_norm && w->lm_head && w->layers && w->rope_table, "null pointer");
  for (int64_t i = 0; i < cfg->n_layers; ++i) {
    const bi_layer_weights& l = w->layers[i];
    BI_REQUIRE(l.attn_norm && l.wqkv && l.wo && l.ffn_norm && l.w13 && l.w2, "null layer weight");
    if (cfg->fp8)
      BI_REQUIRE(l.wqkv8 && l.wqkv_s && l.wo8 && l.wo_s && l.w138 && l.w13_s && l.w28 && l.w2_s,
                 "fp8 model: null FP8 layer weight");
  }
  BI_TRY(bi_rope_table(w->rope_table, cfg->max_pos, (int)cfg->head_dim, (double)cfg->rope_theta, stream));
  bi_model* m = new bi_model;
  m->cfg = *cfg;
  m->embed = w->embed;
  m->final_norm = w->final_norm;
  m->lm_head = w->lm_head;
  m->rope_table = w->rope_table;
  m->layers.assign(w->layers, w->layers + cfg->n_layers);
  *out = m;
  return BI_OK;
}

void bi_model_destroy(bi_model* m) { delete m; }

bi_status bi_model_set_dump(bi_model* m, void* dump, int64_t max_rows) {
  BI_REQUIRE(m, "null model");
  BI_REQUIRE(!dump || (max_rows > 0 && bi::aligned16(dump)), "dump needs max_rows > 0 and 16-byte alignment");
  m->dump = dump;
  m->dump_rows = dump ? max_rows : 0;
  return BI_OK;
}

size_t bi_kv_cache_bytes(const bi_model_config* cfg, int64_t n_blocks) {
  if (!cfg || n_blocks <= 0) return 0;
  const int64_t per_slot = cfg->fp8 ? cfg->head_dim + 4 : cfg->head_dim * 2;  // fp8: codes + one fp32 scale
  return (size_t)cfg->n_layers * n_blocks * cfg->n_heads_kv * 64 * per_slot;
}

size_t bi_forward_workspace_size(const bi_model_config* cfg, int64_t max_tokens, int64_t max_pieces, int64_t max_ctx,
                                 int64_t max_logit_rows, int mode) {
  if (!cfg || max_tokens <= 0 || max_pieces <= 0 || max_ctx <= 0 || max_logit_rows <= 0) return 0;
  return bi::plan_layout(*cfg, max_tokens, max_pieces, max_ctx, max_logit_rows, mode).total;
}

bi_status bi_forward_prefill(bi_model* m, const int32_t* tokens, const int32_t* target_ids, const int64_t* cu_seqlens,
                             const int64_t* start_pos, const int64_t* logit_from, int64_t B, int64_t chunk,
                             const int32_t* block_table, int64_t max_blocks_per_seq, void* k_cache, void* v_cache,
                             int64_t n_blocks, float* logprob_out, int32_t* sampled_out, void* workspace,
                             size_t ws_bytes, int64_t max_tokens, int64_t max_ctx, int64_t max_logit_rows, int mode,
                             void* stream) {
  using namespace bi;
  BI_REQUIRE(m && cu_seqlens && start_pos, "null model or metadata");
  BI_REQUIRE(B >= 0, "B < 0");
  if (B == 0) return BI_OK;
  BI_REQUIRE(tokens && block_table && k_cache && v_cache && logprob_out && workspace, "null pointer");
  BI_REQUIRE(chunk > 0 && max_tokens > 0 && max_logit_rows > 0 && max_ctx > 0, "non-positive limit");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  const bi_model_config& c = m->cfg;
  const int64_t Pm = std::min<int64_t>(kMaxPiecesPerPass, std::max<int64_t>(B, 1));
  const FwdLayout L = plan_layout(c, max_tokens, Pm, max_ctx, max_logit_rows, mode);
  BI_REQUIRE(ws_bytes >= L.total, "forward workspace too small (bi_forward_workspace_size with max_pieces >= min(B, 128))");
  BI_REQUIRE(cu_seqlens[0] == 0, "cu_seqlens[0] must be 0");
  for (int64_t b = 0; b < B; ++b) {
    BI_REQUIRE(cu_seqlens[b + 1] >= cu_seqlens[b], "cu_seqlens must be non-decreasing");
    BI_REQUIRE(start_pos[b] >= 0, "start_pos < 0");
    const int64_t end = start_pos[b] + cu_seqlens[b + 1] - cu_seqlens[b];
    BI_REQUIRE(end <= max_ctx && end <= c.max_pos, "sequence longer than max_ctx / max_pos");
    BI_REQUIRE(cdiv(end, 64) <= max_blocks_per_seq, "block table too short for a sequence");
  }
  BI_REQUIRE(cu_seqlens[B] < (1ll << 31), "too many tokens");

  const std::vector<PassPlan> plan = plan_prefill(cu_seqlens, start_pos, logit_from, B, chunk, max_tokens, Pm);
  const cudaStream_t st = as_stream(stream);
  for (const PassPlan& pp : plan) {
    const PassMeta& pm = pp.pm;
    const PassShape& ps = pp.ps;
    const int64_t rows = ps.rows;
    DevMeta dm{at<int32_t>(workspace, L.piece_seq), at<int32_t>(workspace, L.piece_row0),
               at<int32_t>(workspace, L.piece_pos0), at<int32_t>(workspace, L.ids),
               at<int32_t>(workspace, L.logit_src), at<int32_t>(workspace, L.logit_dst),
               at<int32_t>(workspace, L.logit_tgt), at<int32_t>(workspace, L.row_seq),
               at<int32_t>(workspace, L.row_pos)};
    BI_TRY(launched(launch_pdl(pass_meta_kernel, dim3((unsigned)cdiv(std::max<int64_t>(rows, 1), 256)), dim3(256), 0,
                               st, pm, tokens, target_ids, dm),
                    "pass_meta_kernel"));
    BI_TRY(run_pass(m, workspace, L, ps, max_logit_rows, block_table, max_blocks_per_seq, k_cache, v_cache, n_blocks,
                    target_ids == nullptr, logprob_out, sampled_out, mode, stream));
  }
  return BI_OK;
}

int64_t bi_prefill_plan(const int64_t* cu_seqlens, const int64_t* start_pos, const int64_t* logit_from, int64_t B,
                        int64_t chunk, int64_t max_tokens, int64_t* out, int64_t out_rows) {
  using namespace bi;
  if (!cu_seqlens || !start_pos || B < 0 || chunk <= 0 || max_tokens <= 0 || cu_seqlens[0] != 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    if (cu_seqlens[b + 1] < cu_seqlens[b] || start_pos[b] < 0) return -1;
  const int64_t Pm = std::min<int64_t>(kMaxPiecesPerPass, std::max<int64_t>(B, 1));
  const std::vector<PassPlan> plan = plan_prefill(cu_seqlens, start_pos, logit_from, B, chunk, max_tokens, Pm);
  int64_t n = 0;
  for (size_t p = 0; p < plan.size(); ++p) {
    const PassMeta& pm = plan[p].pm;
    for (int k = 0; k < pm.n_pieces; ++k, ++n) {
      if (!out || n >= out_rows) continue;
      int64_t* r = out + n * 8;
      r[0] = (int64_t)p;
      r[1] = pm.seq[k];
      r[2] = pm.row0[k];
      r[3] = pm.row0[k + 1] - pm.row0[k];
      r[4] = pm.pos0[k];
      r[5] = pm.tok0[k];
      r[6] = pm.lfirst[k];
      r[7] = pm.loff[k];
    }
  }
  return n;
}

bi_status bi_forward_decode(bi_model* m, const int32_t* tokens, const int32_t* pos, int64_t B,
                            const int32_t* block_table, int64_t max_blocks_per_seq, void* k_cache, void* v_cache,
                            int64_t n_blocks, int64_t max_ctx, int32_t* sampled_out, float* logprob_out,
                            void* workspace, size_t ws_bytes, int mode, void* stream) {
  using namespace bi;
  BI_REQUIRE(m, "null model");
  BI_REQUIRE(B >= 0, "B < 0");
  if (B == 0) return BI_OK;
  BI_REQUIRE(tokens && pos && block_table && k_cache && v_cache && sampled_out && logprob_out && workspace,
             "null pointer");
  BI_REQUIRE(max_ctx > 0 && max_ctx <= m->cfg.max_pos, "max_ctx must be in (0, max_pos]");
  BI_REQUIRE(cdiv(max_ctx, 64) <= max_blocks_per_seq, "block table shorter than max_ctx");
  BI_REQUIRE(B <= 65535, "B too large");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  const FwdLayout L = plan_layout(m->cfg, B, B, max_ctx, B, mode);
  BI_REQUIRE(ws_bytes >= L.total, "forward workspace too small (bi_forward_workspace_size(cfg, B, B, max_ctx, B))");
  DevMeta dm{at<int32_t>(workspace, L.piece_seq), at<int32_t>(workspace, L.piece_row0),
             at<int32_t>(workspace, L.piece_pos0), at<int32_t>(workspace, L.ids), at<int32_t>(workspace, L.logit_src),
             at<int32_t>(workspace, L.logit_dst), at<int32_t>(workspace, L.logit_tgt),
             at<int32_t>(workspace, L.row_seq), at<int32_t>(workspace, L.row_pos)};
  const cudaStream_t st = as_stream(stream);
  BI_TRY(launched(launch_pdl(decode_embed_kernel, dim3((unsigned)B), dim3(128), 0, st, tokens, pos, (int)B, dm,
                             static_cast<const __nv_bfloat16*>(m->embed), m->cfg.vocab, m->cfg.d,
                             at<__nv_bfloat16>(workspace, L.h), device_status_ptr()),
                  "decode_embed_kernel"));
  PassShape ps{B, B, 1, max_ctx, B, true};
  return run_pass(m, workspace, L, ps, B, block_table, max_blocks_per_seq, k_cache, v_cache, n_blocks, true,
                  logprob_out, sampled_out, mode, stream);
}

}  // extern "C"
