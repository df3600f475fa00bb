/*
 * bi.h — C ABI of the batch-invariant decoder forward library (libbi.so, sm_103a).
 *
 * What it computes: a pre-norm decoder forward (RMSNorm, GEMMs, RoPE, paged-KV
 * causal GQA attention with a fixed KV split, SwiGLU FFN or a top-k MoE FFN)
 * that ends in each sampled token's logprob.  Every row's result depends only
 * on that row's own inputs and absolute position, so a token gets the same
 * bits in a decode step, in a prefill chunk of any size and in any batch.
 *
 * Sources: "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
 * Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput" (the
 * Article), §2 (requirements: kernel determinism, batch independence, phase
 * consistency, same numerical contract, same discrete choices), §3.1 (training
 * forward calls the inference kernels), §4.1-4.6 (per-operator choices); and the
 * zero-mismatch-rl README ("Key features": fixed-split attention, fixed slot
 * order MoE combine).
 *
 * Conventions (all calls):
 *  - Tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous; bf16 tensors are passed as void*.  The library never frees
 *    caller memory and allocates no device memory in any call (the model
 *    handle holds only host-side data).
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = legacy default stream).  No call synchronises or reads device data
 *    back to the host, so calls can be captured into a CUDA graph once the
 *    same call has run once eagerly (first use configures kernel attributes).
 *  - Shapes are int64_t.  Invalid shapes or NULL required pointers return
 *    BI_ERR_INVALID_ARG (or BI_ERR_UNSUPPORTED_SHAPE for legal but
 *    unimplemented shapes) before anything is launched; bi_last_error() then
 *    describes the problem (thread-local string).
 *  - `mode` is BI_INVARIANT (the batch-invariant path) or BI_FAST, the same
 *    kernels with batch-dependent choices (split-K chosen from M, attention
 *    split size chosen from the batch, vocab split across CTAs) used as the
 *    non-invariant comparison baseline ([Article] §1: the >= 70% bar is
 *    measured against an equally optimised baseline).  BI_FAST results are NOT
 *    batch invariant.
 *  - Device-side waits are bounded; a kernel that gives up, or that sees an
 *    out-of-range index, records a code that bi_device_status() reports as
 *    BI_ERR_TIMEOUT / BI_ERR_DEVICE_CHECK.  Nothing traps.
 */
#ifndef BI_H_
#define BI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1,
  BI_ERR_UNSUPPORTED_SHAPE = 2,
  BI_ERR_CUDA = 3,
  BI_ERR_DEVICE_CHECK = 4,
  BI_ERR_TIMEOUT = 5
} bi_status;

typedef enum { BI_INVARIANT = 0, BI_FAST = 1 } bi_mode;
typedef enum { BI_DTYPE_BF16 = 0, BI_DTYPE_FP32 = 1 } bi_dtype;
typedef enum { BI_EPI_NONE = 0, BI_EPI_SWIGLU = 1 } bi_epilogue;

/* Library version (major * 10000 + minor * 100 + patch). */
int bi_version(void);
/* Description of the last error returned on this host thread ("" if none). */
const char* bi_last_error(void);
/* Number of kernel launches this library has issued from the host in this
 * process (a CUDA graph replay re-runs captured launches without counting). */
int64_t bi_launch_count(void);
/* Synchronises the current device, then returns BI_OK, BI_ERR_TIMEOUT (a
 * bounded device wait gave up) or BI_ERR_DEVICE_CHECK (a kernel saw an
 * out-of-range index) and clears the device status word. */
bi_status bi_device_status(void);

/* ------------------------------------------------------------------ RMSNorm
 * [Article] §3.1 (RMSNorm is one of the forward operators whose values come
 * from the inference kernel), §2 (batch independence).
 * y[r] = bf16( s[r] * (1 / sqrt(sum_i s[r,i]^2 / d + eps)) * gamma ), fp32 math,
 * where s = bf16(residual + x) if `residual` is non-NULL (and s is written back
 * into `residual`), else s = x.  One CTA per row; the sum of squares uses a fixed
 * per-thread stride, a fixed xor-butterfly warp tree and a fixed cross-warp order,
 * so a row's bits never depend on `rows`.
 * x, y: bf16 [rows, d]; residual: bf16 [rows, d] or NULL; gamma: bf16 [d].
 * d % 8 == 0, 8 <= d <= 16384, pointers 16-byte aligned.  y may alias x. */
bi_status bi_rmsnorm(const void* x, void* residual, const void* gamma, void* y, int64_t rows,
                     int64_t d, float eps, int mode, void* stream);

/* --------------------------------------------------------------------- GEMM
 * [Article] §4.1 "Dense GEMM: one accumulation order for every M".
 * C[m, n] = sum_k A[m, k] * W[n, k] with bf16 inputs and fp32 accumulation on
 * the tensor cores.  In BI_INVARIANT mode every element is the sum, in ascending
 * order, of 16-wide K steps (bf16 products, fp32 accumulator), never split: the
 * bits of row m do not depend on M or on the other rows.  Schedules: tcgen05
 * with a TMEM accumulator and TMA-fed 128B-swizzled 128 x BN x 64 tiles; for at
 * most 16 rows of a weight under 4M elements, mma.sync m16n8k16 with loader
 * warps (the same fp32 bits per K step).  BN does not change an element's bits;
 * it is bi_gemm_tile_n's width, or for 17..128 rows (without a fused RoPE) the
 * width that spreads the weight over the GPU.
 * A: bf16 [M, K]; W: bf16 [N, K] (nn.Linear layout); C: bf16 or fp32 [M, N]
 * (c_dtype), or for BI_EPI_SWIGLU: W holds 2F rows (gate rows then up rows)
 * and C is bf16 [M, F] with C = bf16( silu(bf16(g)) * bf16(u) ) computed in
 * fp32 and rounded once ([Article] §4.4, condition 3).
 * K % 64 == 0, N % 8 == 0 (F % 8 == 0 for SwiGLU), pointers 16-byte aligned.
 * `workspace` (may be NULL when bi_gemm_workspace_size() returns 0) holds the
 * fp32 split-K partials of BI_FAST mode. M == 0 is a no-op. */
bi_status bi_gemm(const void* A, int64_t M, int64_t K, const void* W, int64_t N, void* C, int c_dtype,
                  int epilogue, int mode, void* workspace, size_t ws_bytes, void* stream);
size_t bi_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int epilogue, int mode);
/* The N tile width bi_gemm uses for a weight of shape (N, K) at prefill size
 * (more than 128 rows; diagnostic): 16, 32, 64, 128 or 256, a function of (N, K,
 * epilogue) only.  The fused log-softmax (bi_lm_head_logprob) keeps this width
 * at every M, since its records are per tile. */
int bi_gemm_tile_n(int64_t N, int64_t K, int epilogue);

/* Grouped GEMM over 128-row tiles, each tile owned by one expert
 * ([Article] §4.4 "Expert GEMM: two layouts, same row result").
 * A: bf16 [M_rows, K] in a padded layout whose 128-row tile t belongs to
 * expert tile_expert[t] (device int32 [M_rows/128]; -1 = empty tile, skipped);
 * W: bf16 [E, N, K]; C: [M_rows, N] (or [M_rows, N/2] for SwiGLU).  Works for
 * the contiguous (packed by expert, padded to 128) and the masked (fixed
 * capacity per expert) layouts alike; a row's bits do not depend on the layout.
 * M_rows % 128 == 0. */
bi_status bi_grouped_gemm(const void* A, int64_t M_rows, int64_t K, const void* W, int64_t E, int64_t N,
                          const int32_t* tile_expert, void* C, int c_dtype, int epilogue, void* stream);

/* ------------------------------------------------------- RoPE + paged KV write
 * [Article] §4.2 (prefill, decode and training share one KV write and read
 * path; training writes into a private cache the same way).
 * For the T rows of a call, grouped into P "pieces" (consecutive tokens of one
 * sequence): piece p covers rows piece_row0[p] .. piece_row0[p+1]-1 of
 * sequence piece_seq[p] at absolute positions piece_pos0[p] + i.
 * qkv: bf16 [T, (Hq + 2 Hkv) hd] (q heads, k heads, v heads);
 * q_out: bf16 [T, Hq, hd] = rope(q); k_cache / v_cache: bf16
 * [n_blocks, Hkv, 64, hd] (one layer) receive rope(k) and v at
 * block_table[seq, pos / 64], slot pos % 64.  rope_table: fp32 [max_pos, hd]
 * (cos for i < hd/2 in the first half of each row, sin in the second), filled by
 * bi_rope_table().  Rotate-half pairs (i, i + hd/2), applied in fp32, rounded
 * once to bf16. max_q_len bounds the piece lengths (host value). */
bi_status bi_rope_kv_write(const void* qkv, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                           const float* rope_table, int64_t max_pos, const int32_t* block_table,
                           int64_t max_blocks_per_seq, int64_t n_blocks, void* q_out, void* k_cache,
                           void* v_cache, void* stream);
/* QKV projection with RoPE and the paged K/V write fused into the GEMM
 * epilogue: x [T, K] x Wqkv [(Hq + 2 Hkv) hd, K]^T, each q/k/v value rounded to
 * bf16 as bi_gemm would, then q and k rotated and everything written exactly as
 * bi_rope_kv_write does for row t at (row_seq[t], row_pos[t]) (device int32
 * [T]).  Same bits as the two calls, without the bf16 qkv round trip.  The
 * GEMM tile width is a multiple of hd (a tile holds whole heads).  x, wqkv,
 * rope_table, q_out and the caches must be 16-byte aligned.  The caller
 * guarantees 0 <= row_seq[t] < rows of block_table; a position outside
 * [0, max_pos) or a block id outside [0, n_blocks) skips that row's writes and
 * sets the device status (bi_device_status). */
bi_status bi_qkv_rope_kv_write(const void* x, int64_t T, int64_t K, const void* wqkv, int Hq, int Hkv, int hd,
                               const int32_t* row_seq, const int32_t* row_pos, const float* rope_table,
                               int64_t max_pos, const int32_t* block_table, int64_t max_blocks_per_seq,
                               int64_t n_blocks, void* q_out, void* k_cache, void* v_cache, int mode, void* stream);
/* rope_table[p, i] = cos(p * theta^(-2i/hd)), rope_table[p, hd/2 + i] = sin(...),
 * angles and functions evaluated in fp64 on the device, rounded to fp32. */
bi_status bi_rope_table(float* rope_table, int64_t max_pos, int hd, double theta, void* stream);

/* ---------------------------------------------------------------- attention
 * [Article] §4.2 (one read path for prefill and decode; decode's default
 * batch-dependent partition is given up) and the zero-mismatch-rl README
 * ("fixed-split attention").
 * Causal GQA over the paged cache.  Row (token t, q head h) at position p
 * attends to keys 0..p of its sequence through kv head h / (Hq/Hkv).  Keys are
 * processed in splits of `kv_split` absolute positions (512 by default, a
 * multiple of 64) and, inside a split, in tiles of 64 (one cache block) in
 * ascending order with an fp32 online softmax (scores and P in bf16 MMA, P
 * rounded to bf16).  The per-split partials (m, l, acc) are merged in
 * ascending split order:  M = max m_s, L = sum l_s 2^(m_s - M),
 * O = sum acc_s 2^(m_s - M), out = bf16(O / L).  Split and tile boundaries are
 * absolute positions, so a decode row reproduces its prefill row exactly.
 * q: bf16 [T, Hq, hd] (pieces as in bi_rope_kv_write); out: bf16 [T, Hq * hd].
 * hd in {64, 128}; Hq % Hkv == 0; 64 % (Hq/Hkv) == 0.  k_cache / v_cache
 * hold n_blocks pages of [Hkv, 64, hd] bf16; a block id outside [0, n_blocks)
 * is skipped and sets the device status.  max_ctx (host value) bounds every
 * sequence's context length in this call.  workspace must hold
 * bi_attention_workspace_size(T, Hq, hd, max_ctx, kv_split) bytes.
 * In BI_FAST mode the split size is chosen from the batch (flash-decoding
 * heuristic) and results are not batch invariant. */
bi_status bi_attention(const void* q, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                       const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx, int kv_split, float scale,
                       void* workspace, size_t ws_bytes, void* out, int mode, void* stream);
size_t bi_attention_workspace_size(int64_t max_T, int Hq, int hd, int64_t max_ctx, int kv_split);

/* Same computation and kernels as bi_attention (bitwise the same output), for
 * callers that cannot provide a device workspace: code that must not allocate
 * device memory on its hot path (a serving loop whose memory is reserved up
 * front, an allocator owned by another framework that this code cannot call),
 * plugins that a host application gives no scratch buffer, or runtimes with a
 * fixed memory budget.  The pages have no counterpart for this entry point.
 *  - The split partials go to a scratch array compiled into the library, 32 MiB
 *    on every GPU that loads the library, held until the process exits.  A call
 *    whose partials, T * Hq * ceil(max_ctx / split) * (hd + 2) * 4 bytes, exceed
 *    32 MiB returns BI_ERR_INVALID_ARG with the sizes in bi_last_error().
 *  - It allocates nothing: no cudaMalloc / cudaFree, no library allocator.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept with the unique id of the
 *    context it was found in: after cudaDeviceReset, or from another context,
 *    the next call looks it up again (so make that call outside a capture too).
 *  - The sizes are checked against the array on the host before any CUDA
 *    call; the check cannot wrap around for huge T or max_ctx.  As with
 *    bi_attention, the kernels take row indices from piece_row0, so every
 *    piece's rows must lie below T.
 *  - Every call on a device shares the one array and the array keeps the last
 *    call's contents; nothing in it needs to start at zero, because every
 *    partial that the merge reads is written earlier in the same call.  Calls
 *    that may run at the same time on the GPU (different streams, or several
 *    host threads) race on the array: serialise them.
 * Arguments are those of bi_attention without the workspace. */
bi_status bi_attention_static_scratch(const void* q, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                                      const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv,
                                      int hd, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                      int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx, int kv_split,
                                      float scale, void* out, int mode, void* stream);

/* ------------------------------------------------------------- block FP8
 * [Article] §4.1 ("Dense GEMM: keep FP8, one accumulation order for every M"):
 * block-FP8 W8A8, the training forward quantising its bf16 master weights by
 * the deployment rule.  Readings (the pages give no block sizes or scale
 * format): e4m3 "fn" codes, round to nearest even, saturating at 448, sign of
 * zero kept; 128 x 128 weight blocks and 1 x 128 activation blocks; scale of a
 * block = the smallest power of two s with 448 s >= amax (1 when amax = 0), so
 * a code times its scale is exact.
 *
 * bi_quantize_fp8: x bf16 [R, C] (device, row-major, C % 128 == 0) ->
 * q uint8 [R, C] (e4m3 codes of x / s) and scales fp32 [ceil(R / block_rows),
 * C / 128]; block_rows = 1 (activations) or 128 (weights).  Deterministic:
 * every block depends on its own elements only. */
bi_status bi_quantize_fp8(const void* x, int64_t R, int64_t C, int block_rows, void* q, float* scales,
                          void* stream);
/* bi_gemm_fp8: C = dequant(Aq) dequant(Wq)^T.  Aq uint8 [M, K] with sa fp32
 * [M, K/128] (1 x 128 blocks); Wq uint8 [N, K] with sw fp32 [N/128, K/128]
 * (128 x 128 blocks); C [M, N] bf16 or fp32 (c_dtype).  N and K multiples of
 * 128; Aq, Wq, C 16-byte aligned.  Per 128-wide K block the e4m3 products are
 * summed by tcgen05 MMAs in TMEM, then added in fp32, times the exact scale
 * product, in ascending block order: one tile shape and K order for every M
 * (BI_FAST runs the same kernel). */
bi_status bi_gemm_fp8(const void* Aq, const float* sa, int64_t M, int64_t K, const void* Wq, const float* sw,
                      int64_t N, void* C, int c_dtype, int mode, void* stream);
/* bi_rmsnorm_fp8: bi_rmsnorm (no mode argument: one schedule) whose bf16 output
 * rows are also quantised as bi_quantize_fp8 with block_rows = 1 would: codes
 * q uint8 [rows, d], scales q_scale fp32 [rows, d/128].  y (bf16 [rows, d]) may
 * be NULL; residual as in bi_rmsnorm.  d % 128 == 0, 128 <= d <= 16384; x, gamma,
 * y, residual 16-byte and q 8-byte aligned.  The codes and scales are bit-equal
 * to bi_rmsnorm followed by bi_quantize_fp8 (one kernel instead of two).
 *
 * bi_swiglu_fp8 (the SiLU-mul-quant step, [Article] §4.4): g13 bf16 [T, 2F] holds
 * a gate/up GEMM's output (gate columns 0..F-1, up columns F..2F-1);
 * a = bf16(silu(g) u) in fp32, rounded once, silu(g) = g / (1 + exp(-g)), then a's
 * 1 x 128 blocks to codes q uint8 [T, F] and scales q_scale fp32 [T, F/128], as
 * bi_quantize_fp8 would.  F % 128 == 0; g13 16-byte and q 4-byte aligned. */
bi_status bi_rmsnorm_fp8(const void* x, void* residual, const void* gamma, void* y, void* q, float* q_scale,
                         int64_t rows, int64_t d, float eps, void* stream);
bi_status bi_swiglu_fp8(const void* g13, int64_t T, int64_t F, void* q, float* q_scale, void* stream);

/* ---------------------------------------------------------- FP8 KV cache
 * [Article] §4.2 ("FP8 KV cache: keep FP8 storage, unify the read path"): K
 * and V are stored in FP8; prefill, decode and the training recompute all read
 * them through one path, dequantise-and-gather into a bf16 workspace sized by
 * limits, then the same bi_attention.  Readings: e4m3 codes, one power-of-two
 * scale per (token, kv head) vector of hd values for K and for V (smallest s
 * with 448 s >= amax, 1 for an all-zero vector); code x scale is exact in bf16.
 *
 * bi_kv_fp8_write: k, v bf16 [T, Hkv, hd] (device; rows grouped in pieces as in
 * bi_attention) -> codes in k_cache8 / v_cache8 uint8 [n_blocks, Hkv, 64, hd]
 * and scales in k_scale / v_scale fp32 [n_blocks, Hkv, 64] at each row's slot
 * (block_table[seq][pos / 64], pos % 64).  hd in {64, 128}.  A row whose block
 * is out of range is skipped and sets the device status. */
bi_status bi_kv_fp8_write(const void* k, const void* v, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                          const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hkv, int hd,
                          const int32_t* block_table, int64_t max_blocks_per_seq, int64_t n_blocks, void* k_cache8,
                          void* v_cache8, float* k_scale, float* v_scale, void* stream);
/* bi_kv_fp8_gather: for every piece p, the pages holding positions
 * 0 .. piece_pos0[p] + (its rows) - 1 of its sequence, dequantised into the
 * bf16 workspace page p * max_blocks_per_seq + l (k_ws, v_ws bf16
 * [P * max_blocks_per_seq, Hkv, 64, hd]; workspace and cache 16-byte aligned);
 * ws_block_table int32 [P, max_blocks_per_seq] receives those page ids (-1
 * after the last page).  Call bi_attention with the workspace as the cache,
 * ws_block_table as the block table and piece p reading row p of it
 * (piece_seq = 0 .. P-1), n_blocks = P * max_blocks_per_seq. */
bi_status bi_kv_fp8_gather(const void* k_cache8, const void* v_cache8, const float* k_scale, const float* v_scale,
                           int64_t n_blocks, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int Hkv, int hd, const int32_t* block_table,
                           int64_t max_blocks_per_seq, void* k_ws, void* v_ws, int32_t* ws_block_table,
                           void* stream);
/* bi_attention_fp8: bi_attention reading the FP8 cache directly, with the same
 * three schedules and per-row arithmetic.  Each 64-key page's codes are expanded
 * in shared memory into the bf16 values of the codes (unscaled, exact); the K
 * scale then multiplies each score column and the V scale each P element
 * before its bf16 rounding.  With power-of-two scales both products are exact,
 * so every row's bits equal bi_kv_fp8_gather + bi_attention (outputs within a
 * few ulps of fp32's smallest normal number excepted: there, P.V terms below
 * 2^-126 may round differently).  Prefill, decode and recompute all read
 * through this one path.  k_cache8 / v_cache8 uint8 and k_scale / v_scale fp32
 * as written by bi_kv_fp8_write (16-byte aligned); the other arguments as in
 * bi_attention.  out (bf16 [T, Hq*hd]) may be NULL when out_q is given; out_q
 * (uint8 [T, Hq*hd]) and out_scale (fp32 [T, Hq*hd/128]), both NULL or both
 * set, receive the output rows quantised as bi_quantize_fp8 with
 * block_rows = 1 would (Hq*hd % 128 == 0), fused into the split merge. */
bi_status bi_attention_fp8(const void* q, int64_t T, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int64_t max_q_len, int Hq, int Hkv, int hd,
                           const void* k_cache8, const void* v_cache8, const float* k_scale, const float* v_scale,
                           const int32_t* block_table, int64_t max_blocks_per_seq, int64_t n_blocks, int64_t max_ctx,
                           int kv_split, float scale, void* workspace, size_t ws_bytes, void* out, void* out_q,
                           float* out_scale, int mode, void* stream);

/* --------------------------------------------------- Mamba-2 chunked scan
 * [Article] §6 ("Transfer: Nemotron, a Mamba hybrid architecture + NVFP4"):
 * decode replays prefill's chunked arithmetic instead of its own single-step
 * recurrence.  Per head h (group g = h / (H/G) shares B and C):
 *   state_t = exp(loga_t) state_{t-1} + B_t x_t^T,  y_t = C_t^T state_t,
 * computed in chunk form over absolute chunks [cQ, cQ + Q): a row uses the
 * state entering its chunk plus the chunk's earlier rows, and the state is
 * advanced only when a chunk completes, each sum in ascending index order.  So
 * a decode step, a prefill over the whole sequence and any chunking of it give
 * the same bits for every row.
 * Inputs (device): x bf16 [T, H, P], B and C bf16 [T, G, N], loga fp32 [T, H]
 * (<= 0); pieces as in bi_attention (piece_seq [pieces], piece_row0
 * [pieces + 1], piece_pos0 [pieces]): at most one piece per sequence per call,
 * each sequence's pieces passed in position order over successive calls;
 * max_q_len (host) bounds the rows of any piece, and calls with max_q_len = 1
 * (decode steps) run a lighter schedule of the same arithmetic.
 * state: fp32, 16-byte aligned, bi_ssd_state_bytes(H, G, P, N, Q) bytes per
 * sequence (n_seq of them), zeroed by the caller for a new sequence; it holds the state
 * entering the current chunk and that chunk's earlier inputs.  y: fp32
 * [T, H, P].  Q <= 64, N <= 128, P <= 128, each a multiple of 4.  BI_FAST
 * runs the same kernel. */
size_t bi_ssd_state_bytes(int H, int G, int P, int N, int Q);
bi_status bi_ssd_chunk_scan(const void* x, const void* B, const void* C, const float* loga, const int32_t* piece_seq,
                            const int32_t* piece_row0, const int32_t* piece_pos0, int64_t pieces, int64_t max_q_len,
                            int H, int G, int P, int N, int Q, void* state, int64_t n_seq, float* y, int mode,
                            void* stream);

/* ------------------------------------------------------- deterministic Top-K
 * [Article] §4.3 ("Top-K in sparse attention: fix ties and order").
 * Row t of `scores` (device fp32, row stride ld elements) scores the candidate
 * positions 0 .. n_valid[t] - 1 (in-request positions; device int32 [T]).  The
 * K candidates that come first in the order (score descending, then position
 * descending) -- the unique key "score bits, then position bits" -- are
 * selected and written to idx_out[t, 0 .. K) (device int32 [T, K]) in
 * descending position order, followed by -1 when n_valid[t] < K.  Scores
 * compare as numbers (-0 ties +0; -inf is a score); NaN is outside the
 * contract.  K in [1, 4096].  A row with n_valid outside [0, ld] is clamped and
 * sets the device status.
 * BI_FAST: ties at the threshold score go to whichever candidates claim a slot
 * first and the selection is left unsorted (the non-deterministic default the
 * pages replace; same set of scores, not the same positions). */
bi_status bi_topk(const float* scores, int64_t T, int64_t ld, const int32_t* n_valid, int K, int32_t* idx_out,
                  int mode, void* stream);

/* ---------------------------------------------------------- embed / logprob
 * Row gather: out[t] = table[ids[t]] (bf16 [V, d] -> bf16 [T, d]).  Ids outside
 * [0, V) write zeros and record BI_ERR_DEVICE_CHECK. */
bi_status bi_embed(const int32_t* ids, int64_t T, const void* table, int64_t V, int64_t d, void* out,
                   void* stream);

/* [Article] §2 (diff is defined on each sampled token's logprob), §3.1 ("the
 * final logprob").  For each row t of fp32 logits [T, V]:
 *   lse = m + log(sum_v exp(x_v - m)),   lp[t] = x[t, id_t] - lse
 * with one CTA per row, a single pass keeping an online (max, sum) per thread
 * over a fixed index stride, and a fixed butterfly / cross-warp merge order.
 * ids: device int32 [T] or NULL (greedy: id = argmax, ties to the lowest id).
 * argmax_out: device int32 [T] or NULL.  V >= 1, V % 4 == 0.
 * BI_FAST splits the vocab across CTAs when T is small (not batch invariant);
 * it then needs bi_logprob_workspace_size() bytes of workspace. */
bi_status bi_logprob_gather(const float* logits, const int32_t* ids, int64_t T, int64_t V, float* logprob_out,
                            int32_t* argmax_out, int mode, void* workspace, size_t ws_bytes, void* stream);
size_t bi_logprob_workspace_size(int64_t T, int64_t V, int mode);

/* Fused lm_head + log-softmax + gather: logprob_out[t] = x[t, id_t] - lse(x[t, :])
 * with x = X W^T never written to memory.  The GEMM epilogue of each 128 x BN
 * tile keeps, per row and in column order, an fp32 online (max, sum-exp,
 * argmax) and the target's logit; the per-tile records are then merged per
 * row in a fixed order (thread t takes tiles t, t+128, ..., then a fixed
 * butterfly and warp order).  BN is the weight's invariant tile width, so a
 * row's bits do not depend on T.  (The article lists "the final logprob" among
 * the fused forward outputs, [Article] §3.1.)
 * X: bf16 [T, K]; W: bf16 [V, K]; ids: device int32 [T] or NULL (greedy: the
 * argmax, ties to the lowest id); argmax_out: int32 [T] or NULL.  K % 64 == 0,
 * V % 8 == 0.  workspace: bi_lm_head_logprob_workspace_size(T, V, K, mode)
 * bytes.  BI_FAST narrows the vocab tiles for T <= 128 (not batch invariant). */
bi_status bi_lm_head_logprob(const void* X, int64_t T, int64_t K, const void* W, int64_t V, const int32_t* ids,
                             float* logprob_out, int32_t* argmax_out, int mode, void* workspace, size_t ws_bytes,
                             void* stream);
size_t bi_lm_head_logprob_workspace_size(int64_t T, int64_t V, int64_t K, int mode);

/* ---------------------------------------------------------------------- MoE
 * Router: [Article] §2 "the same discrete choices", §4.4 (router output fp32
 * at every batch size).  For each token, the k largest of E fp32 logits
 * (ties to the lower expert id), slot 0 = best; weights = softmax over the k
 * selected logits in slot order.  ids: int32 [T, k], weights: fp32 [T, k].
 * E <= 64, k <= E. */
bi_status bi_moe_route_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, float* weights,
                            void* stream);

/* Contiguous expert layout ([Article] §4.4, training side): a stable counting
 * sort of the T*k (token, slot) pairs by expert, each expert's rows padded to a
 * multiple of 128.  Outputs: row_of_slot int32 [T*k] (row in the padded layout
 * of pair (t, s)), tile_expert int32 [max_rows/128] (-1 for unused tiles) and
 * expert_offsets int32 [E+1].  max_rows >= T*k + 128*E rounded to 128.
 * workspace: bi_moe_permute_workspace_size(T, k, E) bytes. */
bi_status bi_moe_permute(const int32_t* ids, int64_t T, int k, int E, int64_t max_rows, int32_t* row_of_slot,
                         int32_t* tile_expert, int32_t* expert_offsets, void* workspace, size_t ws_bytes,
                         void* stream);
size_t bi_moe_permute_workspace_size(int64_t T, int k, int E);
/* Masked expert layout ([Article] §4.4, rollout side): expert e owns rows
 * [e*capacity, (e+1)*capacity); pairs beyond an expert's capacity are an error
 * (BI_ERR_DEVICE_CHECK).  capacity % 128 == 0. */
bi_status bi_moe_permute_masked(const int32_t* ids, int64_t T, int k, int E, int64_t capacity,
                                int32_t* row_of_slot, int32_t* tile_expert, void* workspace, size_t ws_bytes,
                                void* stream);
/* xp[row_of_slot[t*k+s]] = x[t] for every (t, s) (bf16 rows of length d). */
bi_status bi_moe_gather(const void* x, const int32_t* row_of_slot, int64_t T, int k, int64_t d, void* xp,
                        void* stream);
/* [Article] §4.5 ("accumulated in FP32 in top-k slot order") and the README
 * ("fixed slot order"): out[t] = bf16( sum_{s=0..k-1} w[t,s] * y[row_of_slot[t*k+s]] ),
 * fp32, slots summed sequentially.  y: bf16 [rows, d]; out: bf16 [T, d].
 * BI_FAST uses fp32 atomics (order not fixed) and needs
 * bi_moe_combine_workspace_size() bytes. */
bi_status bi_moe_combine(const void* y, const int32_t* row_of_slot, const float* w, int64_t T, int k, int64_t d,
                         void* out, int mode, void* workspace, size_t ws_bytes, void* stream);
size_t bi_moe_combine_workspace_size(int64_t T, int64_t d, int mode);

/* Whole MoE FFN layer: route, permute (contiguous layout), gather, grouped
 * gate_up GEMM with SwiGLU, grouped down GEMM, slot-order combine.
 * x: bf16 [T, d]; router_logits fp32 [T, E]; w13 bf16 [E, 2F, d]; w2 bf16 [E, d, F];
 * out bf16 [T, d].  workspace: bi_moe_layer_workspace_size() bytes.  Both
 * modes run the same kernels (the slot-order combine measured faster than the
 * fp32-atomic one on this GPU, so the non-invariant layer uses it too). */
bi_status bi_moe_layer(const void* x, const float* router_logits, int64_t T, int64_t d, int E, int k, int64_t F,
                       const void* w13, const void* w2, void* out, int mode, void* workspace, size_t ws_bytes,
                       void* stream);
size_t bi_moe_layer_workspace_size(int64_t T, int64_t d, int E, int k, int64_t F, int mode);

/* ------------------------------------------------------------- model driver
 * [Article] §3.1: the training forward calls the inference kernels; here both
 * the rollout (decode) and the training recompute (chunked prefill) call the
 * same entry points below, which call the same kernels. */
typedef struct {
  int64_t n_layers, d, n_heads_q, n_heads_kv, head_dim, ffn, vocab;
  float eps;          /* RMSNorm epsilon (1e-6) */
  float rope_theta;   /* 10000 */
  int64_t kv_block;   /* tokens per cache block: must be 64 */
  int64_t kv_split;   /* attention KV split, multiple of 64 (512) */
  int64_t max_pos;    /* rows of the RoPE table = maximum context length */
  int64_t fp8;        /* 0: bf16 linear layers and KV cache.  1: block-FP8 W8A8 linear layers (the
                         attention, FFN and their activations; not the embedding or lm_head) and
                         an FP8 KV cache, [Article] §4.1-4.2 (see bi_gemm_fp8, bi_kv_fp8_write) */
} bi_model_config;

typedef struct {
  const void* attn_norm; /* bf16 [d] */
  const void* wqkv;      /* bf16 [(Hq + 2 Hkv) hd, d] */
  const void* wo;        /* bf16 [d, Hq hd] */
  const void* ffn_norm;  /* bf16 [d] */
  const void* w13;       /* bf16 [2F, d]: gate rows, then up rows */
  const void* w2;        /* bf16 [d, F] */
  /* fp8 = 1 only: e4m3 codes and 128 x 128 block scales of the same weights
   * (bi_quantize_fp8 with block_rows = 128; the training side requantises its
   * bf16 masters by this rule before each forward, or keeps the copy) */
  const void* wqkv8; const float* wqkv_s;
  const void* wo8;   const float* wo_s;
  const void* w138;  const float* w13_s;
  const void* w28;   const float* w2_s;
} bi_layer_weights;

typedef struct {
  const void* embed;              /* bf16 [V, d] */
  const void* final_norm;         /* bf16 [d] */
  const void* lm_head;            /* bf16 [V, d] */
  const bi_layer_weights* layers; /* host array [n_layers] (copied) */
  float* rope_table;              /* device fp32 [max_pos, hd], caller-allocated; filled by bi_model_create */
} bi_weights;

typedef struct bi_model bi_model;

/* Validates the config, copies the weight pointers (weights stay owned by the
 * caller and may be overwritten in place between calls: [Article] §4.6,
 * conflict 3) and fills the RoPE table on `stream`. */
bi_status bi_model_create(const bi_model_config* cfg, const bi_weights* w, void* stream, bi_model** out);
void bi_model_destroy(bi_model* m);

/* Layer-by-layer dump for locating the first divergent layer ([Article] §5:
 * "on a mismatch, compare layer by layer for the first divergent layer").
 * While set, every forward pass of at most max_rows rows writes into
 * dump (device bf16 [n_layers + 2, max_rows, d]): slot l < n_layers the residual
 * stream entering layer l, slot n_layers the residual after the last layer,
 * slot n_layers + 1 the final-norm output, rows in pass order (for a prefill
 * processed in one pass, i.e. T <= max_tokens and chunk >= every sequence
 * length, that is the call's row order).  Passes longer than max_rows are not
 * dumped.  NULL disables it.  Adds copies to the stream; results are unchanged. */
bi_status bi_model_set_dump(bi_model* m, void* dump, int64_t max_rows);

/* Paged KV cache of one model: k_cache and v_cache are bf16
 * [n_layers, n_blocks, Hkv, 64, hd]; block_table is int32 [B, max_blocks_per_seq]. */
size_t bi_kv_cache_bytes(const bi_model_config* cfg, int64_t n_blocks);

/* Workspace for bi_forward_prefill / bi_forward_decode: sized only by limits
 * (max_tokens rows per layer pass, max_pieces sequences per pass, max_ctx
 * context, max_logit_rows lm_head rows per launch), never by the batch of a
 * particular call ([Article] §4.6, conflict 2). */
size_t bi_forward_workspace_size(const bi_model_config* cfg, int64_t max_tokens, int64_t max_pieces,
                                 int64_t max_ctx, int64_t max_logit_rows, int mode);

/* Chunked, packed prefill (rollout prompt processing and training recompute).
 * tokens: device int32 [T], sequences packed back to back; cu_seqlens (HOST
 * int64 [B+1]) gives sequence b's rows; start_pos (HOST int64 [B]) is how many
 * tokens of sequence b are already in the cache (its first row sits at that
 * position).  Rows are processed in chunks of at most `chunk` tokens per
 * sequence and passes of at most `max_tokens` rows (the workspace limit).
 * logit_from (HOST int64 [B] or NULL = every row): the first in-call row index
 * of sequence b whose logprob is wanted; rows from there to the sequence end
 * get logits.  target_ids: device int32 [T] (target of each row) or NULL for
 * greedy (argmax).  logprob_out (fp32 [T]) and sampled_out (int32 [T], may be
 * NULL) are written for rows with logits only.  block_table: device int32
 * [B, max_blocks_per_seq]. */
bi_status bi_forward_prefill(bi_model* m, const int32_t* tokens, const int32_t* target_ids,
                             const int64_t* cu_seqlens, const int64_t* start_pos, const int64_t* logit_from,
                             int64_t B, int64_t chunk, const int32_t* block_table, int64_t max_blocks_per_seq,
                             void* k_cache, void* v_cache, int64_t n_blocks, float* logprob_out,
                             int32_t* sampled_out, void* workspace, size_t ws_bytes, int64_t max_tokens,
                             int64_t max_ctx, int64_t max_logit_rows, int mode, void* stream);
/* The pass schedule bi_forward_prefill runs for these sequences (host only, no
 * GPU; a diagnostic).  Arguments as in bi_forward_prefill (cu_seqlens, start_pos,
 * logit_from HOST int64; B sequences; chunk; max_tokens).  Writes one record of 8
 * int64 per piece, in launch order, to out (HOST int64 [out_rows, 8]; may be
 * NULL): (pass, sequence, first row in the pass, rows, first position, first
 * packed token, first row with logits relative to the piece, first logit row in
 * the pass).  Returns the number of pieces (records beyond out_rows are not
 * written), or -1 for invalid arguments. */
int64_t bi_prefill_plan(const int64_t* cu_seqlens, const int64_t* start_pos, const int64_t* logit_from, int64_t B,
                        int64_t chunk, int64_t max_tokens, int64_t* out, int64_t out_rows);

/* One greedy decode step for B sequences: token b (device int32 [B]) sits at
 * position pos[b] (device int32 [B]); its K/V are written to the cache, and the
 * argmax of the next-token distribution and its logprob are written to
 * sampled_out / logprob_out (device [B]).  max_ctx is a static upper bound on
 * pos[b] + 1 (a graph captured with it stays valid while the bound holds).
 * No host reads: capturable into a CUDA graph. */
bi_status bi_forward_decode(bi_model* m, const int32_t* tokens, const int32_t* pos, int64_t B,
                            const int32_t* block_table, int64_t max_blocks_per_seq, void* k_cache, void* v_cache,
                            int64_t n_blocks, int64_t max_ctx, int32_t* sampled_out, float* logprob_out,
                            void* workspace, size_t ws_bytes, int mode, void* stream);

/* Rollout bookkeeping after a decode step (device only, capturable):
 * hist_ids[step, b] = sampled[b], hist_lp[step, b] = logprob[b] with
 * step = *step_counter; then tokens[b] = sampled[b], pos[b] += 1, and
 * *step_counter += 1.  hist_*: [max_steps, B]; steps beyond max_steps are
 * dropped and recorded as BI_ERR_DEVICE_CHECK. */
bi_status bi_decode_advance(const int32_t* sampled, const float* logprob, int32_t* tokens, int32_t* pos,
                            int64_t B, int32_t* step_counter, int32_t* hist_ids, float* hist_lp,
                            int64_t max_steps, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_H_ */
