// Shared device/host helpers of the batch-invariant forward library (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor), the 5th
// generation tensor core (tcgen05 + TMEM) and cp.async, plus the host-side
// error plumbing behind bi_status / bi_last_error.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <string>
#include <utility>

#include "../../include/bi.h"

namespace bi {

// ---------------------------------------------------------------- host errors
void set_error(const std::string& msg);
bi_status fail(bi_status st, const std::string& msg);
bi_status check_launch(const char* what);

#define BI_REQUIRE(cond, msg)                                                    \
  do {                                                                           \
    if (!(cond)) return ::bi::fail(BI_ERR_INVALID_ARG, std::string(__func__) + ": " + (msg)); \
  } while (0)

#define BI_REQUIRE_SHAPE(cond, msg)                                              \
  do {                                                                           \
    if (!(cond)) return ::bi::fail(BI_ERR_UNSUPPORTED_SHAPE, std::string(__func__) + ": " + (msg)); \
  } while (0)

#define BI_TRY(...)                                                              \
  do {                                                                           \
    bi_status _st = (__VA_ARGS__);                                               \
    if (_st != BI_OK) return _st;                                                \
  } while (0)

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int num_sms();

// Device status word: kernels that give up a bounded wait, or that see an
// out-of-range index, record a code here instead of trapping.
enum DeviceCode : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_INDEX = 2 };
int* device_status_ptr();  // device address of the status word (current device and context)


// Device addresses of a module's __device__ symbol, remembered per device
// together with the unique id of the context they were looked up in: a
// context made again (after cudaDeviceReset, or a context the caller created)
// loads the module at a new address, and the changed id makes the next call
// look it up again instead of handing a kernel the stale one.
struct ModuleAddressCache {
  std::mutex mu;
  void* addr[64] = {nullptr};
  unsigned long long ctx[64] = {0};
};
// The current context's unique id (false when none is current or the driver
// lacks cuCtxGetId).
bool current_context_id(unsigned long long* id);
// Address of `symbol` on the current device in the current context, through
// `cache`; false (no address) when the lookup fails.
bool module_symbol_address(const void* symbol, void** out, ModuleAddressCache* cache);

// Internal launchers shared between translation units (same kernels as the
// public entry points, with a row indirection the model driver uses).
// RMSNorm of rows idx[0..rows) of x / residual into the compact y[0..rows).
bi_status rmsnorm_rows(const void* x, void* residual, const void* gamma, void* y, int64_t rows, int64_t d, float eps,
                       const int32_t* idx, void* stream);
// The same with x + residual written to res_out (NULL iff residual is NULL), which
// may be the residual rows themselves or another buffer.
bi_status rmsnorm_rows_to(const void* x, const void* residual, void* res_out, const void* gamma, void* y, int64_t rows,
                          int64_t d, float eps, const int32_t* idx, void* stream);
// Logprob / argmax of each logits row, written to out index dst[row] (dst may be NULL).
bi_status logprob_gather_to(const float* logits, const int32_t* ids, int64_t T, int64_t V, float* logprob_out,
                            int32_t* argmax_out, const int32_t* dst, int mode, void* workspace, size_t ws_bytes,
                            void* stream);

// Per-(row, vocab tile) partial of the fused lm_head + log-softmax: the tile's
// max, sum of exp(x - max), argmax (value, lowest index) and the target's logit
// when the target id falls in the tile.
struct TileLse {
  float m, s, best, xt;
  int idx;
  int pad[3];
};
// Merge the n_tiles partials of each of T rows (fixed order) into the logprob
// of ids[row] (or of the argmax when ids is NULL), written to index dst[row].
bi_status lse_tiles_merge(const TileLse* part, int64_t T, int n_tiles, int tile_n, const int32_t* ids,
                          float* logprob_out, int32_t* argmax_out, const int32_t* dst, void* stream);

// Fused lm_head + log-softmax with results at index dst[row]; its workspace size.
bi_status lm_head_logprob_to(const void* X, int64_t T, int64_t K, const void* W, int64_t V, const int32_t* ids,
                             float* logprob_out, int32_t* argmax_out, const int32_t* dst, int mode, void* workspace,
                             size_t ws_bytes, void* stream);
size_t lm_head_partial_bytes(int64_t T, int64_t V, int64_t K, int mode);
// QKV projection whose epilogue applies RoPE (q, k) and writes k, v into the
// paged cache at each row's (row_seq, row_pos): the same values as bi_gemm
// followed by bi_rope_kv_write, without the bf16 qkv round trip.
bi_status kv_fp8_gather_to(const void* k_cache8, const void* v_cache8, const float* k_scale, const float* v_scale,
                           int64_t n_blocks, const int32_t* piece_seq, const int32_t* piece_row0,
                           const int32_t* piece_pos0, int64_t P, int Hkv, int hd, const int32_t* block_table,
                           int64_t max_blocks_per_seq, int64_t ws_blk, void* k_ws, void* v_ws, int32_t* ws_block_table,
                           cudaStream_t st);
bi_status rope_kv_write_fp8(const void* qkv, int64_t T, const int32_t* row_seq, const int32_t* row_pos, int Hq,
                            int Hkv, int hd, const float* table, int64_t max_pos, const int32_t* block_table,
                            int64_t max_blk, int64_t n_blocks, void* q_out, void* k8, float* ks, void* v8, float* vs,
                            cudaStream_t st);
bi_status swiglu_fp8(const void* g13, int64_t T, int64_t F, void* q, float* qs, cudaStream_t st);
bi_status rmsnorm_fp8_rows(const void* x, void* residual, const void* gamma, void* y, void* q, float* qs,
                           int64_t rows, int64_t d, float eps, void* stream);
bi_status gemm_qkv_rope(const void* A, int64_t M, int64_t K, const void* W, int64_t N, const int32_t* row_seq,
                        const int32_t* row_pos, const float* rope_table, int64_t max_pos, const int32_t* block_table,
                        int64_t max_blk, int64_t n_blocks, void* q_out, void* k_cache, void* v_cache, int Hq, int Hkv,
                        int hd, int mode, void* stream);

// RMSNorm in front of a GEMM: the GEMM's A rows are y = RMSNorm(x (+ res_in)) *
// gamma (the norm kernels' arithmetic) and res_out receives x + res_in.  A
// decode-size call computes y inside the GEMM; otherwise the norm kernel runs
// first and writes y.
struct NormIn {
  const void* x;       // [M, K] bf16
  const void* res_in;  // [M, K] bf16 residual stream, or NULL (the norm of x alone)
  void* res_out;       // [M, K] bf16 x + res_in, a buffer other than res_in; NULL iff res_in is
  const void* gamma;   // [K] bf16
  float eps;
  void* y;             // [M, K] bf16 rows of the norm when it runs as its own kernel
};
// Dense GEMM (BI_EPI_NONE or BI_EPI_SWIGLU, bf16 out) of the normalised rows.
bi_status gemm_norm(const NormIn& norm, int64_t M, int64_t K, const void* W, int64_t N, void* C, int epilogue,
                    int mode, void* workspace, size_t ws_bytes, void* stream);
// gemm_qkv_rope of the normalised rows.
bi_status gemm_qkv_rope_norm(const NormIn& norm, int64_t M, int64_t K, const void* W, int64_t N,
                             const int32_t* row_seq, const int32_t* row_pos, const float* rope_table, int64_t max_pos,
                             const int32_t* block_table, int64_t max_blk, int64_t n_blocks, void* q_out,
                             void* k_cache, void* v_cache, int Hq, int Hkv, int hd, int mode, void* stream);

// TMA descriptor encode (driver entry point looked up through the runtime).
bool encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                         bool swizzle128);
// 8-bit elements (fp8 codes or raw bytes), 128-byte swizzle unless swizzle128 is false.
bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_outer, bool swizzle128 = true);

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while its predecessor in the stream is still finishing; it must execute
// pdl_wait() (below) before touching anything the predecessor writes or reads.
// Every kernel of this library calls pdl_trigger() and pdl_wait() in all of its
// CTAs, so completion stays transitive along the stream.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Status of a launch: its own return code, then the runtime's sticky error.
inline bi_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(BI_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  }
  return check_launch(what);
}

// ---------------------------------------------------------------- device side
#define BI_DEV __device__ __forceinline__

// Let the next kernel in the stream start its launch (its CTAs then wait in pdl_wait).
BI_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the preceding kernel has completed and its memory is visible
// (returns at once when the kernel was launched without the attribute).
BI_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Move registers between warpgroups: every warp of a warpgroup executes the same
// one.  An increase waits until decreases elsewhere in the block have freed
// enough of the registers the block launched with, so the block's split must fit
// that total and every decrease must run before any warp can stop.
template <int N>
BI_DEV void reg_alloc_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory"); }
template <int N>
BI_DEV void reg_alloc_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory"); }

// Bounded waits give up after this many nanoseconds (global timer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

BI_DEV unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

BI_DEV void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

BI_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier
BI_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
BI_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
BI_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

BI_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
BI_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
BI_DEV bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of the barrier to complete; false after the time limit.
BI_DEV bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// ---- TMA
BI_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
BI_DEV void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---- tcgen05 (cta_group::1)
BI_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
BI_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
BI_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
BI_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BI_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem desc) * B(smem desc)^T, bf16 inputs, fp32 accumulate.
BI_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc)^T, e4m3 inputs (K = 32 per instruction), fp32 accumulate.
BI_DEV void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread complete.
BI_DEV void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 lanes x 32 bit, 32 consecutive columns: thread i of the warp gets lane (base + i).
BI_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 32 bit, 2 consecutive columns.
BI_DEV void tmem_ld_32x32b_x2(uint32_t taddr, uint32_t (&r)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
}
// 32 lanes x 32 bit, 16 consecutive columns: thread i of the warp writes lane (base + i).
BI_DEV void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 32 bit, 4 consecutive columns.
BI_DEV void tmem_ld_32x32b_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
// 32 lanes x 32 bit, 16 consecutive columns.
BI_DEV void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
BI_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 32 bit, 32 consecutive columns: thread i of the warp writes lane (base + i).
BI_DEV void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 16 lanes x 4 x 256 bits: thread t holds lanes base + t/4 (registers 4k, 4k + 1) and
// base + t/4 + 8 (4k + 2, 4k + 3) at columns 8k + 2 (t % 4) + {0, 1}, k = 0..3: the
// mma.sync m16n8 accumulator layout, repeated over four 8-column groups.
BI_DEV void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
BI_DEV void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
BI_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// CW (16 or 32) consecutive columns of a warp's 32 TMEM lanes, loaded or stored.
template <int CW>
BI_DEV void tmem_ld_cols_attn(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32) tmem_ld_32x32b_x32(taddr, r);
  else tmem_ld_32x32b_x16(taddr, r);
}
template <int CW>
BI_DEV void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[CW]) {
  if constexpr (CW == 32) tmem_st_32x32b_x32(taddr, r);
  else tmem_st_32x32b_x16(taddr, r);
}

// Shared-memory matrix descriptor for a K-major operand written by TMA with
// 128-byte swizzle: 8-row core groups 1024 bytes apart (stride byte offset),
// descriptor version 1, layout type 2 (SWIZZLE_128B).
BI_DEV uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);      // start address
  d |= (uint64_t)1 << 16;                           // leading byte offset (unused with swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
  d |= (uint64_t)1 << 46;                           // version
  d |= (uint64_t)2 << 61;                           // SWIZZLE_128B
  return d;
}

// Shared-memory matrix descriptor for an MN-major operand with 128-byte
// swizzle: rows of 64 consecutive MN elements (128 bytes) per K index, 8 K rows
// per 1024-byte swizzle atom; `lbo` = bytes between 64-element groups along MN,
// `sbo` = bytes between 8-row groups along K.  (A V page as the paged cache's
// TMA copy leaves it: key rows of 64 head dims, one box per 64 dims.)
BI_DEV uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: kind::f8f6f4, A = B = e4m3 (format 0), D = fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// ---- cp.async (16 bytes, zero-fill when src_bytes == 0)
BI_DEV void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
BI_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// One arrival on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count includes this thread; noinc: the arrival is not added).
BI_DEV void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
BI_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- ldmatrix / mma.sync (legacy warp-level tensor-core path)
BI_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
BI_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16 bf16) * B(16x8 bf16) + D, fp32 accumulate
BI_DEV void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Contiguous global -> shared copy by the bulk-copy engine, completing on `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16).
BI_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---- bf16 helpers
BI_DEV float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
BI_DEV __nv_bfloat16 f2bf(float x) { return __float2bfloat16_rn(x); }
BI_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
BI_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
BI_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace bi
