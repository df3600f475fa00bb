// Host plumbing: error strings, device status word, SM count, TMA descriptor encode.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"

namespace bi {

static thread_local std::string g_last_error;
static std::atomic<long long> g_launches{0};

// The device status word (one per device that loads the library).
__device__ int g_device_status = 0;

void set_error(const std::string& msg) { g_last_error = msg; }

bi_status fail(bi_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

bi_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(BI_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return BI_OK;
}

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  static int cached[64] = {0};
  if (dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// Driver calls reached through the runtime's entry-point table (the library
// links no libcuda): the current context and its unique id.
static PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
static PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

bool current_context_id(unsigned long long* id) {
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

bool module_symbol_address(const void* symbol, void** out, ModuleAddressCache* cache) {
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return false;
  }
  unsigned long long ctx = 0;
  bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(cache->mu);
  if (have_ctx && cache->addr[dev] && cache->ctx[dev] == ctx) {
    *out = cache->addr[dev];
    return true;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) {
    cudaGetLastError();
    return false;
  }
  // the lookup makes the device's primary context current if none was
  if (!have_ctx) have_ctx = current_context_id(&ctx);
  cache->addr[dev] = have_ctx ? p : nullptr;
  cache->ctx[dev] = have_ctx ? ctx : 0;
  *out = p;
  return true;
}

int* device_status_ptr() {
  static ModuleAddressCache cache;
  void* p = nullptr;
  return module_symbol_address(&g_device_status, &p, &cache) ? static_cast<int*>(p) : nullptr;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace bi

extern "C" {

int bi_version(void) { return 100; }

const char* bi_last_error(void) { return bi::g_last_error.c_str(); }

int64_t bi_launch_count(void) { return bi::g_launches.load(std::memory_order_relaxed); }

bi_status bi_device_status(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return bi::fail(BI_ERR_CUDA, std::string("bi_device_status: ") + cudaGetErrorString(e));
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, bi::g_device_status, sizeof(int));
  if (e != cudaSuccess) return bi::fail(BI_ERR_CUDA, std::string("bi_device_status: ") + cudaGetErrorString(e));
  int zero = 0;
  cudaMemcpyToSymbol(bi::g_device_status, &zero, sizeof(int));
  if (v == bi::DEV_TIMEOUT) return bi::fail(BI_ERR_TIMEOUT, "a bounded device wait gave up");
  if (v != 0) return bi::fail(BI_ERR_DEVICE_CHECK, "a kernel saw an out-of-range index (code " + std::to_string(v) + ")");
  return BI_OK;
}

}  // extern "C"
