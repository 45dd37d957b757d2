// TMA descriptor encoding.  cuTensorMapEncodeTiled is a driver API function; it is looked up
// through the runtime's entry-point query so the library does not link against libcuda and
// loads on machines without a GPU driver.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa_sm103.cuh"

namespace fa {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn g_encode = nullptr;
std::once_flag g_once;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<EncodeFn>(fn);
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;

void resolve_ctx() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
}

// A key for the calling thread's current CUDA context: its handle, or, if the driver's
// cuCtxGetCurrent cannot be reached, the current device (one context per device, as with the
// runtime's primary contexts).  Null when no context is current yet.
cudaError_t current_context(void** ctx) {
  std::call_once(g_ctx_once, resolve_ctx);
  *ctx = nullptr;
  if (g_ctx_get != nullptr) {
    CUcontext c = nullptr;
    if (g_ctx_get(&c) == CUDA_SUCCESS) {
      *ctx = static_cast<void*>(c);
      return cudaSuccess;
    }
  }
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  *ctx = reinterpret_cast<void*>(static_cast<uintptr_t>(dev) + 1);
  return cudaSuccess;
}

}  // namespace

cudaError_t symbol_address(SymbolCache& cache, const void* symbol, void** out) {
  *out = nullptr;
  void* ctx = nullptr;
  cudaError_t e = current_context(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(cache.mu);
  if (ctx != nullptr) {
    for (int i = 0; i < cache.n; ++i) {
      if (cache.ctx[i] == ctx) {
        *out = cache.ptr[i];
        return cudaSuccess;
      }
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, symbol);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  if (ctx == nullptr && current_context(&ctx) != cudaSuccess) ctx = nullptr;   // the lookup made
                                                                              // a context current
  if (ctx != nullptr) {
    const int slot = cache.n < SymbolCache::kEntries ? cache.n++ : (cache.next++ % SymbolCache::kEntries);
    cache.ctx[slot] = ctx;
    cache.ptr[slot] = p;
  }
  *out = p;
  return cudaSuccess;
}

cudaError_t encode_tensor_map(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank,
                              const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                              const cuuint32_t* box, const cuuint32_t* elem_strides,
                              CUtensorMapSwizzle swizzle) {
  std::call_once(g_once, resolve);
  if (g_encode == nullptr) return cudaErrorNotSupported;
  CUresult r = g_encode(m, dt, rank, const_cast<void*>(base), dims, strides, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace fa
