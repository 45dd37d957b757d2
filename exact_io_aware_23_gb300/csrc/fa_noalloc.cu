// fa_backward_noalloc: the backward for callers that cannot allocate device memory.
//
// fa_backward needs a caller-provided scratch workspace (the per-row D = rowsum(dO * O)).
// Some callers have no way to provide one: plugin interfaces that hand over only input and
// output pointers, hosts whose memory is entirely reserved by their own allocator, and
// latency-critical paths that may not call cudaMalloc because it synchronises the device.  This
// entry point takes its scratch from a fixed array compiled into the library instead, so it
// allocates nothing.
//
// The array lives in device memory of every GPU that loads the library, for the life of the
// process.  Its device address is looked up (cudaGetSymbolAddress) by the first call made in
// each CUDA context, with that context current, and cached for that context; make that first
// call before any stream capture.  A device reset (cudaDeviceReset) is not supported: the
// primary context can come back under the same handle, and the cached address would be stale.
// Every call shares the one array, so two calls that overlap on the GPU (different streams, or
// different host threads) race on it; serialise them.  Nothing needs to be cleared between
// calls: every call rewrites D for each row before reading it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"
#include "fa_sm103.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB

static __device__ __align__(256) uint8_t g_bwd_scratch[kScratchBytes];

fa::SymbolCache g_scratch_cache;

// Device address of the scratch array in the current context (looked up once per context).
fa_status scratch_address(void** out) {
  if (fa::symbol_address(g_scratch_cache, (const void*)g_bwd_scratch, out) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_backward_noalloc_max_workspace(void) { return kScratchBytes; }

fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal,
                              const uint8_t* block_mask, fa_dtype dtype, const int32_t* kv_lens,
                              void* stream) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return FA_OK;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (fa_backward_workspace_size(B, H, N, d) > kScratchBytes) return FA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  fa_status st = scratch_address(&ws);
  if (st != FA_OK) return st;
  return fa_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, block_mask,
                     dtype, kv_lens, ws, kScratchBytes, stream);
}

}  // extern "C"
