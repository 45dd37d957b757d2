// Launchers of the sm_103a tensor-core kernels and the TMA descriptor helper they share.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "fa_internal.cuh"

namespace fa {

// bf16 / fp16 forward (tcgen05 + TMA), d in {64, 128}.
cudaError_t launch_fwd_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s);
// the balanced block-sparse forward at d = 64 (a plan in `a`): persistent CTAs
cudaError_t launch_fwd_bs_persist_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s);
// d = 64 without a tile mask, packing, split-KV or dropout: 64-key tiles, two CTAs per SM
cudaError_t launch_fwd_bn64_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s);

// bf16 / fp16 backward main kernel (tcgen05 + TMA), d in {64, 128}; runs between the
// preprocess and the dQ conversion kernels.
cudaError_t launch_bwd_sm103(const BwdArgs& a, fa_dtype dt, cudaStream_t s);

// bf16 / fp16 deterministic backward, both tensor-core passes in one launch (tcgen05 + TMA),
// d in {64, 128}: key-stationary CTAs write dK and dV, query-stationary CTAs write dQ; no result
// is added from several CTAs.
cudaError_t launch_bwd_split_sm103(const BwdArgs& a, fa_dtype dt, cudaStream_t s);

// Compute layout of the two-pass backward's CTAs (both passes, one launch): kWG compute
// warpgroups, each over 128 / kWG columns of a 128 x 128 tile, then the producer warp and the
// MMA-issuing warp.  At d = 64 the tensor work per tile is half that of d = 128 and the compute
// warps set the pace: four warpgroups of 32 columns hide more of their latency (same results);
// at d = 128 two of 64 measured faster.
template <int D>
struct BwdLayout {
  static constexpr int kWG = D == 64 ? 4 : 2;
  static constexpr int kCols = 128 / kWG;
  static constexpr int kComputeWarps = 4 * kWG;
  static constexpr int kProducerWarp = kComputeWarps;
  static constexpr int kMmaWarp = kComputeWarps + 1;
  static constexpr int kThreads = 32 * (kComputeWarps + 2);
};

// Per-kernel launch set-up made once per device and kept: the dynamic shared memory the kernel
// is opted in to (raised when a launch asks for more) and its registers per thread, so that a
// launch queries and sets nothing in the runtime once its device has seen the kernel (a short
// call's host time is a visible part of its time).
struct LaunchSetup {
  static constexpr int kDevices = 64;
  std::atomic<int> smem[kDevices] = {};
  std::atomic<int> regs[kDevices] = {};
};

// The current device's SM count, asked of the runtime once per device (a persistent grid's size).
inline cudaError_t sm_count(int* out) {
  static std::atomic<int> cache[LaunchSetup::kDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < LaunchSetup::kDevices;
  int n = cached ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (cached) cache[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return cudaSuccess;
}

template <typename Kern>
cudaError_t prepare_launch(LaunchSetup& c, Kern kern, int smem, int* regs = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < LaunchSetup::kDevices;
  if (!cached || c.smem[dev].load(std::memory_order_acquire) < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (cached) {
      int cur = c.smem[dev].load(std::memory_order_relaxed);
      while (cur < smem && !c.smem[dev].compare_exchange_weak(cur, smem, std::memory_order_release)) {
      }
    }
  }
  if (regs != nullptr) {
    int r = cached ? c.regs[dev].load(std::memory_order_acquire) : 0;
    if (r == 0) {
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
      r = fa.numRegs;
      if (cached) c.regs[dev].store(r, std::memory_order_release);
    }
    *regs = r;
  }
  return cudaSuccess;
}

// Encodes a tiled TMA descriptor through the driver entry point (resolved once per process).
cudaError_t encode_tensor_map(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank,
                              const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                              const cuuint32_t* box, const cuuint32_t* elem_strides,
                              CUtensorMapSwizzle swizzle);

// Device addresses of one of the library's __device__ variables, one per CUDA context that
// looked it up (a context is where a module's globals live: another device, or another context
// on the same device, has its own copy).  A context destroyed while the process runs (for
// example by cudaDeviceReset) can come back under the same handle; its cached address is then
// stale, so the library does not support further calls on a device after a reset.
struct SymbolCache {
  static constexpr int kEntries = 64;
  std::mutex mu;
  void* ctx[kEntries] = {nullptr};
  void* ptr[kEntries] = {nullptr};
  int n = 0;
  int next = 0;
};

// The device address of `symbol` in the calling thread's current context (looked up with
// cudaGetSymbolAddress on the first call in that context, cached afterwards).
cudaError_t symbol_address(SymbolCache& cache, const void* symbol, void** out);

}  // namespace fa
