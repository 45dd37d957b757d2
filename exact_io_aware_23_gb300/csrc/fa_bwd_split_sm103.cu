// The deterministic backward's two tensor-core passes in one launch: the key-stationary dK/dV
// pass (fa_dkdv_sm103.cuh) and the query-stationary dQ pass (fa_dq_sm103.cuh).
//
// The passes are independent once D = rowsum(dO * O) exists, read the same four tensors and
// need one SM each (a CTA of either kind holds most of the shared memory and all of TMEM).  In
// one grid, the dK/dV CTAs come first and the dQ CTAs after them, so the last wave of the first
// pass is filled with the second pass's CTAs instead of idling.  (Alternating the two kinds
// CTA by CTA was measured 30 % slower: each kind then streams its slice's tiles at half the
// rate, and the tiles no longer stay in L2 between the CTAs that share them.)
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_dkdv_sm103.cuh"
#include "fa_dq_sm103.cuh"
#include "fa_internal.cuh"
#include "fa_sm103.cuh"

namespace fa {
namespace {

// Both passes run with BwdLayout<D>'s block, one CTA per SM: at d = 128 320 threads (10 warps,
// three on some of the SM's four 16K-register partitions, so at most 16384 / 96 -> 168
// registers a thread), at d = 64 576 (18 warps, at most 112).
template <int D, bool F16, bool kDrop>
__global__ void __launch_bounds__(BwdLayout<D>::kThreads, 1)
bwd_split_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const BwdArgs a, const int n_kv_units, const int n_q_units) {
  (void)n_q_units;
  // under a tile mask, a plan may reorder the units so that the longest start first
  const int x = a.perm != nullptr ? a.perm[blockIdx.x] : (int)blockIdx.x;
  if (x < n_kv_units) dkdv::run<D, F16, kDrop>(x, tmQ, tmK, tmV, tmDO, a);
  else dqp::run<D, F16, kDrop>(x - n_kv_units, tmQ, tmK, tmV, tmDO, a);
}

cudaError_t make_map(CUtensorMap* m, const void* base, int D, int N, int BH, bool f16) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tensor_map(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           3, base, dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, bool F16, bool kDrop>
cudaError_t launch(const BwdArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mdo;
  const int BH = a.B * a.H;            // query-side work units per tile row (Q, dO, dQ)
  const int BHkv = a.B * a.Hkv;        // key/value-side work units per tile row (K, V, dK, dV)
  // token axis and slice count of the tensor maps: per (b, h) slice, or packed per head
  const bool packed = a.cu_seqlens != nullptr;
  const int q_slices = packed ? a.H : BH, kv_slices = packed ? a.Hkv : BHkv;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, D, a.rows, q_slices, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, D, a.rows, kv_slices, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mv, a.v, D, a.rows, kv_slices, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mdo, a.dO, D, a.rows, q_slices, F16)) != cudaSuccess) return e;
  auto kern = bwd_split_sm103_kernel<D, F16, kDrop>;
  // each pass keeps its barriers 256 bytes below its live-tile bitmap (one bit per tile)
  const int bitmap = a.block_mask != nullptr ? ((a.n_tiles + 127) / 128) * 16 : 0;
  int smem = max(dkdv::Cfg<D, F16>::kSmem, dqp::Cfg<D, F16>::kSmem);
  smem = max(smem, dkdv::Cfg<D, F16>::kBar + 256 + bitmap);
  smem = max(smem, dqp::Cfg<D, F16>::kBar + 256 + bitmap);
  static LaunchSetup setup;
  if ((e = prepare_launch(setup, kern, smem)) != cudaSuccess) return e;
  const int n_t = (a.N + 127) / 128;
  const int n_kv = n_t * BHkv, n_q = n_t * BH;
  kern<<<dim3(n_kv + n_q), BwdLayout<D>::kThreads, smem, s>>>(mq, mk, mv, mdo, a, n_kv, n_q);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_split_sm103(const BwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (a.drop.enabled) {
    if (dt == FA_FP16) return a.d == 64 ? launch<64, true, true>(a, s) : launch<128, true, true>(a, s);
    return a.d == 64 ? launch<64, false, true>(a, s) : launch<128, false, true>(a, s);
  }
  if (dt == FA_FP16) return a.d == 64 ? launch<64, true, false>(a, s) : launch<128, true, false>(a, s);
  return a.d == 64 ? launch<64, false, false>(a, s) : launch<128, false, false>(a, s);
}

}  // namespace fa
