// Launchers of the sm_103a tensor-core kernels and the TMA descriptor helper they share.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.cuh"

namespace fa {

// bf16 / fp16 forward (tcgen05 + TMA), d in {64, 128}.
cudaError_t launch_fwd_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s);

// bf16 / fp16 backward main kernel (tcgen05 + TMA), d in {64, 128}; runs between the
// preprocess and the dQ conversion kernels.
cudaError_t launch_bwd_sm103(const BwdArgs& a, fa_dtype dt, cudaStream_t s);

// bf16 / fp16 deterministic backward, both tensor-core passes in one launch (tcgen05 + TMA),
// d in {64, 128}: key-stationary CTAs write dK and dV, query-stationary CTAs write dQ; no result
// is added from several CTAs.
cudaError_t launch_bwd_split_sm103(const BwdArgs& a, fa_dtype dt, cudaStream_t s);

// Encodes a tiled TMA descriptor through the driver entry point (resolved once per process).
cudaError_t encode_tensor_map(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank,
                              const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                              const cuuint32_t* box, const cuuint32_t* elem_strides,
                              CUtensorMapSwizzle swizzle);

}  // namespace fa
