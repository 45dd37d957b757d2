// CUDA-core (SIMT) attention kernels: the fp32 path of the library, and the backward's
// bandwidth-bound pieces shared with the tensor-core path (D = rowsum(dO * O) and the final
// dQ conversion, for fp32, bf16 and fp16).
//
// Forward ("FlashAttention paper story", tiling and online-softmax paragraphs): one CTA per
// 64-row query block; K/V stream through shared memory 64 keys at a time; every query row
// keeps a running maximum m, a running normaliser l and an un-normalised output, rescales
// them by exp(m_old - m_new) when the maximum grows, and divides by l at the end.  LSE = m +
// ln l is stored for the backward.
//
// Backward ("FlashAttention paper story", backward paragraph: P is recomputed from the stored
// statistics): one CTA per 64-key block keeps its K/V rows and its dK/dV accumulators on chip
// and visits every query block that may attend to it, rebuilding P = exp(scale*S - LSE).  dQ
// is reduced across key blocks with fp32 atomics into the workspace.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int kBr = 64;        // query rows per CTA (forward) / per inner step (backward)
constexpr int kBc = 64;        // keys per step (forward) / per CTA (backward)
constexpr int kThreads = 256;  // 8 warps

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Number of leading keys row i may attend to (all three key conditions are prefixes).
__device__ __forceinline__ int key_limit(int i, int N, int causal, int kv_len) {
  int lim = min(N, kv_len);
  if (causal) lim = min(lim, i + 1);
  return lim;
}

__device__ __forceinline__ int seq_kv_len(const int32_t* kv_lens, int b, int N) {
  if (kv_lens == nullptr) return N;
  int L = kv_lens[b];
  return L < 0 ? 0 : (L > N ? N : L);
}

// Load a [rows, D] tile (rows >= N_valid read as 0) into fp32 shared memory with row stride ld.
template <typename T, int D>
__device__ __forceinline__ void load_tile(float* dst, int ld, const T* src, int row0, int nrows, int N) {
  for (int e = threadIdx.x; e < nrows * D; e += kThreads) {
    int r = e / D, c = e % D;
    int gr = row0 + r;
    dst[r * ld + c] = gr < N ? to_f<T>(src[(size_t)gr * D + c]) : 0.f;
  }
}

// ------------------------------------------------------------------------------------------
// Forward
// ------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdArgs a) {
  extern __shared__ float smem[];
  constexpr int LDK = D + 1;
  float* Ks = smem;                 // [kBc][D+1]
  float* Vs = Ks + kBc * LDK;       // [kBc][D]
  float* Qs = Vs + kBc * D;         // [kBr][D]

  const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * kBr;
  const int N = a.N;
  const size_t head = ((size_t)b * a.H + h) * (size_t)N;
  const T* q = static_cast<const T*>(a.q) + head * D;
  const T* k = static_cast<const T*>(a.k) + head * D;
  const T* v = static_cast<const T*>(a.v) + head * D;
  T* o = static_cast<T*>(a.o) + head * D;
  const int kv_len = seq_kv_len(a.kv_lens, b, N);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int RPW = kBr / (kThreads / 32);   // rows per warp = 8
  constexpr int CPL = D / 32;                  // output columns per lane

  load_tile<T, D>(Qs, D, q, q0, kBr, N);

  float m[RPW], l[RPW], acc[RPW][CPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[r][c] = 0.f;
  }
  const int q_last = min(q0 + kBr, N) - 1;
  const int kv_end = a.causal ? min(kv_len, q_last + 1) : kv_len;

  for (int kv0 = 0; kv0 < kv_end; kv0 += kBc) {
    if (a.block_mask != nullptr &&
        a.block_mask[(size_t)(q0 / kMaskTile) * a.n_tiles + kv0 / kMaskTile] == 0)
      continue;   // tile skipped: its K/V rows are never loaded
    __syncthreads();
    load_tile<T, D>(Ks, LDK, k, kv0, kBc, N);
    load_tile<T, D>(Vs, D, v, kv0, kBc, N);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int lr = warp * RPW + r;
      const int i = q0 + lr;
      const int lim = key_limit(i, N, a.causal, kv_len) - kv0;
      const float* qr = Qs + lr * D;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) {
        const float qc = qr[c];
        s0 = fmaf(qc, Ks[lane * LDK + c], s0);
        s1 = fmaf(qc, Ks[(lane + 32) * LDK + c], s1);
      }
      s0 = lane < lim ? s0 * a.scale : -INFINITY;
      s1 = lane + 32 < lim ? s1 * a.scale : -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(fmaxf(s0, s1)));
      if (m_new == -INFINITY) continue;            // nothing allowed yet for this row
      const float alpha = expf(m[r] - m_new);      // 0 on the first contributing tile
      const float p0 = expf(s0 - m_new), p1 = expf(s1 - m_new);
      l[r] = l[r] * alpha + warp_sum(p0 + p1);
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[r][c] *= alpha;
      for (int j = 0; j < kBc; ++j) {
        const float pj = __shfl_sync(0xffffffffu, j < 32 ? p0 : p1, j & 31);
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[r][c] = fmaf(pj, Vs[j * D + lane + 32 * c], acc[r][c]);
      }
      m[r] = m_new;
    }
  }

#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int i = q0 + warp * RPW + r;
    if (i >= N) continue;
    const bool any = l[r] > 0.f;
    const float inv = any ? 1.f / l[r] : 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[(size_t)i * D + lane + 32 * c] = from_f<T>(acc[r][c] * inv);
    if (lane == 0) a.lse[head + i] = any ? m[r] + logf(l[r]) : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------------
// Backward main kernel (one CTA per 64-key block)
// ------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_simt_kernel(BwdArgs a) {
  extern __shared__ float smem[];
  constexpr int LD = D + 1;
  constexpr int LDP = kBc + 1;
  float* Ks = smem;               // [kBc][LD]
  float* Vs = Ks + kBc * LD;      // [kBc][LD]
  float* Qs = Vs + kBc * LD;      // [kBr][LD]
  float* dOs = Qs + kBr * LD;     // [kBr][LD]
  float* Ps = dOs + kBr * LD;     // [kBr][LDP]
  float* dSs = Ps + kBr * LDP;    // [kBr][LDP]
  float* lse_s = dSs + kBr * LDP; // [kBr]
  float* dl_s = lse_s + kBr;      // [kBr]

  const int b = blockIdx.z, h = blockIdx.y, kv0 = blockIdx.x * kBc;
  const int N = a.N;
  const size_t head = ((size_t)b * a.H + h) * (size_t)N;
  const T* q = static_cast<const T*>(a.q) + head * D;
  const T* k = static_cast<const T*>(a.k) + head * D;
  const T* v = static_cast<const T*>(a.v) + head * D;
  const T* dO = static_cast<const T*>(a.dO) + head * D;
  T* dk = static_cast<T*>(a.dk) + head * D;
  T* dv = static_cast<T*>(a.dv) + head * D;
  float* dq_acc = a.dq_acc + head * D;
  const float* lse = a.lse + head;
  const float* delta = a.delta + head;
  const int kv_len = seq_kv_len(a.kv_lens, b, N);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  constexpr int CPT = D / 16;     // columns per thread in the [64, D] products

  float dk_acc[4][CPT], dv_acc[4][CPT];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int c = 0; c < CPT; ++c) dk_acc[x][c] = dv_acc[x][c] = 0.f;

  if (kv0 < kv_len) {
    load_tile<T, D>(Ks, LD, k, kv0, kBc, N);
    load_tile<T, D>(Vs, LD, v, kv0, kBc, N);
    const int q_begin = a.causal ? (kv0 / kBr) * kBr : 0;
    for (int q0 = q_begin; q0 < N; q0 += kBr) {
      if (a.block_mask != nullptr &&
          a.block_mask[(size_t)(q0 / kMaskTile) * a.n_tiles + kv0 / kMaskTile] == 0)
        continue;
      __syncthreads();
      load_tile<T, D>(Qs, LD, q, q0, kBr, N);
      load_tile<T, D>(dOs, LD, dO, q0, kBr, N);
      for (int r = threadIdx.x; r < kBr; r += kThreads) {
        const bool in = q0 + r < N;
        lse_s[r] = in ? lse[q0 + r] : -INFINITY;
        dl_s[r] = in ? delta[q0 + r] : 0.f;
      }
      __syncthreads();
      // S = Q K^T and dP = dO V^T on a 4x4 micro-tile per thread; then P and dS.
      float s[4][4], dp[4][4];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) s[x][y] = dp[x][y] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        float qv[4], ov[4], kv[4], vv[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          qv[x] = Qs[(ty + 16 * x) * LD + c];
          ov[x] = dOs[(ty + 16 * x) * LD + c];
          kv[x] = Ks[(tx + 16 * x) * LD + c];
          vv[x] = Vs[(tx + 16 * x) * LD + c];
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            s[x][y] = fmaf(qv[x], kv[y], s[x][y]);
            dp[x][y] = fmaf(ov[x], vv[y], dp[x][y]);
          }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = ty + 16 * x, i = q0 + r;
        const int lim = key_limit(i, N, a.causal, kv_len);
        const float L = lse_s[r];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int cc = tx + 16 * y, j = kv0 + cc;
          const bool ok = i < N && j < lim && L != -INFINITY;
          const float p = ok ? expf(s[x][y] * a.scale - L) : 0.f;
          Ps[r * LDP + cc] = p;
          dSs[r * LDP + cc] = p * (dp[x][y] - dl_s[r]);
        }
      }
      __syncthreads();
      // dV += P^T dO, dK += dS^T Q (rows of this key block: ty + 16x; columns tx + 16c)
#pragma unroll 4
      for (int r = 0; r < kBr; ++r) {
        float pv[4], dsv[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          pv[x] = Ps[r * LDP + ty + 16 * x];
          dsv[x] = dSs[r * LDP + ty + 16 * x];
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const float ov = dOs[r * LD + tx + 16 * c];
          const float qv = Qs[r * LD + tx + 16 * c];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            dv_acc[x][c] = fmaf(pv[x], ov, dv_acc[x][c]);
            dk_acc[x][c] = fmaf(dsv[x], qv, dk_acc[x][c]);
          }
        }
      }
      // dQ += dS K (un-scaled; the convert kernel applies scale)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = ty + 16 * x;
        if (q0 + r >= N) continue;
        float dqv[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) dqv[c] = 0.f;
        for (int j = 0; j < kBc; ++j) {
          const float ds = dSs[r * LDP + j];
#pragma unroll
          for (int c = 0; c < CPT; ++c) dqv[c] = fmaf(ds, Ks[j * LD + tx + 16 * c], dqv[c]);
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c) atomicAdd(dq_acc + (size_t)(q0 + r) * D + tx + 16 * c, dqv[c]);
      }
    }
  }
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int j = kv0 + ty + 16 * x;
    if (j >= N) continue;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      dk[(size_t)j * D + tx + 16 * c] = from_f<T>(dk_acc[x][c] * a.scale);
      dv[(size_t)j * D + tx + 16 * c] = from_f<T>(dv_acc[x][c]);
    }
  }
}

// D_i = sum_c dO_ic * O_ic (O as stored), and zero row i of the dQ accumulator if there is one.
// One warp per row.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_preprocess_kernel(BwdArgs a) {
  const size_t rows = q_rows_total(a);
  const size_t row = (size_t)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const T* o = static_cast<const T*>(a.o) + row * D;
  const T* dO = static_cast<const T*>(a.dO) + row * D;
  float acc = 0.f;
#pragma unroll
  for (int c = lane; c < D; c += 32) {
    acc = fmaf(to_f<T>(dO[c]), to_f<T>(o[c]), acc);
    if (a.dq_acc != nullptr) a.dq_acc[row * D + c] = 0.f;
  }
  acc = warp_sum(acc);
  if (lane == 0) a.delta[row] = acc;
}

// dQ = scale * dQ_acc, converted to the output dtype.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dq_convert_kernel(BwdArgs a, size_t n) {
  T* dq = static_cast<T*>(a.dq);
  for (size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x; e < n; e += (size_t)gridDim.x * kThreads)
    dq[e] = from_f<T>(a.dq_acc[e] * a.scale);
}

// Split-KV merge ("FlashAttention：让精确注意力服从内存层次", section "Online softmax": two
// tiles' statistics (m, l, u) merge as m = max(m_a, m_b), l = e^{m_a-m} l_a + e^{m_b-m} l_b,
// u = e^{m_a-m} u_a + e^{m_b-m} u_b).  Each range s holds O_s = u_s / l_s and LSE_s = m_s + ln l_s,
// so with w_s = exp(LSE_s - max LSE): O = sum w_s O_s / sum w_s, LSE = max LSE + ln sum w_s.
// One warp per query row; a range with no allowed key (LSE_s = -inf) contributes nothing.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) splitkv_merge_kernel(SplitMergeArgs m) {
  const int row = blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= m.rows) return;
  float mx = -INFINITY;
  for (int sp = lane; sp < m.n_splits; sp += 32) mx = fmaxf(mx, m.lse_part[(size_t)sp * m.rows + row]);
  mx = warp_max(mx);
  constexpr int CPL = D / 32;
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int sp = 0; sp < m.n_splits; ++sp) {
      const float L = m.lse_part[(size_t)sp * m.rows + row];
      if (L == -INFINITY) continue;
      const float w = expf(L - mx);
      wsum += w;
      const float* src = m.o_part + ((size_t)sp * m.rows + row) * D;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[c] = fmaf(w, src[lane + 32 * c], acc[c]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  T* o = static_cast<T*>(m.o) + (size_t)row * D;
#pragma unroll
  for (int c = 0; c < CPL; ++c) o[lane + 32 * c] = from_f<T>(acc[c] * inv);
  if (lane == 0) m.lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

template <typename T, int D>
cudaError_t merge_launch(const SplitMergeArgs& m, cudaStream_t s) {
  const int blocks = (m.rows + kThreads / 32 - 1) / (kThreads / 32);
  splitkv_merge_kernel<T, D><<<blocks, kThreads, 0, s>>>(m);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t fwd_launch(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (kBc * (D + 1) + kBc * D + kBr * D);
  auto kern = fwd_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.N + kBr - 1) / kBr, a.H, a.B);
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_launch(const BwdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (2 * kBc * (D + 1) + 2 * kBr * (D + 1) + 2 * kBr * (kBc + 1) + 2 * kBr);
  auto kern = bwd_simt_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.N + kBc - 1) / kBc, a.H, a.B);
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t pre_launch(const BwdArgs& a, cudaStream_t s) {
  const size_t rows = q_rows_total(a);
  const size_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
  bwd_preprocess_kernel<T, D><<<(unsigned)blocks, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t conv_launch(const BwdArgs& a, cudaStream_t s) {
  const size_t n = q_rows_total(a) * a.d;
  size_t blocks = (n + kThreads - 1) / kThreads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  bwd_dq_convert_kernel<T><<<(unsigned)blocks, kThreads, 0, s>>>(a, n);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (dt != FA_FP32) return cudaErrorInvalidValue;     // 16-bit inputs run on the tensor cores
  return a.d == 64 ? fwd_launch<float, 64>(a, s) : fwd_launch<float, 128>(a, s);
}

cudaError_t launch_bwd_simt(const BwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (dt != FA_FP32) return cudaErrorInvalidValue;
  return a.d == 64 ? bwd_launch<float, 64>(a, s) : bwd_launch<float, 128>(a, s);
}

cudaError_t launch_bwd_preprocess(const BwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_FP32) return a.d == 64 ? pre_launch<float, 64>(a, s) : pre_launch<float, 128>(a, s);
  if (dt == FA_FP16) return a.d == 64 ? pre_launch<__half, 64>(a, s) : pre_launch<__half, 128>(a, s);
  return a.d == 64 ? pre_launch<__nv_bfloat16, 64>(a, s) : pre_launch<__nv_bfloat16, 128>(a, s);
}

cudaError_t launch_splitkv_merge(const SplitMergeArgs& m, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_FP16) return m.d == 64 ? merge_launch<__half, 64>(m, s) : merge_launch<__half, 128>(m, s);
  return m.d == 64 ? merge_launch<__nv_bfloat16, 64>(m, s) : merge_launch<__nv_bfloat16, 128>(m, s);
}

cudaError_t launch_bwd_dq_convert(const BwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_FP32) return conv_launch<float>(a, s);
  if (dt == FA_FP16) return conv_launch<__half>(a, s);
  return conv_launch<__nv_bfloat16>(a, s);
}

}  // namespace fa
