// Work plan of the balanced block-sparse forward.
//
// A tile mask can give some query rows far more live key tiles than others (the global rows of a
// local + global pattern see every key tile; "FlashAttention paper story", block-sparse paragraph:
// local windows plus global tokens).  One CTA per 256-row Q-tile pair then leaves those pairs as
// one long chain that outlasts all the other work.  The plan cuts every pair whose live key
// tiles exceed a target chain length into ranges of about equal length, each run by its own CTA
// (extra CTAs drawn from a fixed budget per (b, h) slice); the ranges' partial results are merged
// with the (m, l, u) merge law ("FlashAttention：让精确注意力服从内存层次", section "Online
// softmax").  The plan depends only on the mask, so it is the same on every call: the results are
// reproducible to the bit.
//
// Two launches: one warp per pair counts the pair's live key tiles (either row of the pair live,
// causal tiles past the diagonal excluded) and keeps them as a bitmap, then one CTA turns the
// counts into the plan:
//   target length  L = max(32, (live tiles of all slices / SMs) / 4)
//   ranges         S_p = ceil(c_p / L) when c_p > L (at most 32), else 1; pairs are split in
//                  order while their extra CTAs (S_p - 1) fit the budget, the rest run whole
//   entries        the split pairs' ranges first (they are the longest chains), then the whole
//                  pairs (the last pairs first when causal: they have the most tiles), then empty.
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_internal.cuh"

namespace fa {
namespace {

constexpr int kMaxPairs = 3072;     // N <= 786432 with a tile mask
constexpr int kMaxRanges = 32;
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(256) pair_count_kernel(PlanArgs p) {
  const int pair = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (pair >= p.n_pairs) return;
  const int r0 = 2 * pair, r1 = 2 * pair + 1;
  const int jmax = p.causal ? min(p.T, r1 + 1) : p.T;
  const uint8_t* m0 = p.block_mask + (size_t)r0 * p.T;
  const uint8_t* m1 = r1 < p.T ? p.block_mask + (size_t)r1 * p.T : nullptr;
  // one ballot per 32 key tiles: the pair's live-tile bitmap (kept for the persistent forward)
  // and its count
  int c = 0;
  for (int w = 0; w < p.words; ++w) {
    const int j = w * 32 + lane;
    const bool live = j < jmax && (m0[j] != 0 || (m1 != nullptr && m1[j] != 0));
    const uint32_t bits = __ballot_sync(0xffffffffu, live);
    c += __popc(bits);
    if (lane == 0) p.pair_bits[(size_t)pair * p.words + w] = bits;
  }
  if (lane == 0) p.counts[pair] = c;
}

// In-place exclusive prefix sum of v[0, n), n <= 3 * blockDim.x; returns the total.  Every thread
// of the block must call it.
__device__ int block_exclusive_scan(int* v, int n) {
  __shared__ int warp_sum[32];
  __shared__ int total;
  const int t = threadIdx.x, lane = t % 32, w = t / 32;
  const int i0 = 3 * t;
  const int x0 = i0 < n ? v[i0] : 0, x1 = i0 + 1 < n ? v[i0 + 1] : 0, x2 = i0 + 2 < n ? v[i0 + 2] : 0;
  const int own = x0 + x1 + x2;
  int inc = own;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_sum[w] = inc;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x / 32;
    const int ws = lane < nw ? warp_sum[lane] : 0;
    int wi = ws;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) warp_sum[lane] = wi - ws;
    if (lane == 31) total = wi;
  }
  __syncthreads();
  const int ex = warp_sum[w] + inc - own;
  if (i0 < n) v[i0] = ex;
  if (i0 + 1 < n) v[i0 + 1] = ex + x0;
  if (i0 + 2 < n) v[i0 + 2] = ex + x0 + x1;
  __syncthreads();
  return total;
}

__device__ __forceinline__ int ranges_wanted(int c, int target) {
  return c > target ? min(kMaxRanges, (c + target - 1) / target) : 1;
}

__global__ void __launch_bounds__(kPlanThreads) blocksparse_plan_kernel(PlanArgs p) {
  __shared__ int s_cnt[kMaxPairs], s_a[kMaxPairs], s_b[kMaxPairs];
  __shared__ int s_sum[32];
  __shared__ int s_target;
  const int P = p.n_pairs, t = threadIdx.x;
  int part = 0;
  for (int i = t; i < P; i += kPlanThreads) {
    s_cnt[i] = p.counts[i];
    part += s_cnt[i];
  }
  part = __reduce_add_sync(0xffffffffu, part);
  if (t % 32 == 0) s_sum[t / 32] = part;
  __syncthreads();
  if (t == 0) {
    long long total = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) total += s_sum[w];
    const long long per_sm = total * p.BH / (p.sms > 0 ? p.sms : 1);
    s_target = (int)max(32LL, per_sm / 4);
  }
  __syncthreads();
  const int target = s_target;
  for (int i = t; i < P; i += kPlanThreads) s_a[i] = ranges_wanted(s_cnt[i], target) - 1;
  __syncthreads();
  block_exclusive_scan(s_a, P);                     // extra CTAs wanted by the pairs before i
  for (int i = t; i < P; i += kPlanThreads) {
    int S = ranges_wanted(s_cnt[i], target);
    if (s_a[i] + S - 1 > p.extra) S = 1;            // over the budget: this pair runs whole
    s_a[i] = S;
    s_b[i] = S > 1 ? S : 0;
    s_cnt[i] = S > 1 ? 0 : 1;
  }
  __syncthreads();
  const int n_split = block_exclusive_scan(s_b, P);     // first entry (and slot) of a split pair
  const int n_whole = block_exclusive_scan(s_cnt, P);   // rank of a whole pair
  for (int i = t; i < P; i += kPlanThreads) {
    const int S = s_a[i];
    if (S > 1) {
      for (int r = 0; r < S; ++r) p.plan[s_b[i] + r] = make_int4(i, r, S, s_b[i] + r);
    } else {
      const int k = p.causal ? n_whole - 1 - s_cnt[i] : s_cnt[i];
      p.plan[n_split + k] = make_int4(i, 0, 1, -1);
    }
  }
  for (int e = n_split + n_whole + t; e < P + p.extra; e += kPlanThreads) p.plan[e] = make_int4(-1, 0, 0, 0);
  for (int e = t; e < p.BH * p.n_slots; e += kPlanThreads) p.merge_count[e] = 0;
  if (t == 0) *p.next_unit = 0;
}

// ---- the backward's unit order ----------------------------------------------------------------
//
// In the two-pass backward a key tile's dK/dV CTA visits the tile's live query tiles and a query
// tile's dQ CTA its live key tiles.  Under a local + global mask the global columns and rows make
// a few units hundreds of tiles long; left in place (dK/dV units first, then dQ units) the long dQ
// units start only when every dK/dV CTA has been scheduled, and their chains run on alone at the
// end.  Ordered so that every unit more than twice as long as the average comes first, all long
// chains start in the first wave.  Each unit computes the same numbers in any order (no result is
// added from several CTAs), so the order changes no bit of the results.

// One CTA per 8 mask rows, one warp per row: the row's live-tile count, and its share of every
// column's count (summed in shared memory, then added to the global column counts).
__global__ void __launch_bounds__(256) tile_count_kernel(OrderArgs p) {
  extern __shared__ int colsum[];                  // [T]
  const int T = p.T, t = threadIdx.x, lane = t % 32;
  for (int j = t; j < T; j += 256) colsum[j] = 0;
  __syncthreads();
  const int i = blockIdx.x * 8 + t / 32;
  if (i < T) {
    const uint8_t* row = p.block_mask + (size_t)i * T;
    const int jmax = p.causal ? min(T, i + 1) : T;
    int c = 0;
    for (int j = lane; j < jmax; j += 32) {
      if (row[j] != 0) {
        ++c;
        atomicAdd(colsum + j, 1);
      }
    }
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) p.counts[T + i] = c;
  }
  __syncthreads();
  for (int j = t; j < T; j += 256)
    if (colsum[j] != 0) atomicAdd(p.counts + j, colsum[j]);
}

__global__ void __launch_bounds__(kPlanThreads) backward_order_kernel(OrderArgs p) {
  __shared__ int s_sum[32];
  __shared__ int s_avg2;
  const int n = 2 * p.T, t = threadIdx.x;
  int part = 0;
  for (int e = t; e < n; e += kPlanThreads) part += p.counts[e];
  part = __reduce_add_sync(0xffffffffu, part);
  if (t % 32 == 0) s_sum[t / 32] = part;
  __syncthreads();
  if (t == 0) {
    long long total = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) total += s_sum[w];
    s_avg2 = (int)((2 * total + n - 1) / n);       // twice the average length
  }
  __syncthreads();
  // rank among the long entries (first), then among the others; each group keeps the entry order
  int n_long = 0;
  for (int base = 0; base < n; base += 3 * kPlanThreads) {
    const int m = min(n - base, 3 * kPlanThreads);
    for (int e = t; e < m; e += kPlanThreads) p.rank[base + e] = p.counts[base + e] > s_avg2 ? 1 : 0;
    __syncthreads();
    const int tot = block_exclusive_scan(p.rank + base, m);
    for (int e = t; e < m; e += kPlanThreads) {
      const bool lng = p.counts[base + e] > s_avg2;
      const int r = p.rank[base + e] + n_long;     // long entries before this one
      p.rank[base + e] = lng ? r : -1 - ((base + e) - r);    // short: -(1 + short entries before)
    }
    __syncthreads();
    n_long += tot;
  }
  for (int e = t; e < n; e += kPlanThreads) {
    const int r = p.rank[e];
    const int pos = r >= 0 ? r : n_long + (-1 - r);
    p.order[pos] = make_int2(e < p.T ? 0 : 1, e < p.T ? e : e - p.T);
  }
  __syncthreads();
  // CTA offsets: the dK/dV units of a key tile are the key/value slices, the dQ units the query slices
  for (int base = 0, carry = 0; base < n; base += 3 * kPlanThreads) {
    const int m = min(n - base, 3 * kPlanThreads);
    for (int e = t; e < m; e += kPlanThreads) p.order_off[base + e] = p.order[base + e].x == 0 ? p.BHkv : p.BH;
    __syncthreads();
    const int tot = block_exclusive_scan(p.order_off + base, m);
    for (int e = t; e < m; e += kPlanThreads) p.order_off[base + e] += carry;
    __syncthreads();
    carry += tot;
    if (base + m >= n && t == 0) p.order_off[n] = carry;
  }
  __syncthreads();
  // the permutation: entry e's CTAs run the units the unplanned launch gives to
  // key tile j (CTAs j*BHkv + slice) or query tile i (after all dK/dV CTAs, slices fastest, the
  // last tiles first when causal)
  const int n_kv = p.T * p.BHkv;
  for (int e = t; e < n; e += kPlanThreads) {
    const int2 en = p.order[e];
    const int off = p.order_off[e];
    const int it = p.causal ? p.T - 1 - en.y : en.y;
    const int base_x = en.x == 0 ? en.y * p.BHkv : n_kv + it * p.BH;
    const int size = en.x == 0 ? p.BHkv : p.BH;
    for (int k = 0; k < size; ++k) p.perm[off + k] = base_x + k;
  }
}

}  // namespace

cudaError_t launch_backward_order(const OrderArgs& p, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.counts, 0, (size_t)p.T * sizeof(int), s);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)p.T * sizeof(int);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(tile_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  tile_count_kernel<<<(p.T + 7) / 8, 256, smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  backward_order_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_blocksparse_plan(const PlanArgs& p, cudaStream_t s) {
  if (p.n_pairs > kMaxPairs || 2 * p.extra > p.n_slots) return cudaErrorInvalidValue;
  pair_count_kernel<<<(p.n_pairs + 7) / 8, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  blocksparse_plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
