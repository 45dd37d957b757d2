// Internal declarations shared by the translation units of libfa: launch parameters and the
// launchers each kernel file exports to the C-ABI layer (fa_api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

constexpr int kMaskTile = 128;   // granularity of the block-sparse tile mask

// Error word written by kernels (one per device, read by fa_check_device_status).
enum DeviceError : int { kDevOk = 0, kDevTimeout = 1, kDevMisaligned = 2, kDevBadOffsets = 3 };

struct DebugKnobs {
  int inject;              // 1: skip the first K/V tile load of every CTA (watchdog test)
  uint32_t wait_limit_ms;  // bound of every mbarrier wait
};

// Dropout on P (see dropout_sm103.cuh for the generator and the mask layout).  Zero-initialised
// arguments mean no dropout.
struct DropoutArgs {
  int enabled;
  uint32_t seed_lo, seed_hi;   // Philox key
  uint32_t offset;             // Philox counter word 3
  int k8;                      // keep iff the element's 8-bit uniform is below k8 (0..256)
  float scale;                 // 256 / k8, or 0 when k8 == 0
  uint32_t rk0[10], rk1[10];   // the generator's key in each of its ten rounds (host-computed)
};

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, d;
  int Hkv;                    // key/value heads (H for plain attention; H / G with grouped queries)
  float scale;
  int causal;
  const uint8_t* block_mask;  // [T, T] or null
  int n_tiles;                // T = ceil(N / 128)
  const int32_t* kv_lens;     // [B] or null
  int* err;                   // device error word
  DebugKnobs dbg;
  int heads_fastest;          // launch order: (b, h) slice fastest (unequal work per tile)
  // Split-KV (fa_forward_splitkv): keys per slice, key-tile ranges per Q-tile pair and the fp32
  // partial results ([n_splits][B*H][N][d] and [n_splits][B*H][N]); Nk = N, n_splits = 1 and
  // o_part = null for fa_forward.
  int Nk;
  int n_splits;
  int tiles_per_split;
  float* o_part;
  float* lse_part;
  // Packed sequences (ragged offsets): null, or [B + 1] device offsets of B sequences packed
  // back to back along each head's token axis of `rows` tokens; N is then the longest
  // sequence and Q, K, V, O are [H or Hkv, rows, d].  Without them rows = N.
  const int32_t* cu_seqlens;
  int rows;
  DropoutArgs drop;
  // Balanced block-sparse forward (fa_forward_blocksparse): a work plan maps CTA x to slice
  // x % (B*H) and plan entry x / (B*H) = {Q-tile pair, range r, ranges S, partial slot}, pair < 0
  // for no work.  A pair split into S > 1 ranges of its live key tiles writes fp32 partials
  // (O_r = u_r / l_r and LSE_r) to slots [slot - r, slot - r + S) of its slice
  // (o_part: [B*H][n_slots][256][d], lse_part: [B*H][n_slots][256]); the range that finishes last
  // (merge_count[B*H][n_slots], counted at the first slot) merges them.  Null plan: one CTA per pair.
  const int4* plan;
  int plan_entries;
  int n_slots;
  int* merge_count;
  // Persistent balanced forward (d = 64): one CTA per SM claims the plan's units (entry x slice,
  // in plan order) from next_unit, zeroed by the plan; pair_bits[pair][bit_words] are the
  // pairs' live key tiles.  Null next_unit: one CTA per unit.
  int* next_unit;
  const uint32_t* pair_bits;
  int bit_words;
};

// The work plan of the balanced block-sparse forward (see FwdArgs::plan).
struct PlanArgs {
  const uint8_t* block_mask;  // [T, T]
  int T, n_pairs, causal;
  int extra;                  // extra CTAs per slice (the split budget)
  int n_slots;                // partial slots per slice (>= n_pairs' share of split ranges)
  int BH, sms;
  int* counts;                // [n_pairs] live key tiles of each Q-tile pair (scratch)
  int4* plan;                 // [n_pairs + extra]
  int* merge_count;           // [BH][n_slots], zeroed
  uint32_t* pair_bits;        // [n_pairs][words]: bit j of a pair's row = key tile j is live
  int words;                  // (T + 31) / 32
  int* next_unit;             // zeroed: the persistent forward's unit counter
};

struct SplitMergeArgs {       // combines the split-KV partials with the (m, l, u) merge law
  const float* o_part;
  const float* lse_part;
  void* o;
  float* lse;
  int rows;                   // B * H * N
  int d;
  int n_splits;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;    // workspace: fp32 [B, H, N, d]; null in the two-pass backward
  float* delta;     // workspace: fp32 [B, H, N], D_i = rowsum(dO_i * O_i)
  int B, H, N, d;
  int Hkv;          // key/value heads (K, V, dK, dV are [B, Hkv, N, d])
  float scale;
  int causal;
  const uint8_t* block_mask;
  int n_tiles;
  const int32_t* kv_lens;
  int* err;
  DebugKnobs dbg;
  int heads_fastest;          // launch order: (b, h) slice fastest (unequal work per tile)
  const int32_t* cu_seqlens;  // packed sequences, as in FwdArgs
  int rows;
  DropoutArgs drop;
  // Order of the two-pass backward's units under a tile mask: CTA x runs the unit that CTA
  // perm[x] runs without a plan (dK/dV units of key tile j at j*B*Hkv + slice, then dQ units).
  // Null: that order itself.
  const int* perm;
};

// The unit order of the two-pass backward under a tile mask (see BwdArgs::order).
struct OrderArgs {
  const uint8_t* block_mask;  // [T, T]
  int T, causal;
  int BH, BHkv;               // query slices, key/value slices
  int* counts;                // [2T] live tiles of key tile j (first T), of query tile i (next T)
  int* rank;                  // [2T] scratch
  int2* order;                // [2T] scratch: {kind, tile} in launch order
  int* order_off;             // [2T + 1] scratch: first CTA of each entry
  int* perm;                  // [T * (BHkv + BH)]
};

// Rows of the query-side tensors (Q, O, dO, dQ, LSE, D) over all slices.
__host__ __device__ inline size_t q_rows_total(const BwdArgs& a) {
  return a.cu_seqlens != nullptr ? (size_t)a.H * a.rows : (size_t)a.B * a.H * a.N;
}

// One packed sequence: its first row on the token axis and its length; false when the offsets
// break the documented contract (then nothing of that sequence is read or written).
__device__ __forceinline__ bool packed_sequence(const int32_t* cu, int b, int max_len, int rows,
                                                int* row0, int* len) {
  const int r0 = cu[b], r1 = cu[b + 1];
  *row0 = r0;
  *len = r1 - r0;
  return r0 >= 0 && r1 >= r0 && r1 - r0 <= max_len && r1 <= rows;
}

// CUDA-core (SIMT) kernels: the fp32 path.
cudaError_t launch_fwd_simt(const FwdArgs& a, fa_dtype dt, cudaStream_t s);
cudaError_t launch_bwd_simt(const BwdArgs& a, fa_dtype dt, cudaStream_t s);

// Shared backward pieces: D = rowsum(dO * O) with dQ accumulator zeroing (when there is an
// accumulator), and the final dQ scale + convert.
cudaError_t launch_bwd_preprocess(const BwdArgs& a, fa_dtype dt, cudaStream_t s);
cudaError_t launch_bwd_dq_convert(const BwdArgs& a, fa_dtype dt, cudaStream_t s);

// Split-KV merge: O = sum_s w_s O_s / sum_s w_s, LSE = m + ln sum_s w_s, w_s = exp(LSE_s - m).
cudaError_t launch_splitkv_merge(const SplitMergeArgs& m, fa_dtype dt, cudaStream_t s);

// Live key tiles per Q-tile pair of a tile mask, then the split plan (fa_plan.cu).
cudaError_t launch_blocksparse_plan(const PlanArgs& p, cudaStream_t s);

// Live tiles per key tile and per query tile of a tile mask, then the backward's unit order.
cudaError_t launch_backward_order(const OrderArgs& p, cudaStream_t s);

// Bytes of the backward's unit-order buffers for N keys and BH slices (a multiple of 256).
inline size_t backward_order_bytes(size_t BH, int N) {
  const size_t T = (size_t)(N + 127) / 128;
  const size_t ints = 2 * T + 2 * T + 4 * T + (2 * T + 1) + 2 * T * BH;
  return (ints * sizeof(int) + 255) / 256 * 256;
}

}  // namespace fa
