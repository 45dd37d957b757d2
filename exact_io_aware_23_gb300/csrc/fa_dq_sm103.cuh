// dQ pass of the deterministic attention backward for sm_103a (bf16 or fp16 in, fp32 accumulate),
// d in {64, 128}.
//
// The backward recomputes P from the stored per-row statistic ("FlashAttention paper story",
// backward paragraph; "FlashAttention: Exact Attention with Less GPU Memory", "Tiling, and
// paying arithmetic to avoid memory").  For dQ of one query row i:
//     P_ij = exp(scale*S_ij - LSE_i),  dP_ij = dO_i . V_j,  dS_ij = P_ij (dP_ij - D_i),
//     dQ_i = scale * sum_j dS_ij K_j.
// The key-stationary kernel (fa_bwd_sm103.cu) adds each key tile's share of dQ into an fp32
// workspace from many CTAs at once, so the order of the additions (and the last bits of dQ)
// depends on scheduling.  Here one CTA owns a 128-row query tile and visits its live key tiles in
// ascending order, accumulating dQ in TMEM: the result is the same bits on every run.  The cost
// is recomputing S and dP (two more products per tile pair than the fused kernel spends on dQ).
//
// GB300 design: one CTA per 128-row query tile of one (b, h) slice: kWG compute warpgroups
// (BwdLayout: four at d = 64, two at d = 128), then the two warps below.
//   producer    TMA producer: Q_i and dO_i once; K_j and V_j through two rings.  V_j is free
//               once dP has read it, K_j only after dQ has: the K ring is the deeper one, so the
//               next K tile is loaded a whole tile ahead of the product that needs it.
//   MMA warp    MMA issuer: S = Q_i K_j^T into one of two S buffers (SS); dQ += dS K_{j-1}
//               for the previous tile (TS: dS read from TMEM, K MN-major in shared memory),
//               then dP = dO_i V_j^T (SS).  The tensor pipe runs the next tile's S while the
//               compute warps work on this one.
//   compute     warpgroup w over the tile's keys [w*c, (w+1)*c), c = 128 / kWG; thread = query
//               row = TMEM lane.  P from S (exp2 of scale*log2e*S - LSE*log2e), dS = P (dP - D)
//               packed to bf16/fp16 pairs into the first c/2 columns of the warpgroup's own c
//               S columns (no other warp reads them).  At the end the warpgroups convert dQ's
//               columns, 32 or more each, and store them.
//   TMEM: dQ [0,128) (d columns used), S buffers [128,256) and [256,384), dP [384,512).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "dropout_sm103.cuh"
#include "fa_internal.cuh"
#include "fa_sm103.cuh"
#include "ptx_sm103.cuh"

namespace fa {
namespace dqp {

constexpr int BM = 128;          // query rows per CTA
constexpr int BN = 128;          // keys per tile
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool F16>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;                  // one 128-row operand tile
  static constexpr int kKSlots = D == 64 ? 4 : 3;            // K ring
  static constexpr int kVSlots = D == 64 ? 4 : 2;            // V ring
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kK = kDO + kTile;                     // K slot s at kK + s*kTile
  static constexpr int kV = kK + kKSlots * kTile;            // V slot s at kV + s*kTile
  static constexpr int kBar = kV + kVSlots * kTile;
  static constexpr int kSmem = kBar + 256;
  static constexpr uint32_t kDQ = 0, kS = 128, kDP = 384;    // TMEM columns; S buffer b at kS + 128b
  static constexpr uint32_t kIdescS = ptx::idesc_f32acc(128, 128, false, false, F16);  // S, dP
  static constexpr uint32_t kIdescDQ = ptx::idesc_f32acc(128, D, false, true, F16);    // dQ
};

struct Bars {             // at most 256 bytes (the live-tile bitmap follows)
  uint64_t q_full;
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[4];
  uint64_t v_empty[4];
  uint64_t s_full[2];
  uint64_t dp_full;
  uint64_t ds_ready;
  uint64_t dq_done;
  uint32_t tmem_base;
};

static_assert(sizeof(Bars) <= 256, "the live-tile bitmap starts 256 bytes after the barriers");

enum : int { kNone = 0, kPartial = 1, kFull = 2 };

// Key tiles of one query tile: [0, j_end) bounded by the causal diagonal and the valid key
// length; a tile mask removes more (then `bits` lists the live ones).
struct Geo {
  int i, q0, N, kv_lim, causal, T, j_end;
  const uint8_t* bm;
  const uint32_t* bits;
  __device__ int kind(int j) const {
    const int r0 = q0, r1 = min(q0 + BM, N) - 1;
    const int c0 = j * BN, c1 = c0 + BN - 1;
    if (bm != nullptr && bm[(size_t)i * T + j] == 0) return kNone;
    if (c0 >= kv_lim || (causal && c0 > r1)) return kNone;
    if (c1 < kv_lim && (!causal || c1 <= r0)) return kFull;
    return kPartial;
  }
  __device__ int next(int j) const {
    if (bits == nullptr) return j;
    while (j < j_end) {
      const uint32_t w = bits[j >> 5] >> (j & 31);
      if (w != 0u) return min(j + __ffs(w) - 1, j_end);
      j = (j | 31) + 1;
    }
    return j_end;
  }
};

template <int D, bool F16, bool kDrop>
__device__ __forceinline__ void run(const int unit, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const CUtensorMap& tmDO,
                                    const BwdArgs& a) {
  using C = Cfg<D, F16>;
  using L = BwdLayout<D>;
  constexpr int kCols = L::kCols;                // keys per compute warpgroup
  constexpr int kNR = kCols / 32;                // 32-column TMEM loads per operand
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {      // the operand tiles need 1 KB alignment
    if (threadIdx.x == 0) atomicExch(a.err, 2);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  // Work order: with masks the (b, h) slice varies fastest and, when causal, the longest query
  // tiles (the last ones) start first; without, one slice's tiles run together and share its
  // K/V stream in L2.
  const int BH = a.B * a.H;
  const int n_qt = (a.N + BM - 1) / BM;
  const int bh = a.heads_fastest ? unit % BH : unit / n_qt;
  const int it = a.heads_fastest ? unit / BH : unit % n_qt;
  const int b = bh / a.H, h = bh % a.H;
  const uint32_t lim_ms = a.dbg.wait_limit_ms;

  Geo g;
  g.i = a.causal ? n_qt - 1 - it : it;
  g.q0 = g.i * BM;
  int row0 = 0, len = a.N;                       // this slice's rows on the token axis
  if (a.cu_seqlens != nullptr) {
    // Packed sequences: the grid is sized for the longest one; query tiles past this sequence's
    // end have nothing to do, and offsets outside the contract are reported, not followed.
    if (!packed_sequence(a.cu_seqlens, b, a.N, a.rows, &row0, &len)) {
      if (threadIdx.x == 0) atomicExch(a.err, kDevBadOffsets);
      return;
    }
    if (g.q0 >= len) return;
  }
  const int qs = a.cu_seqlens != nullptr ? h : bh;                              // Q, dO, dQ slice
  // grouped-query attention: query head h reads key/value head h / (H / Hkv)
  const int ks = (a.cu_seqlens != nullptr ? 0 : b * a.Hkv) + h / (a.H / a.Hkv);  // K, V slice
  g.N = len;
  int kvl = len;
  if (a.kv_lens != nullptr) kvl = max(0, min(a.N, (int)a.kv_lens[b]));
  g.kv_lim = kvl;
  g.causal = a.causal;
  g.T = a.n_tiles;
  g.bm = a.block_mask;
  g.j_end = (kvl + BN - 1) / BN;
  if (a.causal) g.j_end = min(g.j_end, g.i + 1);

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
    for (int s = 0; s < C::kKSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->k_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->k_empty[s]), 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->v_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->v_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_ready), L::kComputeWarps);
    ptx::mbar_init(ptx::smem_u32(&bars->dq_done), 1);
    ptx::fence_mbar_init();
  }
  if (warp == L::kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  g.bits = nullptr;
  if (a.block_mask != nullptr) {                 // live-tile bitmap, one ballot per 32 tiles
    uint32_t* live_bits = reinterpret_cast<uint32_t*>(smem + C::kBar + 256);
    g.bits = live_bits;
    for (int w = warp; w < (g.j_end + 31) / 32; w += L::kThreads / 32) {
      const int j = w * 32 + lane;
      const uint32_t word = __ballot_sync(0xffffffffu, j < g.j_end && g.kind(j) != kNone);
      if (lane == 0) live_bits[w] = word;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const bool any = g.next(0) < g.j_end;

  if (warp == L::kProducerWarp) {
    // ------------------------------- TMA producer -----------------------------------------------
    if (lane == 0 && any) {
      bool ok = true;
      int n = 0;
      const uint32_t qb = ptx::smem_u32(&bars->q_full);
      ptx::mbar_arrive_expect_tx(qb, 2 * C::kTile);
      for (int hh = 0; hh < D / 64; ++hh) {
        ptx::tma_load_3d(sbase + C::kQ + hh * 128 * 128, &tmQ, qb, hh * 64, row0 + g.q0, qs);
        ptx::tma_load_3d(sbase + C::kDO + hh * 128 * 128, &tmDO, qb, hh * 64, row0 + g.q0, qs);
      }
      for (int j = g.next(0); j < g.j_end && ok; j = g.next(j + 1), ++n) {
        const int kslot = n % C::kKSlots, vslot = n % C::kVSlots;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->k_empty[kslot]), ((uint32_t)(n / C::kKSlots) & 1u) ^ 1u,
                            lim_ms, a.err);
        if (!ok) break;
        const uint32_t kb = ptx::smem_u32(&bars->k_full[kslot]);
        ptx::mbar_arrive_expect_tx(kb, C::kTile);
        for (int hh = 0; hh < D / 64; ++hh)
          ptx::tma_load_3d(sbase + C::kK + kslot * C::kTile + hh * 128 * 128, &tmK, kb, hh * 64, row0 + j * BN, ks);
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->v_empty[vslot]), ((uint32_t)(n / C::kVSlots) & 1u) ^ 1u,
                            lim_ms, a.err);
        if (!ok) { ++n; break; }
        const uint32_t vb = ptx::smem_u32(&bars->v_full[vslot]);
        ptx::mbar_arrive_expect_tx(vb, C::kTile);
        for (int hh = 0; hh < D / 64; ++hh)
          ptx::tma_load_3d(sbase + C::kV + vslot * C::kTile + hh * 128 * 128, &tmV, vb, hh * 64, row0 + j * BN, ks);
      }
      // drain: copies in flight must land before shared memory is released
      ptx::mbar_wait(qb, 0, lim_ms, a.err);
      for (int m = max(0, n - C::kKSlots); m < n; ++m)
        ptx::mbar_wait(ptx::smem_u32(&bars->k_full[m % C::kKSlots]), (uint32_t)(m / C::kKSlots) & 1u,
                       lim_ms, a.err);
      for (int m = max(0, n - C::kVSlots); m < n; ++m)
        ptx::mbar_wait(ptx::smem_u32(&bars->v_full[m % C::kVSlots]), (uint32_t)(m / C::kVSlots) & 1u,
                       lim_ms, a.err);
    }
  } else if (warp == L::kMmaWarp) {
    // ------------------------------- MMA issuer -------------------------------------------------
    if (lane == 0) {
      bool ok = true;
      int n = 0;
      // dQ += dS(m) K(m): A = dS packed in S buffer m&1 (keys c*w .. c*w+c-1 in its columns
      // c*w .. c*w+c/2-1), B = K_m with the key index as K (MN-major, 16 keys = 2048 bytes a
      // step)
      auto dq_mma = [&](int m) {
        constexpr int kSteps = kCols / 16;           // k-steps per warpgroup's columns
        const uint32_t sb = C::kS + (uint32_t)(m & 1) * 128;
        const uint32_t sk = sbase + C::kK + (m % C::kKSlots) * C::kTile;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_ts(tmem + C::kDQ, tmem + sb + (kk / kSteps) * kCols + (kk % kSteps) * 8,
                      ptx::sdesc_sw128(sk + kk * 2048, 128 * 128, 1024), C::kIdescDQ,
                      (m > 0 || kk > 0) ? 1u : 0u);
      };
      if (any) {
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_full), 0, lim_ms, a.err);
        for (int j = g.next(0); j < g.j_end && ok; j = g.next(j + 1), ++n) {
          const int kslot = n % C::kKSlots, vslot = n % C::kVSlots;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->k_full[kslot]), (uint32_t)(n / C::kKSlots) & 1u,
                              lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t sk = sbase + C::kK + kslot * C::kTile;
          // S(n) = Q K_j^T (K-major operands, k-steps of 16 along d).  Its buffer last held
          // dS(n-2), read by dQ(n-2), which was issued before this.
          const uint32_t sb = C::kS + (uint32_t)(n & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            ptx::mma_ss(tmem + sb, ptx::sdesc_sw128(sbase + C::kQ + off, 16, 1024),
                        ptx::sdesc_sw128(sk + off, 16, 1024), C::kIdescS, kk > 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->s_full[n & 1]));
          if (n > 0) {
            // tile n-1 done by the compute warps: dS(n-1) is in TMEM and dP(n-1) has been read
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->ds_ready), (uint32_t)(n - 1) & 1u, lim_ms, a.err);
            if (!ok) break;
            ptx::tc_fence_after();
            dq_mma(n - 1);
          }
          // dP(n) = dO V_j^T.  No commit frees V_j or K_{j-1}: dP(n) is issued after every product
          // that reads them, so the compute warps, on seeing dP(n), free both (a commit stalls
          // the tensor pipe for about as long as one MMA).
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->v_full[vslot]), (uint32_t)(n / C::kVSlots) & 1u,
                              lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t sv = sbase + C::kV + vslot * C::kTile;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            ptx::mma_ss(tmem + C::kDP, ptx::sdesc_sw128(sbase + C::kDO + off, 16, 1024),
                        ptx::sdesc_sw128(sv + off, 16, 1024), C::kIdescS, kk > 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->dp_full));
        }
        if (ok && n > 0) {
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->ds_ready), (uint32_t)(n - 1) & 1u, lim_ms, a.err);
          if (ok) {
            ptx::tc_fence_after();
            dq_mma(n - 1);
          }
        }
      }
      ptx::mma_commit(ptx::smem_u32(&bars->dq_done));
      ptx::mbar_wait(ptx::smem_u32(&bars->dq_done), 0, lim_ms, a.err);
    }
  } else {
    // ------------------------------- compute warpgroups -----------------------------------------
    const int wg = warp / 4, sub = warp % 4;
    const int r = sub * 32 + lane;                   // query row within the tile (TMEM lane)
    const int q = g.q0 + r;
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const float c = a.scale * kLog2e;
    const float2 c2 = make_float2(c, c);
    const size_t row = (size_t)qs * a.rows + row0 + q;
    float L = q < g.N ? a.lse[row] : -INFINITY;
    const float nl = L == -INFINITY ? -INFINITY : -L * kLog2e;   // P vanishes on empty rows
    const float2 nl2 = make_float2(nl, nl);
    const float dd = q < g.N ? a.delta[row] : 0.f;
    const float2 dd2 = make_float2(dd, dd);
    bool ok = true;
    int n = 0;
    const uint32_t tq = (uint32_t)lane & 3u;         // this row within its 4-row dropout block
    DropTest dtest{};
    if constexpr (kDrop) dtest = drop_test(a.drop);
    for (int j = g.next(0); j < g.j_end; j = g.next(j + 1), ++n) {
      const int kind = g.kind(j);
      const int k0 = j * BN + wg * kCols;           // first key of this warpgroup's columns
      const uint32_t sb = C::kS + (uint32_t)(n & 1) * 128 + wg * kCols;
      // dropout: this row's drop flags over the warpgroup's keys, 16 per word (generated while
      // the scores are still being computed; the quad shares its calls)
      uint32_t flags[kCols / 16];
      if constexpr (kDrop) {
#pragma unroll
        for (int m = 0; m < kCols / 16; ++m) {
          const uint4 r = philox4x32_10((uint32_t)(k0 / 4) + 4u * m + tq, (uint32_t)q >> 2, (uint32_t)bh,
                                        a.drop.offset, a.drop);
          flags[m] = gather_row_flags(pack_flags(r, dtest), tq);
        }
      }
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_full[n & 1]), (uint32_t)(n >> 1) & 1u, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      float p[kCols];
      {
        uint32_t raw[kNR][32];
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) ptx::tmem_ld32(tmem + lane_off + sb + hc * 32, raw[hc]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) {
          ptx::reg_fence(raw[hc]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = hc * 32 + e;
            const float2 x = ptx::fma2(make_float2(__uint_as_float(raw[hc][e]), __uint_as_float(raw[hc][e + 1])),
                                       c2, nl2);
            float v0 = ptx::ex2(x.x), v1 = ptx::ex2(x.y);
            if (kind == kPartial) {
              const int key = k0 + col;
              v0 = (key < g.kv_lim && (!g.causal || key <= q)) ? v0 : 0.f;
              v1 = (key + 1 < g.kv_lim && (!g.causal || key + 1 <= q)) ? v1 : 0.f;
            }
            p[col] = v0;
            p[col + 1] = v1;
          }
        }
      }
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), (uint32_t)n & 1u, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      if (warp == 0 && lane == 0) {
        // dP(n) has completed, and with it every MMA issued before it: V_j is free, and so is
        // K_{j-1} (its dQ product came before dP(n))
        ptx::mbar_arrive(ptx::smem_u32(&bars->v_empty[n % C::kVSlots]));
        if (n > 0) ptx::mbar_arrive(ptx::smem_u32(&bars->k_empty[(n - 1) % C::kKSlots]));
      }
      {
        uint32_t raw[kNR][32];
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) ptx::tmem_ld32(tmem + lane_off + C::kDP + wg * kCols + hc * 32, raw[hc]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) {
          ptx::reg_fence(raw[hc]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = hc * 32 + e;
            float2 dpv = make_float2(__uint_as_float(raw[hc][e]), __uint_as_float(raw[hc][e + 1]));
            if constexpr (kDrop) {                   // dP = (dO V^T) * M * 256/k8
              const uint32_t x = flags[col / 16] << ((((uint32_t)col >> 2) & 3u) ^ tq);
              dpv.x = __uint_as_float(raw[hc][e] & ~row_elem_mask(x, col & 3));
              dpv.y = __uint_as_float(raw[hc][e + 1] & ~row_elem_mask(x, (col & 3) + 1));
              dpv = ptx::mul2(dpv, make_float2(a.drop.scale, a.drop.scale));
            }
            const float2 dpd = ptx::sub2(dpv, dd2);
            const float2 ds = ptx::mul2(make_float2(p[col], p[col + 1]), dpd);
            p[col] = ds.x;
            p[col + 1] = ds.y;
          }
        }
      }
      {
        uint32_t pk[kCols / 2];
#pragma unroll
        for (int e = 0; e < kCols / 2; ++e) pk[e] = ptx::pack2<F16>(p[2 * e], p[2 * e + 1]);
        ptx::tmem_st(tmem + lane_off + sb, pk);
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ds_ready));
    }
    // ------------------------------- epilogue: dQ = scale * acc, 32 or more columns a warpgroup -
    const bool have = ok && n > 0;
    if (have) {
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->dq_done), 0, lim_ms, a.err);
      ptx::tc_fence_after();
    }
    constexpr int kOutCols = D / L::kWG < 32 ? 32 : D / L::kWG;   // at d = 64 with four, two idle
    const int c0 = wg * kOutCols;
    uint16_t* out = static_cast<uint16_t*>(a.dq) + row * D + c0;
#pragma unroll 1
    for (int hc = 0; hc < (c0 < D ? kOutCols / 32 : 0); ++hc) {
      uint32_t raw[32];
      if (have && ok) {
        ptx::tmem_ld32(tmem + lane_off + C::kDQ + c0 + hc * 32, raw);
        ptx::tmem_wait_ld();
        ptx::reg_fence(raw);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) raw[e] = 0u;
      }
      if (q < g.N) {
        uint4* dst = reinterpret_cast<uint4*>(out + hc * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint4 w;
          w.x = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 0]) * a.scale, __uint_as_float(raw[8 * v4 + 1]) * a.scale);
          w.y = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 2]) * a.scale, __uint_as_float(raw[8 * v4 + 3]) * a.scale);
          w.z = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 4]) * a.scale, __uint_as_float(raw[8 * v4 + 5]) * a.scale);
          w.w = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 6]) * a.scale, __uint_as_float(raw[8 * v4 + 7]) * a.scale);
          dst[v4] = w;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == L::kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace dqp
}  // namespace fa
