// dK/dV pass of the deterministic attention backward for sm_103a (bf16 or fp16 in, fp32
// accumulate), d in {64, 128}.
//
// The backward recomputes P from the stored per-row statistic ("FlashAttention paper story",
// backward paragraph; "FlashAttention: Exact Attention with Less GPU Memory", "Tiling, and
// paying arithmetic to avoid memory").  For one key tile j, over every live query tile i:
//     P^T = exp(scale*S^T - LSE),  dV_j += P^T dO_i,  dP^T = V_j dO_i^T,
//     dS^T = P^T * (dP^T - D),     dK_j += scale * dS^T Q_i.
// dQ is left to the query-stationary kernel (fa_dq_sm103.cu), so nothing here is added from
// several CTAs and the results do not depend on scheduling.
//
// GB300 design: one CTA per 128-key tile of one (b, h) key/value slice, visiting every live
// query tile of every query head that reads the slice (one, or the G heads of a group under
// grouped-query attention).  Key rows sit on the TMEM lanes: a thread owns one key.  kWG compute
// warpgroups (BwdLayout: four at d = 64, two at d = 128) then the two warps below.
//   producer    TMA producer: K_j, V_j once; Q_i through a three-slot ring and dO_i through a
//               two-slot ring (a Q tile is read until dK, a dO tile only until dV), and the
//               tile's -LSE*log2(e) and D vectors through a two-slot ring in shared memory.
//   MMA warp    MMA issuer, one thread, in the order
//                   dV += P^T(n) dO_n,  S^T(n+1) = K Q_{n+1}^T,  dK += dS^T(n) Q_n,
//                   dP^T(n+1) = V dO_{n+1}^T
//               so the tensor pipe computes the next tile's S^T while the compute warps build
//               dS^T(n), and dK(n), dP^T(n+1) while they build P^T(n+1).
//   compute     warpgroup w over the tile's query columns [w*c, (w+1)*c), c = 128 / kWG: P^T
//               and dS^T in registers, packed to bf16/fp16 pairs into the first c/2 columns of
//               the warpgroup's own c columns of X and Y (no other warp reads those).
//   TMEM: dV [0,d), dK [d,2d), X = S^T / P^T [2d, 2d+128), Y = dP^T / dS^T [2d+128, 2d+256).
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
namespace dkdv {

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per CTA
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool F16>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;                  // one 128-row operand tile
  static constexpr int kQSlots = D == 64 ? 4 : 3;
  static constexpr int kOSlots = D == 64 ? 4 : 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;                      // Q slot s at kQ + s*kTile
  static constexpr int kO = kQ + kQSlots * kTile;            // dO slot s at kO + s*kTile
  static constexpr int kVec = kO + kOSlots * kTile;          // vector slot s: lse2[128], delta[128]
  static constexpr int kBar = kVec + 2 * 1024;
  static constexpr int kSmem = kBar + 256;
  // TMEM columns.  At d = 64 the accumulators leave room for a second S^T buffer, so S^T(n+1)
  // is computed while the compute warps still work on tile n (X0/X1 alternate); at d = 128 the
  // 512 columns hold dV, dK, one X and Y.
  static constexpr bool kXDouble = D == 64;
  static constexpr uint32_t kDV = 0, kDK = D, kX0 = 2 * D, kX1 = kXDouble ? 2 * D + 128 : 2 * D;
  static constexpr uint32_t kY = kXDouble ? 2 * D + 256 : 2 * D + 128;
  static __device__ __forceinline__ uint32_t x_col(int n) { return (n & 1) ? kX1 : kX0; }
  static constexpr uint32_t kIdescST = ptx::idesc_f32acc(128, 128, false, false, F16);  // S^T, dP^T
  static constexpr uint32_t kIdescAcc = ptx::idesc_f32acc(128, D, false, true, F16);    // dV, dK
};

struct Bars {             // at most 256 bytes (the live-tile bitmap follows)
  uint64_t kv_full;
  uint64_t q_full[4];
  uint64_t q_empty[4];
  uint64_t o_full[4];
  uint64_t o_empty[4];
  uint64_t vec_full[2];
  uint64_t vec_empty[2];
  uint64_t s_full[2];     // S^T(n) in TMEM: barrier n & 1, phase n >> 1
  uint64_t dp_full;
  uint64_t p_ready;
  uint64_t ds_ready;
  uint64_t acc_done;
  uint32_t tmem_base;
};

static_assert(sizeof(Bars) <= 256, "the live-tile bitmap starts 256 bytes after the barriers");

enum : int { kNone = 0, kPartial = 1, kFull = 2 };

// Query tiles of one key tile: [i_begin, i_end) bounded by the causal diagonal and the valid key
// length; a tile mask removes more (then `bits` lists the live ones).
struct Geo {
  int k0, N, kv_lim, causal, T;
  const uint8_t* bm;
  int i_begin, i_end;
  const uint32_t* bits;
  __device__ int kind(int i) const {
    const int r0 = i * BM, r1 = min(r0 + BM, N) - 1;
    const int c0 = k0, c1 = k0 + BN - 1;
    if (bm != nullptr && bm[(size_t)i * T + k0 / BN] == 0) return kNone;
    if (c0 >= kv_lim || (causal && c0 > r1)) return kNone;
    if (c1 < kv_lim && (!causal || c1 <= r0)) return kFull;
    return kPartial;
  }
  __device__ int next(int i) const {
    if (bits == nullptr) return i;
    while (i < i_end) {
      const uint32_t w = bits[i >> 5] >> (i & 31);
      if (w != 0u) return min(i + __ffs(w) - 1, i_end);
      i = (i | 31) + 1;
    }
    return i_end;
  }
};

template <int D, bool F16, bool kDrop>
__device__ __forceinline__ void run(const int unit, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                    const CUtensorMap& tmV, const CUtensorMap& tmDO,
                                    const BwdArgs& a) {
  using C = Cfg<D, F16>;
  using L = BwdLayout<D>;
  constexpr int kCols = L::kCols;                // query columns per compute warpgroup
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {      // the operand tiles need 1 KB alignment
    if (threadIdx.x == 0) atomicExch(a.err, 2);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  // Work order: with masks the key/value slice varies fastest, so every slice's heaviest key
  // tiles (the first ones when causal) run in the first waves; without, one slice's key tiles
  // run together and share its Q/dO stream in L2.
  const int BH = a.B * a.Hkv;
  const int n_kt = (a.N + BN - 1) / BN;
  const int bh = a.heads_fastest ? unit % BH : unit / n_kt;   // K/V slice
  const int jt = a.heads_fastest ? unit / BH : unit % n_kt;   // key tile
  const int b = bh / a.Hkv, hk = bh % a.Hkv;
  const int G = a.H / a.Hkv;
  int row0 = 0, len = a.N;                       // this slice's rows on the token axis
  if (a.cu_seqlens != nullptr) {
    // Packed sequences: the grid is sized for the longest one; key tiles past this sequence's
    // end have nothing to do, and offsets outside the contract are reported, not followed.
    if (!packed_sequence(a.cu_seqlens, b, a.N, a.rows, &row0, &len)) {
      if (threadIdx.x == 0) atomicExch(a.err, kDevBadOffsets);
      return;
    }
    if (jt * BN >= len) return;
  }
  const int ks = a.cu_seqlens != nullptr ? hk : bh;                            // K, V, dK, dV slice
  const int bhq0 = (a.cu_seqlens != nullptr ? 0 : b * a.H) + hk * G;            // first query slice
  const uint32_t lim_ms = a.dbg.wait_limit_ms;

  Geo g;
  g.k0 = jt * BN;
  g.N = len;
  int kvl = len;
  if (a.kv_lens != nullptr) kvl = max(0, min(a.N, (int)a.kv_lens[b]));
  g.kv_lim = kvl;
  g.causal = a.causal;
  g.T = a.n_tiles;
  g.bm = a.block_mask;
  g.i_begin = a.causal ? jt : 0;
  g.i_end = g.k0 < g.kv_lim ? (len + BM - 1) / BM : 0;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->kv_full), 1);
    for (int s = 0; s < C::kQSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->q_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->q_empty[s]), 1);
    }
    for (int s = 0; s < C::kOSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->o_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->o_empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->vec_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->vec_full[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->vec_empty[0]), L::kComputeWarps);
    ptx::mbar_init(ptx::smem_u32(&bars->vec_empty[1]), L::kComputeWarps);
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->s_full[1]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->p_ready), L::kComputeWarps);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_ready), L::kComputeWarps);
    ptx::mbar_init(ptx::smem_u32(&bars->acc_done), 1);
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
    for (int w = warp; w < (g.i_end + 31) / 32; w += L::kThreads / 32) {
      const int i = w * 32 + lane;
      const uint32_t word = __ballot_sync(0xffffffffu, i >= g.i_begin && i < g.i_end && g.kind(i) != kNone);
      if (lane == 0) live_bits[w] = word;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int n_live = 0;                                // live query tiles of one head
  for (int i = g.next(g.i_begin); i < g.i_end; i = g.next(i + 1)) ++n_live;
  const int total = n_live * G;                  // tiles this CTA visits

  if (warp == L::kProducerWarp) {
    // ------------------------------- producer (whole warp) --------------------------------------
    if (total > 0) {
      bool ok = true;
      int n = 0;
      if (lane == 0) {
        const uint32_t kb = ptx::smem_u32(&bars->kv_full);
        ptx::mbar_arrive_expect_tx(kb, 2 * C::kTile);
        for (int hh = 0; hh < D / 64; ++hh) {
          ptx::tma_load_3d(sbase + C::kK + hh * 128 * 128, &tmK, kb, hh * 64, row0 + g.k0, ks);
          ptx::tma_load_3d(sbase + C::kV + hh * 128 * 128, &tmV, kb, hh * 64, row0 + g.k0, ks);
        }
      }
      // Per tile: start the Q and dO copies first, then fetch the tile's vectors (plain loads,
      // whose latency then overlaps the copies').  nq / no count the copies started, for the drain.
      int nq = 0, no = 0;
      for (int hg = 0; hg < G && ok; ++hg)
      for (int i = g.next(g.i_begin); i < g.i_end && ok; i = g.next(i + 1), ++n) {
        const int bhq = bhq0 + hg;
        const int qs = n % C::kQSlots, os = n % C::kOSlots, vs = n & 1;
        if (lane == 0) {
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_empty[qs]), ((uint32_t)(n / C::kQSlots) & 1u) ^ 1u,
                              lim_ms, a.err);
          if (ok) {
            const uint32_t qb = ptx::smem_u32(&bars->q_full[qs]);
            ptx::mbar_arrive_expect_tx(qb, C::kTile);
            for (int hh = 0; hh < D / 64; ++hh)
              ptx::tma_load_3d(sbase + C::kQ + qs * C::kTile + hh * 128 * 128, &tmQ, qb, hh * 64, row0 + i * BM, bhq);
            ++nq;
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->o_empty[os]), ((uint32_t)(n / C::kOSlots) & 1u) ^ 1u,
                                lim_ms, a.err);
          }
          if (ok) {
            const uint32_t ob = ptx::smem_u32(&bars->o_full[os]);
            ptx::mbar_arrive_expect_tx(ob, C::kTile);
            for (int hh = 0; hh < D / 64; ++hh)
              ptx::tma_load_3d(sbase + C::kO + os * C::kTile + hh * 128 * 128, &tmDO, ob, hh * 64, row0 + i * BM, bhq);
            ++no;
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->vec_empty[vs]), ((uint32_t)(n >> 1) & 1u) ^ 1u,
                                lim_ms, a.err);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // -LSE as a log2-domain bias (-inf where P must vanish) and D for the tile's rows
        float* lse2 = reinterpret_cast<float*>(smem + C::kVec + vs * 1024);
        float* dl = lse2 + 128;
        // all eight loads of a lane first (the stores below could alias them as far as the
        // compiler knows, which would otherwise serialise four round trips to memory)
        float Lv[4], Dv[4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int q = i * BM + lane + 32 * k4;
          const size_t row = (size_t)bhq * a.rows + row0 + q;
          Lv[k4] = q < g.N ? __ldg(a.lse + row) : -INFINITY;
          Dv[k4] = q < g.N ? __ldg(a.delta + row) : 0.f;
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          lse2[lane + 32 * k4] = Lv[k4] == -INFINITY ? -INFINITY : -Lv[k4] * kLog2e;
          dl[lane + 32 * k4] = Dv[k4];
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->vec_full[vs]));
      }
      if (lane == 0) {   // drain: copies in flight must land before shared memory is released
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full), 0, lim_ms, a.err);
        for (int m = max(0, nq - C::kQSlots); m < nq; ++m)
          ptx::mbar_wait(ptx::smem_u32(&bars->q_full[m % C::kQSlots]), (uint32_t)(m / C::kQSlots) & 1u,
                         lim_ms, a.err);
        for (int m = max(0, no - C::kOSlots); m < no; ++m)
          ptx::mbar_wait(ptx::smem_u32(&bars->o_full[m % C::kOSlots]), (uint32_t)(m / C::kOSlots) & 1u,
                         lim_ms, a.err);
      }
    }
  } else if (warp == L::kMmaWarp) {
    // ------------------------------- MMA issuer -------------------------------------------------
    if (lane == 0) {
      // S^T = K Q^T into X, dP^T = V dO^T into Y (K-major operands, k-steps of 16 along d)
      auto st_mma = [&](uint32_t dst, uint32_t src_kv, uint32_t src_q) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
          ptx::mma_ss(tmem + dst, ptx::sdesc_sw128(src_kv + off, 16, 1024),
                      ptx::sdesc_sw128(src_q + off, 16, 1024), C::kIdescST, kk > 0);
        }
      };
      // acc (+)= A^T-tile from TMEM x B: A = P^T or dS^T packed in X or Y (queries c*w ..
      // c*w+c-1 in columns c*w .. c*w+c/2-1), B = dO or Q with the query index as K (MN-major,
      // 16 queries = 2048 bytes per step)
      auto acc_mma = [&](uint32_t acc, uint32_t src, uint32_t sb, bool first) {
        constexpr int kSteps = kCols / 16;           // k-steps per warpgroup's columns
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          ptx::mma_ts(tmem + acc, tmem + src + (kk / kSteps) * kCols + (kk % kSteps) * 8,
                      ptx::sdesc_sw128(sb + kk * 2048, 128 * 128, 1024), C::kIdescAcc,
                      (!first || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      if (total > 0) {
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full), 0, lim_ms, a.err);
        if (ok) ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_full[0]), 0, lim_ms, a.err);
        if (ok) {
          ptx::tc_fence_after();
          st_mma(C::x_col(0), sbase + C::kK, sbase + C::kQ);
          ptx::mma_commit(ptx::smem_u32(&bars->s_full[0]));
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->o_full[0]), 0, lim_ms, a.err);
        }
        if (ok) {
          ptx::tc_fence_after();
          st_mma(C::kY, sbase + C::kV, sbase + C::kO);
          ptx::mma_commit(ptx::smem_u32(&bars->dp_full));
        }
        for (int n = 0; n < total && ok; ++n) {
          const int qs = n % C::kQSlots, os = n % C::kOSlots;
          const int qs1 = (n + 1) % C::kQSlots, os1 = (n + 1) % C::kOSlots;
          const bool more = n + 1 < total;
          // S^T(n+1) into X((n+1)&1): with two X buffers it goes first, ahead of dV(n) (the
          // buffer's last reader, dV(n-1), was issued before it); with one, behind dV(n)
          auto next_st = [&]() -> bool {
            if (!ptx::mbar_wait(ptx::smem_u32(&bars->q_full[qs1]), (uint32_t)((n + 1) / C::kQSlots) & 1u,
                                lim_ms, a.err))
              return false;
            ptx::tc_fence_after();
            st_mma(C::x_col(n + 1), sbase + C::kK, sbase + C::kQ + qs1 * C::kTile);
            ptx::mma_commit(ptx::smem_u32(&bars->s_full[(n + 1) & 1]));
            return true;
          };
          if (C::kXDouble && more) {
            ok = next_st();
            if (!ok) break;
          }
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->p_ready), (uint32_t)n & 1u, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          acc_mma(C::kDV, C::x_col(n), sbase + C::kO + os * C::kTile, n == 0);
          ptx::mma_commit(ptx::smem_u32(&bars->o_empty[os]));
          if (!C::kXDouble && more) {
            ok = next_st();
            if (!ok) break;
          }
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->ds_ready), (uint32_t)n & 1u, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          acc_mma(C::kDK, C::kY, sbase + C::kQ + qs * C::kTile, n == 0);
          // no commit frees Q_n: dP^T(n+1), issued next, comes after both products that read it,
          // so the compute warps free it on seeing dP^T(n+1) (a commit stalls the tensor pipe
          // for about as long as one MMA)
          if (more) {                                 // dP^T(n+1) into Y, behind dK(n)
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->o_full[os1]), (uint32_t)((n + 1) / C::kOSlots) & 1u,
                                lim_ms, a.err);
            if (!ok) break;
            ptx::tc_fence_after();
            st_mma(C::kY, sbase + C::kV, sbase + C::kO + os1 * C::kTile);
            ptx::mma_commit(ptx::smem_u32(&bars->dp_full));
          }
        }
      }
      ptx::mma_commit(ptx::smem_u32(&bars->acc_done));
      ptx::mbar_wait(ptx::smem_u32(&bars->acc_done), 0, lim_ms, a.err);
    }
  } else {
    // ------------------------------- compute warpgroups -----------------------------------------
    const int wg = warp / 4, sub = warp % 4;
    const int kr = sub * 32 + lane;                  // key row within the tile (TMEM lane)
    const int key = g.k0 + kr;
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const float c = a.scale * kLog2e;
    const float2 c2 = make_float2(c, c);
    const bool key_ok = key < g.kv_lim;
    const uint32_t tY = tmem + lane_off + C::kY + wg * kCols;
    constexpr int kNR = kCols / 32;                  // 32-column TMEM loads per operand
    bool ok = true;
    int n = 0;
    const uint32_t sq = (uint32_t)lane & 3u;         // this key within its 4-key dropout block
    DropTest dtest{};
    if constexpr (kDrop) dtest = drop_test(a.drop);
    for (int hg = 0; hg < G && ok; ++hg)
    for (int i = g.next(g.i_begin); i < g.i_end; i = g.next(i + 1), ++n) {
      const int vs = n & 1;
      // dropout: this key's drop flags over the warpgroup's queries, 16 per word (generated
      // while the scores are still being computed; the quad shares its calls); the mask slice is
      // that of query head hk*G + hg
      uint32_t flags[kCols / 16];
      if constexpr (kDrop) {
        const uint32_t mh = (uint32_t)(b * a.H + hk * G + hg);
#pragma unroll
        for (int m = 0; m < kCols / 16; ++m) {
          const uint4 r = philox4x32_10((uint32_t)key >> 2, (uint32_t)((i * BM + wg * kCols) / 4) + 4u * m + sq,
                                        mh, a.drop.offset, a.drop);
          flags[m] = gather_col_flags(pack_flags(r, dtest), sq);
        }
      }
      const int kind = g.kind(i);                    // (a read of the mask: before the waits)
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->vec_full[vs]), (uint32_t)(n >> 1) & 1u, lim_ms, a.err);
      if (ok) ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_full[n & 1]), (uint32_t)(n >> 1) & 1u, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tX = tmem + lane_off + C::x_col(n) + wg * kCols;   // S^T(n), then P^T(n)
      const float* lse2 = reinterpret_cast<const float*>(smem + C::kVec + vs * 1024) + wg * kCols;
      const float* dl = lse2 + 128;
      const int q0 = i * BM + wg * kCols;            // first query column of this warpgroup
      // P^T for this thread's key row over the warpgroup's query columns
      float p[kCols];
      {
        uint32_t raw[kNR][32];
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) ptx::tmem_ld32(tX + hc * 32, raw[hc]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) {
          ptx::reg_fence(raw[hc]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {          // column pairs: packed fp32 arithmetic
            const int col = hc * 32 + e;
            const float2 nl = *reinterpret_cast<const float2*>(lse2 + col);
            const float2 x = ptx::fma2(make_float2(__uint_as_float(raw[hc][e]), __uint_as_float(raw[hc][e + 1])),
                                       c2, nl);
            float v0 = ptx::ex2(x.x), v1 = ptx::ex2(x.y);
            if (kind == kPartial) {
              v0 = (key_ok && (!g.causal || key <= q0 + col)) ? v0 : 0.f;
              v1 = (key_ok && (!g.causal || key <= q0 + col + 1)) ? v1 : 0.f;
            }
            p[col] = v0;
            p[col + 1] = v1;
          }
        }
      }
      {
        uint32_t pk[kCols / 2];
#pragma unroll
        for (int e = 0; e < kCols / 2; ++e) {
          if constexpr (kDrop) {                     // dV takes the dropped-out probabilities
            const uint32_t k = (((uint32_t)e >> 1) & 3u) ^ sq;   // queries 2e, 2e+1: group e/2
            pk[e] = ptx::pack2<F16>(p[2 * e], p[2 * e + 1]) & ~col_pair_mask(flags[e / 8], e & 1, k);
          } else {
            pk[e] = ptx::pack2<F16>(p[2 * e], p[2 * e + 1]);
          }
        }
        ptx::tmem_st(tX, pk);
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_ready));
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), (uint32_t)n & 1u, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      // dP^T(n) has completed, and with it dK(n-1), the last product to read Q_{n-1}
      if (n > 0 && warp == 0 && lane == 0)
        ptx::mbar_arrive(ptx::smem_u32(&bars->q_empty[(n - 1) % C::kQSlots]));
      // dS^T = P^T * (dP^T - D)
      {
        uint32_t raw[kNR][32];
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) ptx::tmem_ld32(tY + hc * 32, raw[hc]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int hc = 0; hc < kNR; ++hc) {
          ptx::reg_fence(raw[hc]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = hc * 32 + e;
            float2 dpv = make_float2(__uint_as_float(raw[hc][e]), __uint_as_float(raw[hc][e + 1]));
            if constexpr (kDrop) {                   // dP = (dO V^T) * M * 256/k8
              const uint32_t k = (((uint32_t)col >> 2) & 3u) ^ sq;
              const uint32_t fw = flags[col / 16];
              dpv.x = __uint_as_float(raw[hc][e] & ~col_elem_mask(fw, col & 3, k));
              dpv.y = __uint_as_float(raw[hc][e + 1] & ~col_elem_mask(fw, (col & 3) + 1, k));
              dpv = ptx::mul2(dpv, make_float2(a.drop.scale, a.drop.scale));
            }
            const float2 dd = ptx::sub2(dpv, *reinterpret_cast<const float2*>(dl + col));
            const float2 ds = ptx::mul2(make_float2(p[col], p[col + 1]), dd);
            p[col] = ds.x;
            p[col + 1] = ds.y;
          }
        }
      }
      {
        uint32_t pk[kCols / 2];
#pragma unroll
        for (int e = 0; e < kCols / 2; ++e) pk[e] = ptx::pack2<F16>(p[2 * e], p[2 * e + 1]);
        ptx::tmem_st(tY, pk);
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&bars->ds_ready));
        ptx::mbar_arrive(ptx::smem_u32(&bars->vec_empty[vs]));   // this tile's vectors are read
      }
    }
    // ------------------------------- epilogue: dV (first half of the warpgroups), dK (second) ---
    const bool have = ok && n > 0;
    if (have) {
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_done), 0, lim_ms, a.err);
      ptx::tc_fence_after();
    }
    constexpr int kPer = L::kWG / 2;                 // warpgroups per output, each D / kPer columns
    const bool is_dv = wg < kPer;
    const int c0 = (wg % kPer) * (D / kPer);
    const float mult = is_dv ? (kDrop ? a.drop.scale : 1.f) : a.scale;
    uint16_t* out = static_cast<uint16_t*>(is_dv ? a.dv : a.dk) + ((size_t)ks * a.rows + row0 + key) * D + c0;
    const uint32_t src = (is_dv ? C::kDV : C::kDK) + c0;
#pragma unroll 1
    for (int hc = 0; hc < D / kPer / 32; ++hc) {
      uint32_t raw[32];
      if (have && ok) {
        ptx::tmem_ld32(tmem + lane_off + src + hc * 32, raw);
        ptx::tmem_wait_ld();
        ptx::reg_fence(raw);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) raw[e] = 0u;
      }
      if (key < g.N) {
        uint4* dst = reinterpret_cast<uint4*>(out + hc * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint4 w;
          w.x = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 0]) * mult, __uint_as_float(raw[8 * v4 + 1]) * mult);
          w.y = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 2]) * mult, __uint_as_float(raw[8 * v4 + 3]) * mult);
          w.z = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 4]) * mult, __uint_as_float(raw[8 * v4 + 5]) * mult);
          w.w = ptx::pack2<F16>(__uint_as_float(raw[8 * v4 + 6]) * mult, __uint_as_float(raw[8 * v4 + 7]) * mult);
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

}  // namespace dkdv
}  // namespace fa
