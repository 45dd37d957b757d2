// Tensor-core attention backward for sm_103a (bf16 or fp16 in, fp32 accumulate), d in {64, 128}.
//
// The method ("FlashAttention paper story", backward paragraph; "FlashAttention: Exact Attention
// with Less GPU Memory", "Tiling, and paying arithmetic to avoid memory"): only the per-row
// softmax statistic is kept from the forward; the backward recomputes the scores and P tile by
// tile on chip.  With D_i = rowsum(dO_i * O_i) (computed by the preprocess kernel):
//     P = exp(scale*S - LSE),  dV += P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//     dK += scale * dS^T Q,  dQ += scale * dS K.
//
// GB300 design: one CTA per 128-key tile j of one (b, h) key/value slice, 320 threads, looping
// over every live 128-row query tile i of every query head that reads that slice (one head,
// or the G heads of a group under grouped-query attention).  The transposed products keep the key rows on the TMEM lanes, so
// one thread owns one key row of S^T, dP^T, P^T and dS^T:
//   warp 8      TMA producer: K_j, V_j once; Q_i, dO_i through a two-stage ring, with the
//               tile's LSE (as a log2-domain bias) and D vectors staged beside them.
//   warp 9      MMA issuer: S^T = K_j Q_i^T and dP^T = V_j dO_i^T (SS); dV += P^T dO_i as
//               soon as P^T is back in TMEM (overlapping the dS^T work), then dK += dS^T Q_i
//               (TS: P^T, dS^T read from TMEM) and dQ_i = dS K_j (SS: dS staged in shared
//               memory) in N = 64 parts.
//   warps 0-7   two warpgroups, query columns [0,64) and [64,128): P^T and dS^T in registers,
//               written back to TMEM as bf16 and dS also to shared memory.  Then each warp
//               copies its 32 rows of the tile's dQ (its warpgroup's half of d) from TMEM into
//               the tile's Q/dO stage, which no MMA reads any more, and the TMA unit adds them
//               into the fp32 workspace (bulk tensor reduce-add); the stage is handed back to
//               the producer once the TMA unit has read it.
//   TMEM d=128: dV [0,128) dK [128,256) X=S^T [256,384) Y=dP^T [384,512); P^T packed in
//               X[0,64), dS^T packed in Y[0,64); once dK has read dS^T, the two dQ halves go to
//               Y[0,64) and Y[64,128), so the next tile's S^T (into X) overlaps the dQ drain.
//   TMEM d=64:  dV [0,64) dK [64,128) X [128,256) Y [256,384) dQ [384,448).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.cuh"
#include "fa_sm103.cuh"
#include "ptx_sm103.cuh"

namespace fa {
namespace {

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per CTA
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool F16>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;                  // one 128-row operand tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ0 = kV + kTile;                     // stage s: Q at kQ0 + s*2*kTile
  static constexpr int kDS = kQ0 + 4 * kTile;                // dS [128 keys][128 queries] bf16
  static constexpr int kVec = kDS + 128 * 128 * 2;           // stage s: lse2[128], delta[128]
  static constexpr int kBar = kVec + 2 * 2 * 128 * 4;
  static constexpr int kSmem = kBar + 256;
  // TMEM columns
  static constexpr uint32_t kDV = 0, kDK = D, kX = 2 * D, kY = 2 * D + 128;
  static constexpr uint32_t kIdescST = ptx::idesc_f32acc(128, 128, false, false, F16);  // S^T, dP^T
  static constexpr uint32_t kIdescAcc = ptx::idesc_f32acc(128, D, false, true, F16);    // dV, dK
  static constexpr uint32_t kIdescDQ = ptx::idesc_f32acc(128, 64, true, true, F16);     // dQ parts
  static constexpr int kDQParts = D / 64;                    // N = 64 columns of d per part
};

struct Bars {             // at most 128 bytes (the live-tile bitmap follows)
  uint64_t kv_full;
  uint64_t st_full[2];
  uint64_t st_empty[2];
  uint64_t s_full;
  uint64_t dp_full;
  uint64_t s_read;
  uint64_t dp_read;
  uint64_t p_ready;
  uint64_t ds_ready;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t acc_done;
  uint32_t tmem_base;
};

static_assert(sizeof(Bars) <= 128, "the live-tile bitmap starts 128 bytes after the barriers");

enum : int { kNone = 0, kPartial = 1, kFull = 2 };

struct Geo {
  int k0, N, kv_lim, causal, T;
  const uint8_t* bm;
  int i_begin, i_end;    // query tiles that may be live
  __device__ int kind(int i) const {
    const int r0 = i * BM, r1 = min(r0 + BM, N) - 1;
    const int c0 = k0, c1 = k0 + BN - 1;
    if (bm != nullptr && bm[(size_t)i * T + k0 / BN] == 0) return kNone;
    if (c0 >= kv_lim || (causal && c0 > r1)) return kNone;
    if (c1 < kv_lim && (!causal || c1 <= r0)) return kFull;
    return kPartial;
  }
  // Without a tile mask the live query tiles are exactly [i_begin, i_end).  With one, `bits`
  // (shared memory, built once per CTA) marks the live tiles and the next one is found a word
  // at a time.
  const uint32_t* bits;
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

template <int D, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
bwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                 const __grid_constant__ CUtensorMap tmDQ, BwdArgs a) {
  using C = Cfg<D, F16>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {      // the operand tiles need 1 KB alignment
    if (threadIdx.x == 0) atomicExch(a.err, 2);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBar);
  const uint32_t sbase = ptx::smem_u32(smem);
  // Work order.  With masks, the (b, h) slice varies fastest, so every slice's heaviest key
  // tiles (the first ones when causal, the global columns of a block-sparse mask) run in the
  // first waves.  Without, one slice's key tiles run together and share its Q/dO stream in L2.
  // A CTA owns one key tile of one key/value head; with grouped-query attention the G = H / Hkv
  // query heads that share that key/value head are all visited by it, so dK and dV accumulate
  // over the whole group on chip.
  const int BH = a.B * a.Hkv;
  const int n_kt = (a.N + BN - 1) / BN;
  const int bh = a.heads_fastest ? (int)(blockIdx.x % BH) : (int)(blockIdx.x / n_kt);   // K/V slice
  const int jt = a.heads_fastest ? (int)(blockIdx.x / BH) : (int)(blockIdx.x % n_kt);   // key tile
  const int b = bh / a.Hkv;
  const int G = a.H / a.Hkv;
  const int bhq0 = b * a.H + (bh % a.Hkv) * G;   // first query slice of the group
  const uint32_t lim_ms = a.dbg.wait_limit_ms;

  Geo g;
  g.k0 = jt * BN;
  g.N = a.N;
  int kvl = a.N;
  if (a.kv_lens != nullptr) kvl = max(0, min(a.N, (int)a.kv_lens[b]));
  g.kv_lim = kvl;
  g.causal = a.causal;
  g.T = a.n_tiles;
  g.bm = a.block_mask;
  g.i_begin = a.causal ? jt : 0;
  g.i_end = g.k0 < g.kv_lim ? (a.N + BM - 1) / BM : 0;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->st_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->st_empty[s]), 8);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->s_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->s_read), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->dp_read), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->p_ready), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->ds_ready), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->dq_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->dq_free), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->acc_done), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  g.bits = nullptr;
  if (a.block_mask != nullptr) {                 // live-tile bitmap, one ballot per 32 tiles
    uint32_t* live_bits = reinterpret_cast<uint32_t*>(smem + C::kBar + 128);
    g.bits = live_bits;
    for (int w = warp; w < (g.i_end + 31) / 32; w += kThreads / 32) {
      const int i = w * 32 + lane;
      const uint32_t word = __ballot_sync(0xffffffffu, i >= g.i_begin && i < g.i_end && g.kind(i) != kNone);
      if (lane == 0) live_bits[w] = word;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------- producer (whole warp) --------------------------------------
    bool ok = true;
    int n = 0;
    if (g.next(g.i_begin) < g.i_end) {
      if (lane == 0) {
        const uint32_t kb = ptx::smem_u32(&bars->kv_full);
        ptx::mbar_arrive_expect_tx(kb, 2 * C::kTile);
        for (int hh = 0; hh < D / 64; ++hh) {
          ptx::tma_load_3d(sbase + C::kK + hh * 128 * 128, &tmK, kb, hh * 64, g.k0, bh);
          ptx::tma_load_3d(sbase + C::kV + hh * 128 * 128, &tmV, kb, hh * 64, g.k0, bh);
        }
      }
      for (int hg = 0; hg < G && ok; ++hg)
      for (int i = g.next(g.i_begin); i < g.i_end && ok; i = g.next(i + 1), ++n) {
        const int bhq = bhq0 + hg;
        const int st = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        if (lane == 0) ok = ptx::mbar_wait(ptx::smem_u32(&bars->st_empty[st]), ph ^ 1, lim_ms, a.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // -LSE (as a log2-domain bias; -inf where P must vanish) and D for the tile's rows
        float* lse2 = reinterpret_cast<float*>(smem + C::kVec + st * 1024);
        float* dl = lse2 + 128;
        // all eight loads of a lane first, then the stores (which could alias the loads as far
        // as the compiler knows)
        float Lv[4], Dv[4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int q = i * BM + lane + 32 * k4;
          Lv[k4] = q < a.N ? __ldg(a.lse + (size_t)bhq * a.N + q) : -INFINITY;
          Dv[k4] = q < a.N ? __ldg(a.delta + (size_t)bhq * a.N + q) : 0.f;
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          lse2[lane + 32 * k4] = Lv[k4] == -INFINITY ? -INFINITY : -Lv[k4] * kLog2e;   // negated
          dl[lane + 32 * k4] = Dv[k4];
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = ptx::smem_u32(&bars->st_full[st]);
          ptx::mbar_arrive_expect_tx(fb, 2 * C::kTile);
          const uint32_t sq = sbase + C::kQ0 + st * 2 * C::kTile;
          for (int hh = 0; hh < D / 64; ++hh) {
            ptx::tma_load_3d(sq + hh * 128 * 128, &tmQ, fb, hh * 64, i * BM, bhq);
            ptx::tma_load_3d(sq + C::kTile + hh * 128 * 128, &tmDO, fb, hh * 64, i * BM, bhq);
          }
        }
      }
      if (lane == 0) {   // drain: copies in flight must land before shared memory is released
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full), 0, lim_ms, a.err);
        for (int m = max(0, n - 2); m < n; ++m)
          ptx::mbar_wait(ptx::smem_u32(&bars->st_full[m & 1]), (m >> 1) & 1, lim_ms, a.err);
      }
    }
  } else if (warp == 9) {
    // ------------------------------- MMA issuer -------------------------------------------------
    if (lane == 0) {
      bool ok = true;
      int n = 0;
      if (g.next(g.i_begin) < g.i_end) {
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full), 0, lim_ms, a.err);
        for (int hg = 0; hg < G && ok; ++hg)
        for (int i = g.next(g.i_begin); i < g.i_end && ok; i = g.next(i + 1), ++n) {
          const int st = n & 1;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->st_full[st]), (n >> 1) & 1, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t sq = sbase + C::kQ0 + st * 2 * C::kTile;
          const uint32_t sdo = sq + C::kTile;
          // S^T = K Q^T, dP^T = V dO^T (K-major operands, k-steps of 16 along d)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            ptx::mma_ss(tmem + C::kX, ptx::sdesc_sw128(sbase + C::kK + off, 16, 1024),
                        ptx::sdesc_sw128(sq + off, 16, 1024), C::kIdescST, kk > 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->s_full));
          if (n > 0 && D == 128) {     // Y holds the previous tile's dQ until it is drained
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->dq_free), (n - 1) & 1, lim_ms, a.err);
            if (!ok) break;
            ptx::tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            ptx::mma_ss(tmem + C::kY, ptx::sdesc_sw128(sbase + C::kV + off, 16, 1024),
                        ptx::sdesc_sw128(sdo + off, 16, 1024), C::kIdescST, kk > 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->dp_full));
          // dV += P^T dO as soon as P^T is in TMEM (the dS^T work overlaps it).  A from TMEM: 16
          // queries = 8 packed columns per step; B = dO with the query index as K (MN-major,
          // 16 rows = 2048 bytes per step).
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->p_ready), n & 1, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            ptx::mma_ts(tmem + C::kDV, tmem + C::kX + kk * 8,
                        ptx::sdesc_sw128(sdo + kk * 2048, 128 * 128, 1024), C::kIdescAcc,
                        (n > 0 || kk > 0) ? 1u : 0u);
          // dK += dS^T Q once dS^T is ready
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->ds_ready), n & 1, lim_ms, a.err);
          if (ok && n > 0 && D == 64)
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->dq_free), (n - 1) & 1, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            ptx::mma_ts(tmem + C::kDK, tmem + C::kY + kk * 8,
                        ptx::sdesc_sw128(sq + kk * 2048, 128 * 128, 1024), C::kIdescAcc,
                        (n > 0 || kk > 0) ? 1u : 0u);
          // dQ_i = dS K_j, 64 columns of d per part: A = dS (queries x keys, query-major in
          // shared memory), B = K (keys x d, d-major); 16 keys = 2048 bytes per step.
#pragma unroll
          for (int part = 0; part < C::kDQParts; ++part) {
            const uint32_t dst = D == 128 ? C::kY + part * 64 : 384;
            const uint32_t kb = sbase + C::kK + part * 128 * 128;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              ptx::mma_ss(tmem + dst, ptx::sdesc_sw128(sbase + C::kDS + kk * 2048, 128 * 128, 1024),
                          ptx::sdesc_sw128(kb + kk * 2048, 128 * 128, 1024), C::kIdescDQ, kk > 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->dq_full));
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
    bool ok = true;
    int n = 0;
    int pend_st = -1;                                // stage whose staged dQ is still being read
    for (int hg = 0; hg < G && ok; ++hg)
    for (int i = g.next(g.i_begin); i < g.i_end; i = g.next(i + 1), ++n) {
      const int bhq = bhq0 + hg;
      const int st = n & 1;
      const int kind = g.kind(i);                    // (a read of the mask: before the waits)
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->st_full[st]), (n >> 1) & 1, lim_ms, a.err);
      if (ok) ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_full), n & 1, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(smem + C::kVec + st * 1024) + wg * 64;
      const float* dl = lse2 + 128;
      const int q0 = i * BM + wg * 64;               // first query column of this warpgroup
      // P^T for this thread's key row over 64 query columns
      float p[64];
      {
        uint32_t raw[2][32];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) ptx::tmem_ld32(tmem + lane_off + C::kX + wg * 64 + hc * 32, raw[hc]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          ptx::reg_fence(raw[hc]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {        // column pairs: packed fp32 arithmetic
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
      // all of S^T is read (by both warpgroups) before P^T overwrites part of it
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->s_read));
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_read), n & 1, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = ptx::pack2<F16>(p[2 * e], p[2 * e + 1]);
        ptx::tmem_st32(tmem + lane_off + C::kX + wg * 32, pk);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_ready));
        if (lane == 0 && pend_st >= 0) {              // previous tile's staged dQ has been read
          ptx::bulk_wait_read0();
          ptx::mbar_arrive(ptx::smem_u32(&bars->st_empty[pend_st]));
          pend_st = -1;
        }
        __syncwarp();
      }
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->dp_full), n & 1, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      // dS^T = P^T * (dP^T - D)
      {
        uint32_t raw[2][32];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) ptx::tmem_ld32(tmem + lane_off + C::kY + wg * 64 + hc * 32, raw[hc]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          ptx::reg_fence(raw[hc]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = hc * 32 + e;
            const float2 dd = ptx::sub2(make_float2(__uint_as_float(raw[hc][e]), __uint_as_float(raw[hc][e + 1])),
                                        *reinterpret_cast<const float2*>(dl + col));
            const float2 ds = ptx::mul2(make_float2(p[col], p[col + 1]), dd);
            p[col] = ds.x;
            p[col + 1] = ds.y;
          }
        }
      }
      ptx::tc_fence_before();                         // all of dP^T read before dS^T overwrites Y
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->dp_read));
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->dp_read), n & 1, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = ptx::pack2<F16>(p[2 * e], p[2 * e + 1]);
        ptx::tmem_st32(tmem + lane_off + C::kY + wg * 32, pk);
        // dS into shared memory, query-major 128-byte-swizzled: row = key, 64 queries per atom
        uint8_t* row = smem + C::kDS + wg * (128 * 128) + kr * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint4 w = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          *reinterpret_cast<uint4*>(row + ((ch ^ (kr & 7)) << 4)) = w;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->ds_ready));
      // dQ of this query tile: lane = query row; this warpgroup takes half of d, in boxes of 32
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->dq_full), n & 1, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      {
        constexpr int kBoxes = D / 64;                 // 32-column boxes per warp
        const uint32_t src = D == 128 ? C::kY + wg * 64 : 384 + wg * 32;
        uint32_t dqv[kBoxes][32];
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) ptx::tmem_ld32(tmem + lane_off + src + bx * 32, dqv[bx]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) ptx::reg_fence(dqv[bx]);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->dq_free));   // TMEM dQ may be reused
        // stage: 32 rows x 32 fp32 per box, 128-byte swizzled, inside this tile's Q/dO buffer
        uint8_t* stage = smem + C::kQ0 + st * 2 * C::kTile;
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) {
          uint8_t* box = stage + ((wg * kBoxes + bx) * 4 + sub) * 4096;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(box + lane * 128 + ((ch ^ (lane & 7)) << 4)) =
                make_uint4(dqv[bx][4 * ch], dqv[bx][4 * ch + 1], dqv[bx][4 * ch + 2], dqv[bx][4 * ch + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row0 = i * BM + sub * 32;
          if (row0 < a.N) {
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
              ptx::tma_reduce_add_3d(&tmDQ, ptx::smem_u32(stage + ((wg * kBoxes + bx) * 4 + sub) * 4096),
                                     wg * (D / 2) + bx * 32, row0, bhq);
            ptx::bulk_commit();
          }
          pend_st = st;   // handed back to the producer once the TMA unit has read it
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      ptx::bulk_wait0();                              // every reduction has landed in global memory
      if (pend_st >= 0) ptx::mbar_arrive(ptx::smem_u32(&bars->st_empty[pend_st]));
    }
    // ------------------------------- epilogue: dV (warpgroup 0), dK (warpgroup 1) --------------
    const bool have = ok && n > 0;
    if (have) {
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_done), 0, lim_ms, a.err);
      ptx::tc_fence_after();
    }
    const float mult = wg == 0 ? 1.f : a.scale;
    uint16_t* out = static_cast<uint16_t*>(wg == 0 ? a.dv : a.dk) + ((size_t)bh * a.N + key) * D;
    const uint32_t src = wg == 0 ? C::kDV : C::kDK;
#pragma unroll 1
    for (int hc = 0; hc < D / 32; ++hc) {
      uint32_t raw[32];
      if (have && ok) {
        ptx::tmem_ld32(tmem + lane_off + src + hc * 32, raw);
        ptx::tmem_wait_ld();
        ptx::reg_fence(raw);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) raw[e] = 0u;
      }
      if (key < a.N) {
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
  if (warp == 9) ptx::tmem_dealloc(tmem, kTmemCols);
}

cudaError_t make_map(CUtensorMap* m, const void* base, int D, int N, int BH, bool f16) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tensor_map(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, bool F16>
cudaError_t launch(const BwdArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int BH = a.B * a.H;            // query slices (Q, dO, dQ)
  const int BHkv = a.B * a.Hkv;        // key/value slices (K, V, dK, dV)
  cudaError_t e;
  if ((e = make_map(&mq, a.q, D, a.N, BH, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, D, a.N, BHkv, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mv, a.v, D, a.N, BHkv, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mdo, a.dO, D, a.N, BH, F16)) != cudaSuccess) return e;
  {
    // fp32 dQ workspace viewed as (d, N, B*H); boxes of 32 columns x 32 rows
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)a.N * D * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if ((e = encode_tensor_map(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.dq_acc, dims, strides, box,
                               estr, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
  }
  auto kern = bwd_sm103_kernel<D, F16>;
  // barriers (128 bytes) + the live-tile bitmap of a block-sparse mask (one bit per query tile)
  int smem = Cfg<D, F16>::kSmem;
  if (a.block_mask != nullptr) smem = max(smem, Cfg<D, F16>::kBar + 128 + ((a.n_tiles + 127) / 128) * 16);
  static LaunchSetup setup;
  e = prepare_launch(setup, kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(((a.N + BN - 1) / BN) * BHkv);
  kern<<<grid, kThreads, smem, s>>>(mq, mk, mv, mdo, mdq, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_sm103(const BwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_FP16) return a.d == 64 ? launch<64, true>(a, s) : launch<128, true>(a, s);
  return a.d == 64 ? launch<64, false>(a, s) : launch<128, false>(a, s);
}

}  // namespace fa
