// Attention forward at d = 64 with 64-key tiles, two CTAs on every SM (bf16 or fp16 in, fp32
// accumulate): the plain forward at that head size (no tile mask, packing, split-KV or dropout).
//
// The method and the per-tile pipeline are those of fa_fwd_sm103.cu ("FlashAttention paper
// story", tiling and online-softmax paragraphs; "FlashAttention：让精确注意力服从内存层次",
// section "Online softmax"): two 128-row Q tiles per CTA, K/V tiles through rings of their own,
// S and O in TMEM, the two softmax warpgroups ping-ponging, a lazily raised maximum.  What
// differs is the key tile: 64 keys instead of 128.  That halves the TMEM a CTA needs (S_0, S_1,
// O_0, O_1 in 256 columns) and, with 8 KB K/V tiles, its shared memory (97 KB), so two CTAs fit
// on an SM.  At N = 512-1024 a CTA has only a handful of key tiles and its fixed costs (set-up,
// the first copies from HBM, the epilogue) weigh as much as its tiles; with one CTA per SM a
// BERT- or GPT-2-shaped batch takes two or three waves, each paying them in turn, and with two
// it fits in about one wave.  At longer N the two CTAs' softmax chains overlap each other's
// waits (the one-CTA kernel at d = 64 is bound by that chain's latency, not by a pipe), which
// measured 9-11 % faster at N = 4096-8192 as well.  Masks handled: causal and key padding.
//
// GB300 layout of one CTA (384 threads, 80 registers each at launch): warp 8 producer (Q, K),
// warp 10 producer (V), warp 9 MMA issuer, warps 0-7 softmax (one query row a thread; registers
// re-split to 96 for them and 48 for warps 8-11); TMEM S_0 [0,64), S_1 [64,128), O_0 [128,192),
// O_1 [192,256); P_t overwrites the first 32 columns of S_t as packed 16-bit pairs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.cuh"
#include "fa_sm103.cuh"
#include "ptx_sm103.cuh"

namespace fa {
namespace {

constexpr int D = 64;            // head size
constexpr int BM = 128;          // rows per Q tile
constexpr int BN = 64;           // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kTmemCols = 256;
constexpr int kRegsSoftmax = 96;  // registers per thread after the re-split: 8 softmax warps
constexpr int kRegsOther = 48;    // ... and the producer / MMA warpgroup
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { kNone = 0, kPartial = 1, kFull = 2 };

template <bool F16>
struct Cfg {
  static constexpr int kQTileBytes = BM * D * 2;                // one Q tile (16 KB)
  static constexpr int kTileBytes = BN * D * 2;                 // one K or V tile (8 KB)
  static constexpr int kKSlots = 4;                             // K ring: slots [0, kKSlots)
  static constexpr int kVSlots = 4;                             // V ring: the next kVSlots
  static constexpr int kSlots = kKSlots + kVSlots;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kQTileBytes;
  static constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;            // + barriers + alignment slack
  static constexpr uint32_t kIdescS = ptx::idesc_f32acc(BM, BN, false, false, F16);
  static constexpr uint32_t kIdescO = ptx::idesc_f32acc(BM, D, false, true, F16);
};

struct Bars {            // all mbarriers of one CTA (8 bytes each)
  uint64_t q_full;
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t pv_done[2];
  uint64_t mma_done;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint32_t tmem_base;
};

static_assert(sizeof(Bars) <= 256, "the barrier area is 256 bytes");

// This CTA's tile geometry: which key tiles exist and how each Q tile must treat them.
struct Geo {
  int bh;          // (b, h) slice: Q/O slice index
  int ks;          // K/V slice index
  int q0;          // first query row of Q tile 0
  int N, kv_lim;   // keys with index >= kv_lim are masked (padding and tail)
  int causal;
  int j_end;       // key tiles [0, j_end) may be live

  __device__ int kind(int t, int j) const {
    const int r0 = q0 + t * BM;
    if (r0 >= N) return kNone;
    const int r1 = min(r0 + BM, N) - 1;
    const int c0 = j * BN, c1 = c0 + BN - 1;
    if (c0 >= kv_lim || (causal && c0 > r1)) return kNone;
    if (c1 < kv_lim && (!causal || c1 <= r0)) return kFull;
    return kPartial;
  }
};

template <bool F16>
__global__ void __launch_bounds__(kThreads, 2)
fwd_bn64_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  using C = Cfg<F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
  const uint32_t sQ = ptx::smem_u32(smem + C::kQOff);
  const uint32_t sKV = ptx::smem_u32(smem + C::kKVOff);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // Work order as in the one-CTA-per-SM forward: with a causal mask or key padding the (b, h)
  // slice varies fastest and the heaviest Q-tile pairs come first; without, one slice's pairs
  // run together.
  auto make_geo = [&]() {
    const int BH = a.B * a.H;
    const int n_pairs = (a.N + 2 * BM - 1) / (2 * BM);
    const int unit = blockIdx.x;
    const int bh = a.heads_fastest ? unit % BH : unit / n_pairs;
    const int slot = a.heads_fastest ? unit / BH : unit % n_pairs;
    const int pair = a.causal ? n_pairs - 1 - slot : slot;
    const int b = bh / a.H, h = bh % a.H;
    Geo g;
    g.bh = bh;
    g.q0 = pair * 2 * BM;
    g.N = a.N;
    // grouped-query attention: query head h reads key/value head h / (H / Hkv)
    g.ks = b * a.Hkv + h / (a.H / a.Hkv);
    g.kv_lim = a.kv_lens != nullptr ? max(0, min(a.Nk, (int)a.kv_lens[b])) : a.Nk;
    g.causal = a.causal;
    int last_key = g.kv_lim;
    if (a.causal) last_key = min(last_key, min(g.q0 + 2 * BM, g.N));
    g.j_end = (last_key + BN - 1) / BN;
    return g;
  };
  const uint32_t lim_ms = a.dbg.wait_limit_ms;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(ptx::smem_u32(&bars->s_full[t]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->p_ready[t]), 4);
      ptx::mbar_init(ptx::smem_u32(&bars->pv_done[t]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->mma_done), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->kv_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->kv_empty[s]), 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
    ptx::regs_dec<kRegsOther>();
    const Geo g = make_geo();
    if (warp == 8 && lane == 0) {
      // ------------------------------- TMA producer (Q, K) ------------------------------------
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      const uint32_t qbar = ptx::smem_u32(&bars->q_full);
      ptx::mbar_arrive_expect_tx(qbar, 2 * C::kQTileBytes);
      for (int t = 0; t < 2; ++t)
        ptx::tma_load_3d(sQ + t * C::kQTileBytes, &tmQ, qbar, 0, g.q0 + t * BM, g.bh);
      int n = 0;                                   // K tiles issued
      bool ok = true;
      for (int j = 0; j < g.j_end && ok; ++j, ++n) {
        const int slot = n % C::kKSlots;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[slot]), ((n / C::kKSlots) & 1) ^ 1, lim_ms, a.err);
        if (!ok) break;
        if (a.dbg.inject == 1 && n == 0) continue;      // test hook: never deliver this tile
        const uint32_t fb = ptx::smem_u32(&bars->kv_full[slot]);
        ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
        ptx::tma_load_3d(sKV + slot * C::kTileBytes, &tmK, fb, 0, j * BN, g.ks);
      }
      // Drain: every copy this thread issued must have landed before shared memory is released.
      ptx::mbar_wait(qbar, 0, lim_ms, a.err);
      for (int m = max(0, n - C::kKSlots); m < n; ++m) {
        if (a.dbg.inject == 1 && m == 0) continue;
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[m % C::kKSlots]), (m / C::kKSlots) & 1, lim_ms, a.err);
      }
    } else if (warp == 10 && lane == 0) {
      // ------------------------------- TMA producer of V ------------------------------------
      int n = 0;                                   // V tiles issued
      bool ok = true;
      for (int j = 0; j < g.j_end && ok; ++j, ++n) {
        const int slot = C::kKSlots + n % C::kVSlots;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[slot]), ((n / C::kVSlots) & 1) ^ 1, lim_ms, a.err);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&bars->kv_full[slot]);
        ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
        ptx::tma_load_3d(sKV + slot * C::kTileBytes, &tmV, fb, 0, j * BN, g.ks);
      }
      for (int m = max(0, n - C::kVSlots); m < n; ++m)
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[C::kKSlots + m % C::kVSlots]), (m / C::kVSlots) & 1, lim_ms, a.err);
    } else if (warp == 9 && lane == 0) {
      // ------------------------------- MMA issuer ---------------------------------------------
      // Per key tile j: O_0 += P_0 V_{j-1}, S_0 = Q_0 K_j^T, O_1 += P_1 V_{j-1}, S_1 = Q_1 K_j^T.
      bool ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_full), 0, lim_ms, a.err);
      ptx::tc_fence_after();
      int idx = 0;
      int prev_v = -1;
      uint32_t prev_vph = 0;
      for (int j = 0; j < g.j_end && ok; ++j, ++idx) {
        const int kslot = idx % C::kKSlots;
        const uint32_t kph = (idx / C::kKSlots) & 1;
        const int vslot = C::kKSlots + idx % C::kVSlots;
        const uint32_t vph = (idx / C::kVSlots) & 1;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[kslot]), kph, lim_ms, a.err);
        if (ok && idx > 0) ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[prev_v]), prev_vph, lim_ms, a.err);
        if (!ok) break;
        ptx::tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          if (idx > 0) {
            // O_t += P_t V_{j_prev}: P_t of the previous key tile sits in S_t's columns.
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->p_ready[t]), (idx - 1) & 1, lim_ms, a.err);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t vbase = sKV + prev_v * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              const uint64_t bdesc = ptx::sdesc_sw128(vbase + kk * 16 * 128, BN * 128, 1024);
              ptx::mma_ts(tmem + 128 + t * D, tmem + t * BN + kk * 8, bdesc, C::kIdescO,
                          (idx > 1 || kk > 0) ? 1u : 0u);
            }
          }
          // S_t = Q_t K_j^T
          const uint32_t qbase = sQ + t * C::kQTileBytes;
          const uint32_t kbase = sKV + kslot * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t adesc = ptx::sdesc_sw128(qbase + kk * 32, 16, 1024);
            const uint64_t bdesc = ptx::sdesc_sw128(kbase + kk * 32, 16, 1024);
            ptx::mma_ss(tmem + t * BN, adesc, bdesc, C::kIdescS, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->s_full[t]));
        }
        // No commit frees K_j or V_{j-1}: S_1(j) is issued after every product that reads them,
        // so the softmax of Q tile 1, on seeing S_1(j), frees both.
        prev_v = vslot;
        prev_vph = vph;
      }
      if (ok && idx > 0) {
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[prev_v]), prev_vph, lim_ms, a.err);
        ptx::tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->p_ready[t]), (idx - 1) & 1, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t vbase = sKV + prev_v * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bdesc = ptx::sdesc_sw128(vbase + kk * 16 * 128, BN * 128, 1024);
            ptx::mma_ts(tmem + 128 + t * D, tmem + t * BN + kk * 8, bdesc, C::kIdescO,
                        (idx > 1 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->pv_done[t]));
        }
      }
      // every MMA this thread issued has finished before TMEM and shared memory are released
      ptx::mma_commit(ptx::smem_u32(&bars->mma_done));
      ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, lim_ms, a.err);
    }
  } else {
    // ------------------------------- softmax warpgroups -----------------------------------------
    ptx::regs_inc<kRegsSoftmax>();
    const Geo g = make_geo();
    const int t = warp / 4;
    const int sub = warp % 4;
    const int r = sub * 32 + lane;                  // TMEM lane == row within the Q tile
    const int i = g.q0 + t * BM + r;                // query row in the head
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tO = tmem + lane_off + 128 + t * D;
    const float c = a.scale * kLog2e;               // scores -> log2 domain
    int row_lim = g.kv_lim;
    if (a.causal) row_lim = min(row_lim, i + 1);
    // How this Q tile treats key tile j, as two thresholds (fewer live registers than the
    // geometry): full below j_full, partly masked below j_none, skipped from there on.
    int j_full = 0, j_none = 0;
    while (j_none < g.j_end && g.kind(t, j_none) != kNone) ++j_none;
    while (j_full < j_none && g.kind(t, j_full) == kFull) ++j_full;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int idx = 0;
    for (; idx < g.j_end; ++idx) {
      const int j = idx;
      const int kind = j < j_full ? kFull : j < j_none ? kPartial : kNone;
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_full[t]), idx & 1, lim_ms, a.err);
      if (!ok) break;
      ptx::tc_fence_after();
      if (t == 1 && sub == 0 && lane == 0) {
        // S_1(j) has completed, and with it every MMA issued before it: both S products of key
        // tile j (K_j's slot is free) and both PV products of the previous tile (V's slot too).
        ptx::mbar_arrive(ptx::smem_u32(&bars->kv_empty[idx % C::kKSlots]));
        if (idx > 0) ptx::mbar_arrive(ptx::smem_u32(&bars->kv_empty[C::kKSlots + (idx - 1) % C::kVSlots]));
      }
      uint32_t pk[32];
      if (kind == kNone) {
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = 0u;
        ptx::tmem_st32(tS, pk);
      } else {
        float s[BN];
        {
          uint32_t raw[2][32];                       // all 64 scores, one wait
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) ptx::tmem_ld32(tS + q2 * 32, raw[q2]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            ptx::reg_fence(raw[q2]);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[q2 * 32 + e] = __uint_as_float(raw[q2][e]);
          }
        }
        if (kind == kPartial) {
          const int lim = row_lim - j * BN;
#pragma unroll
          for (int e = 0; e < BN; ++e) s[e] = e < lim ? s[e] : -INFINITY;
        }
        float m4[4];                                 // 4 independent 3-input-max chains
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
        for (int q = 4; q < BN / 2; ++q) m4[q & 3] = ptx::max3(m4[q & 3], s[2 * q], s[2 * q + 1]);
        const float mx = fmaxf(ptx::max3(m4[0], m4[1], m4[2]), m4[3]);
        const float m_cand = mx * c;
        const bool need = m_cand > m_run + kRescaleLog2;   // false when the row is still empty
        const float alpha = need ? ptx::ex2(m_run - m_cand) : 1.f;
        if (need) {
          l_run *= alpha;
          m_run = m_cand;
        }
        const float msub = m_run == -INFINITY ? 0.f : m_run;
        // p = exp2(s*c - m) on column pairs; 2 independent packed partial sums
        const float2 c2 = make_float2(c, c), nm2 = make_float2(-msub, -msub);
        float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 x = ptx::fma2(make_float2(s[2 * e], s[2 * e + 1]), c2, nm2);
          const float2 pp = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
          ls[e & 1] = ptx::add2(ls[e & 1], pp);        // the normaliser counts every allowed key
          pk[e] = ptx::pack2<F16>(pp.x, pp.y);
        }
        ptx::tmem_st32(tS, pk);
        const float2 lsum = ptx::add2(ls[0], ls[1]);
        l_run += lsum.x + lsum.y;
        if (__any_sync(0xffffffffu, need) && idx > 0) {
          // O_t *= alpha for this warp's rows: after the scores are spent (fewer live
          // registers), before P_t is released to the O_t += P_t V_j product.  PV of the previous
          // tile has completed: the commit that signalled s_full was issued after it.
#pragma unroll 1
          for (int q2 = 0; q2 < D / 32; ++q2) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + q2 * 32, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st32(tO + q2 * 32, o);
          }
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->p_ready[t]));
    }
    // ------------------------------- epilogue ----------------------------------------------------
    const bool have_o = ok && idx > 0;
    if (have_o) {
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->pv_done[t]), 0, lim_ms, a.err);
      ptx::tc_fence_after();
    }
    const bool any = l_run > 0.f;
    const float inv = any ? 1.f / l_run : 0.f;
    const size_t row = (size_t)g.bh * a.N + i;     // this query row of the [B*H, N] axis
    uint16_t* orow = static_cast<uint16_t*>(a.o) + row * D;
#pragma unroll 1
    for (int q2 = 0; q2 < D / 32; ++q2) {
      uint32_t o[32];
      if (have_o && ok) {
        ptx::tmem_ld32(tO + q2 * 32, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (i < g.N) {
        uint4* dst = reinterpret_cast<uint4*>(orow + q2 * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint4 w;
          w.x = ptx::pack2<F16>(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
          w.y = ptx::pack2<F16>(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
          w.z = ptx::pack2<F16>(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
          w.w = ptx::pack2<F16>(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
          dst[v4] = w;
        }
      }
    }
    if (i < g.N) a.lse[row] = any ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 9) ptx::tmem_dealloc(tmem, kTmemCols);
}

// [slices, N, 64] 16-bit tensor; boxes of 64 columns x `rows` rows
cudaError_t make_map(CUtensorMap* m, const void* base, int N, int BH, int rows, bool f16) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tensor_map(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool F16>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.N, a.B * a.H, BM, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.Nk, a.B * a.Hkv, BN, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mv, a.v, a.Nk, a.B * a.Hkv, BN, F16)) != cudaSuccess) return e;
  auto kern = fwd_bn64_sm103_kernel<F16>;
  const int smem = Cfg<F16>::kSmem;
  // The warp groups re-split the CTA's registers; that only completes if the launch holds at
  // least that many.
  static LaunchSetup setup;
  int regs = 0;
  if ((e = prepare_launch(setup, kern, smem, &regs)) != cudaSuccess) return e;
  if (regs * kThreads < 128 * kRegsOther + 256 * kRegsSoftmax) return cudaErrorInvalidConfiguration;
  // Two CTAs per SM need the largest shared-memory carve-out (asked for once per device).
  static std::atomic<int> carve_set[LaunchSetup::kDevices] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < LaunchSetup::kDevices;
  if (!cached || carve_set[dev].load(std::memory_order_acquire) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (cached) carve_set[dev].store(1, std::memory_order_release);
  }
  const int grid = ((a.N + 2 * BM - 1) / (2 * BM)) * a.B * a.H;
  kern<<<grid, kThreads, smem, s>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bn64_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (a.d != 64 || a.drop.enabled || a.plan != nullptr || a.block_mask != nullptr || a.cu_seqlens != nullptr ||
      a.n_splits != 1 || a.o_part != nullptr || a.Nk != a.N || a.rows != a.N)
    return cudaErrorInvalidValue;
  return dt == FA_FP16 ? launch<true>(a, s) : launch<false>(a, s);
}

}  // namespace fa
