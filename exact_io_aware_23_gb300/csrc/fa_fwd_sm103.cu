// Tensor-core attention forward for sm_103a (bf16 or fp16 in, fp32 accumulate), d in {64, 128}.
//
// The method ("FlashAttention paper story", tiling and online-softmax paragraphs; "FlashAttention：
// 让精确注意力服从内存层次", section "Online softmax" and its merge law): Q is cut into row
// tiles, K/V into column tiles; each query row keeps a running maximum m and normaliser l and an
// un-normalised output; scores and probabilities of one tile live only on chip.  O = u / l and
// LSE = m + ln l are written once at the end.
//
// GB300 design (one CTA = two 128-row Q tiles of one (b, h) slice, 384 threads):
//   warp 8      TMA producer: Q tiles once, then K_j for every live key tile j through a ring of
//               shared-memory slots (mbarrier full/empty pairs).  Masked tiles are never loaded
//               ("FlashAttention paper story", block-sparse paragraph).
//   warp 10     TMA producer of V_j, through a ring of its own.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T (SS MMA, 128 x 128 x d) into TMEM, and
//               O_t += P_t V_j (TS MMA: P_t read from TMEM, V_j from shared memory).
//   warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1: each thread owns one query row
//               (one TMEM lane), reads its 128 scores, masks, updates m and l with exp2, and
//               writes P as bf16 back into the TMEM columns of S.  The two tiles ping-pong, so
//               one tile's softmax overlaps the other tile's MMAs.
//   TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [256+d,256+2d).
// The running maximum is only raised when a row's new maximum exceeds it by more than
// 2^8 (kRescaleLog2): P and l use the same stale maximum, so the result is unchanged and the O
// rescale (a TMEM read-modify-write) is rare.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "dropout_sm103.cuh"
#include "fa_internal.cuh"
#include "fa_sm103.cuh"
#include "ptx_sm103.cuh"

namespace fa {
namespace {

constexpr int BM = 128;          // rows per Q tile
constexpr int BN = 128;          // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : int { kNone = 0, kPartial = 1, kFull = 2 };

template <int D, bool F16>
struct Cfg {
  static constexpr int kTileBytes = BN * D * 2;                 // one K or V tile; one Q tile
  static constexpr int kSlots = D == 128 ? 5 : 8;               // K and V slots in all
  static constexpr int kKSlots = D == 128 ? 3 : 4;              // K ring: slots [0, kKSlots)
  static constexpr int kVSlots = kSlots - kKSlots;              // V ring: the rest
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
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
  int merge_last;        // balanced block-sparse plan: this CTA merges its pair's ranges
};

static_assert(sizeof(Bars) <= 256, "the live-tile bitmap starts 256 bytes after the barriers");

// Per-CTA tile geometry: which key tiles exist and how each Q tile must treat them.
struct Geo {
  int bh;          // (b, h) slice
  int row0;        // first row of the slice on the token axis (packed sequences; else 0)
  int qs, ks;      // slice index of Q/O and of K/V in the tensor maps and row arithmetic
  int split;       // key-tile range (split-KV)
  int j0;          // first key tile of this CTA's range
  int q0;          // first query row of Q tile 0
  int N, kv_lim;   // keys with j >= kv_lim are masked (padding and tail)
  int causal;
  const uint8_t* bm;
  int T;
  int j_end;       // key tiles [0, j_end) may be live

  __device__ int kind(int t, int j) const {
    const int r0 = q0 + t * BM;
    if (r0 >= N) return kNone;
    const int r1 = min(r0 + BM, N) - 1;
    const int c0 = j * BN, c1 = c0 + BN - 1;
    if (bm != nullptr && bm[(size_t)(r0 / BM) * T + j] == 0) return kNone;
    if (c0 >= kv_lim || (causal && c0 > r1)) return kNone;
    if (c1 < kv_lim && (!causal || c1 <= r0)) return kFull;
    return kPartial;
  }
  __device__ bool live(int j) const { return kind(0, j) != kNone || kind(1, j) != kNone; }
  // Without a tile mask the live key tiles are exactly [0, j_end).  With one, `bits` (shared
  // memory, built once per CTA) marks the live tiles and the next one is found a word at a time.
  const uint32_t* bits;
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

// kPlan: the balanced block-sparse variant (a work plan, split pairs, the last range merging);
// a separate instantiation, so the others carry none of its code.
template <int D, bool F16, bool kDrop, bool kPlan>
__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  using C = Cfg<D, F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
  const uint32_t sQ = ptx::smem_u32(smem + C::kQOff);
  const uint32_t sKV = ptx::smem_u32(smem + C::kKVOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  uint32_t* const live_bits = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 256);
  // Each role builds its own copy after its register reallocation (cheap integer work), so no
  // value computed here has to survive, spilled, into the role loops.
  // Balanced block-sparse plan: this CTA's entry {pair, range, ranges, slot}; no work for pair < 0.
  int4 work = make_int4(0, 0, 1, -1);
  if constexpr (kPlan) {
    work = a.plan[blockIdx.x / (a.B * a.H)];
    if (work.x < 0) return;
  }
  // with_range: restrict [j0, j_end) to this CTA's range of live key tiles (needs the bitmap)
  auto make_geo = [&](bool with_range) {
    // Work order.  With masks, the (b, h) slice varies fastest, so every slice's heaviest Q-tile
    // pair runs in the first waves (the last pairs when causal, the global rows of a
    // block-sparse mask).  Without, one slice's pairs run together and share its K/V stream in L2.
    // Split-KV: the range of key tiles varies slowest.  With a plan: slice fastest, then the
    // plan's entries in order (the split ranges first).
    const int BH = a.B * a.H;
    const int n_pairs = (a.N + 2 * BM - 1) / (2 * BM);
    const int unit = blockIdx.x % (n_pairs * BH);
    const int split = kPlan ? 0 : blockIdx.x / (n_pairs * BH);
    const int bh = kPlan ? (int)(blockIdx.x % BH) : a.heads_fastest ? unit % BH : unit / n_pairs;
    const int slot = a.heads_fastest ? unit / BH : unit % n_pairs;
    const int pair = kPlan ? work.x : a.causal ? n_pairs - 1 - slot : slot;
    const int b = bh / a.H, h = bh % a.H;
    Geo g;
    g.bh = bh;
    g.split = split;
    g.q0 = pair * 2 * BM;
    g.N = a.N;
    g.row0 = 0;
    int kvl = a.Nk;
    if (a.cu_seqlens != nullptr) {                 // packed: this sequence's rows of head h
      int len = 0;
      if (!packed_sequence(a.cu_seqlens, b, a.N, a.rows, &g.row0, &len)) g.row0 = -1;
      g.N = kvl = len;
    }
    g.qs = a.cu_seqlens != nullptr ? h : bh;
    // grouped-query attention: query head h reads key/value head h / (H / Hkv)
    g.ks = (a.cu_seqlens != nullptr ? 0 : b * a.Hkv) + h / (a.H / a.Hkv);
    if (a.kv_lens != nullptr) kvl = max(0, min(a.Nk, (int)a.kv_lens[b]));
    g.kv_lim = kvl;
    g.causal = a.causal;
    g.bm = a.block_mask;
    g.T = a.n_tiles;
    int last_key = g.kv_lim;
    if (a.causal) last_key = min(last_key, min(g.q0 + 2 * BM, g.N));
    g.j_end = (last_key + BN - 1) / BN;
    g.j0 = 0;
    if (a.n_splits > 1) {
      g.j0 = min(split * a.tiles_per_split, g.j_end);
      g.j_end = min(g.j_end, g.j0 + a.tiles_per_split);
    }
    g.bits = a.block_mask != nullptr ? live_bits : nullptr;
    if (kPlan && with_range && work.z > 1 && g.bits != nullptr) {
      // range r of S over this CTA's live tiles: live tiles [r c / S, (r + 1) c / S) (the last
      // range to the end), turned into tile indices through the bitmap
      const int words = (g.j_end + 31) / 32;
      int c = 0;
      for (int w = 0; w < words; ++w) c += __popc(g.bits[w]);
      const int lo = (int)(((long long)work.y * c) / work.z);
      const int hi = work.y == work.z - 1 ? c : (int)(((long long)(work.y + 1) * c) / work.z);
      auto tile_of = [&](int k) {             // tile index of live tile number k (j_end if none)
        for (int w = 0; w < words; ++w) {
          uint32_t bits = g.bits[w];
          const int n = __popc(bits);
          if (k < n) {
            for (int i = 0; i < k; ++i) bits &= bits - 1;
            return w * 32 + __ffs(bits) - 1;
          }
          k -= n;
        }
        return g.j_end;
      };
      const int j_hi = hi >= c ? g.j_end : tile_of(hi);
      g.j0 = tile_of(lo);
      g.j_end = j_hi;
    }
    return g;
  };
  const uint32_t lim_ms = a.dbg.wait_limit_ms;
  if (a.cu_seqlens != nullptr) {
    // Packed sequences: the grid is sized for the longest one; tiles past this sequence's end
    // have nothing to do, and offsets outside the contract are reported, not followed.
    const Geo g0 = make_geo(false);
    if (g0.row0 < 0) {
      if (threadIdx.x == 0) atomicExch(a.err, kDevBadOffsets);
      return;
    }
    if (g0.q0 >= g0.N) return;
  }

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
  if (a.block_mask != nullptr) {   // live-tile bitmap, one ballot per 32 tiles, words spread over all warps
    const Geo g = make_geo(false);
    for (int w = warp; w < (g.j_end + 31) / 32; w += kThreads / 32) {
      const int j = w * 32 + lane;
      const uint32_t word = __ballot_sync(0xffffffffu, j < g.j_end && g.live(j));
      if (lane == 0) live_bits[w] = word;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
    ptx::regs_dec<88>();
    const Geo g = make_geo(true);
    if (warp == 8 && lane == 0) {
      // ------------------------------- TMA producer -------------------------------------------
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      const uint32_t qbar = ptx::smem_u32(&bars->q_full);
      ptx::mbar_arrive_expect_tx(qbar, 2 * C::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int hh = 0; hh < D / 64; ++hh)
          ptx::tma_load_3d(sQ + t * C::kTileBytes + hh * BM * 128, &tmQ, qbar, hh * 64, g.row0 + g.q0 + t * BM, g.qs);
      int n = 0;                                   // K tiles issued
      bool ok = true;
      for (int j = g.next(g.j0); j < g.j_end && ok; j = g.next(j + 1), ++n) {
        const int slot = n % C::kKSlots;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[slot]), ((n / C::kKSlots) & 1) ^ 1, lim_ms, a.err);
        if (!ok) break;
        if (a.dbg.inject == 1 && n == 0) continue;      // test hook: never deliver this tile
        const uint32_t fb = ptx::smem_u32(&bars->kv_full[slot]);
        ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
        for (int hh = 0; hh < D / 64; ++hh)
          ptx::tma_load_3d(sKV + slot * C::kTileBytes + hh * BN * 128, &tmK, fb, hh * 64, g.row0 + j * BN, g.ks);
      }
      // Drain: every copy this thread issued must have landed before shared memory is released.
      ptx::mbar_wait(qbar, 0, lim_ms, a.err);
      for (int m = max(0, n - C::kKSlots); m < n; ++m) {
        if (a.dbg.inject == 1 && m == 0) continue;
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[m % C::kKSlots]), (m / C::kKSlots) & 1, lim_ms, a.err);
      }
    } else if (warp == 10 && lane == 0) {
      // ------------------------------- TMA producer of V ------------------------------------
      // K and V have rings of their own, each with its own producer thread, so a K tile (freed
      // as soon as both S products have read it) is refilled without queueing behind a V slot
      // (freed only after both PV products of the next key tile).
      int n = 0;                                   // V tiles issued
      bool ok = true;
      for (int j = g.next(g.j0); j < g.j_end && ok; j = g.next(j + 1), ++n) {
        const int slot = C::kKSlots + n % C::kVSlots;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[slot]), ((n / C::kVSlots) & 1) ^ 1, lim_ms, a.err);
        if (!ok) break;
        const uint32_t fb = ptx::smem_u32(&bars->kv_full[slot]);
        ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
        for (int hh = 0; hh < D / 64; ++hh)
          ptx::tma_load_3d(sKV + slot * C::kTileBytes + hh * BN * 128, &tmV, fb, hh * 64, g.row0 + j * BN, g.ks);
      }
      for (int m = max(0, n - C::kVSlots); m < n; ++m)
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[C::kKSlots + m % C::kVSlots]), (m / C::kVSlots) & 1, lim_ms, a.err);
    } else if (warp == 9 && lane == 0) {
      // ------------------------------- MMA issuer ---------------------------------------------
      bool ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_full), 0, lim_ms, a.err);
      ptx::tc_fence_after();
      int idx = 0;
      int prev_v = -1;
      uint32_t prev_vph = 0;
      for (int j = g.next(g.j0); j < g.j_end && ok; j = g.next(j + 1), ++idx) {
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
              ptx::mma_ts(tmem + 256 + t * D, tmem + t * BN + kk * 8, bdesc, C::kIdescO,
                          (idx > 1 || kk > 0) ? 1u : 0u);
            }
          }
          // S_t = Q_t K_j^T
          const uint32_t qbase = sQ + t * C::kTileBytes;
          const uint32_t kbase = sKV + kslot * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (BM * 128) + (kk % 4) * 32;
            const uint64_t adesc = ptx::sdesc_sw128(qbase + off, 16, 1024);
            const uint64_t bdesc = ptx::sdesc_sw128(kbase + off, 16, 1024);
            ptx::mma_ss(tmem + t * BN, adesc, bdesc, C::kIdescS, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->s_full[t]));
        }
        // No commit frees K_j or V_{j-1}: S_1(j) is issued after every product that reads them,
        // so the softmax of Q tile 1, on seeing S_1(j), frees both (a commit stalls the tensor
        // pipe for about as long as one MMA).
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
            ptx::mma_ts(tmem + 256 + t * D, tmem + t * BN + kk * 8, bdesc, C::kIdescO,
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
    ptx::regs_inc<200>();
    const Geo g = make_geo(true);
    const int t = warp / 4;
    const int sub = warp % 4;
    const int r = sub * 32 + lane;                  // TMEM lane == row within the Q tile
    const int i = g.q0 + t * BM + r;                // query row in the head
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const float c = a.scale * kLog2e;               // scores -> log2 domain
    int row_lim = g.kv_lim;
    if (a.causal) row_lim = min(row_lim, i + 1);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int idx = 0;
    const uint32_t tq = (uint32_t)lane & 3u;       // this row within its 4-row dropout block
    DropTest dtest{};
    if constexpr (kDrop) dtest = drop_test(a.drop);
    for (int j = g.next(g.j0); j < g.j_end; j = g.next(j + 1), ++idx) {
      // how this Q tile treats key tile j (under a tile mask a read of the mask: issued before the
      // wait for S, so its latency does not delay the loads of S)
      const int kind = g.kind(t, j);
      // dropout: this row's drop flags for the tile's 128 keys, 16 per word (generated while the
      // scores are still being computed; the quad shares its calls)
      uint32_t flags[8];
      if constexpr (kDrop) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 r = philox4x32_10((uint32_t)(j * BN / 4) + 4u * m + tq, (uint32_t)i >> 2, (uint32_t)g.bh,
                                        a.drop.offset, a.drop);
          flags[m] = gather_row_flags(pack_flags(r, dtest), tq);
        }
      }
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
        ptx::tmem_st32(tS + 32, pk);
      } else {
        float s[BN];
        {
          uint32_t raw[4][32];                       // all 128 scores, one wait
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) ptx::tmem_ld32(tS + q4 * 32, raw[q4]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            ptx::reg_fence(raw[q4]);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[q4 * 32 + e] = __uint_as_float(raw[q4][e]);
          }
        }
        if (kind == kPartial) {
          const int lim = row_lim - j * BN;
#pragma unroll
          for (int e = 0; e < BN; ++e) s[e] = e < lim ? s[e] : -INFINITY;
        }
        float m8[8];                                 // 8 independent 3-input-max chains
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
        for (int q = 8; q < BN / 2; ++q) m8[q & 7] = ptx::max3(m8[q & 7], s[2 * q], s[2 * q + 1]);
        const float mx = ptx::max3(ptx::max3(m8[0], m8[1], m8[2]), ptx::max3(m8[3], m8[4], m8[5]),
                                   fmaxf(m8[6], m8[7]));
        const float m_cand = mx * c;
        const bool need = m_cand > m_run + kRescaleLog2;   // false when the row is still empty
        const float alpha = need ? ptx::ex2(m_run - m_cand) : 1.f;
        if (__any_sync(0xffffffffu, need) && idx > 0) {
          // O_t *= alpha for this warp's rows (PV of the previous tile has completed: the
          // commit that signalled s_full was issued after it).
#pragma unroll 1
          for (int q4 = 0; q4 < D / 32; ++q4) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + q4 * 32, o);
            ptx::tmem_wait_ld();
            ptx::reg_fence(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st32(tO + q4 * 32, o);
          }
        }
        if (need) {
          l_run *= alpha;
          m_run = m_cand;
        }
        const float msub = m_run == -INFINITY ? 0.f : m_run;
        // p = exp2(s*c - m) on column pairs; 4 independent packed partial sums
        const float2 c2 = make_float2(c, c), nm2 = make_float2(-msub, -msub);
        float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = ptx::fma2(make_float2(s[half * 64 + 2 * e], s[half * 64 + 2 * e + 1]), c2, nm2);
            const float2 pp = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            ls[e & 3] = ptx::add2(ls[e & 3], pp);      // the normaliser counts every allowed key
            if constexpr (kDrop) {                  // keys 4u + 2h, 4u + 2h + 1 of word half*4 + e/8
              const uint32_t u = ((uint32_t)e >> 1) & 3u;
              const uint32_t x = flags[half * 4 + e / 8] << (u ^ tq);
              pk[e] = ptx::pack2<F16>(pp.x, pp.y) & ~row_pair_mask(x, e & 1);
            } else {
              pk[e] = ptx::pack2<F16>(pp.x, pp.y);
            }
          }
          ptx::tmem_st32(tS + half * 32, pk);
        }
        const float2 lsum = ptx::add2(ptx::add2(ls[0], ls[1]), ptx::add2(ls[2], ls[3]));
        l_run += lsum.x + lsum.y;
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
    const float inv = any ? (kDrop ? a.drop.scale : 1.f) / l_run : 0.f;
    const size_t row = (size_t)g.qs * a.rows + g.row0 + i;      // this query row on its axis
    uint16_t* orow = static_cast<uint16_t*>(a.o) + row * D;
    // split-KV, or a split pair of a balanced plan: this range's normalised partial output (fp32)
    // and log-sum-exp
    const bool planned_split = kPlan && work.z > 1;
    const size_t prow = planned_split ? ((size_t)g.bh * a.n_slots + work.w) * (2 * BM) + (i - g.q0)
                                      : (size_t)g.split * a.B * a.H * a.N + row;
    float* porow = (a.o_part != nullptr && (!kPlan || planned_split)) ? a.o_part + prow * D : nullptr;
#pragma unroll 1
    for (int q4 = 0; q4 < D / 32; ++q4) {
      uint32_t o[32];
      if (have_o && ok) {
        ptx::tmem_ld32(tO + q4 * 32, o);
        ptx::tmem_wait_ld();
        ptx::reg_fence(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (i < g.N && porow != nullptr) {
        float4* dst = reinterpret_cast<float4*>(porow + q4 * 32);
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4)
          dst[v4] = make_float4(__uint_as_float(o[4 * v4 + 0]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
      } else if (i < g.N) {
        uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
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
    if (i < g.N) {
      const float L = any ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      if (porow != nullptr) a.lse_part[prow] = L;
      else a.lse[row] = L;
    }
    if (kPlan && planned_split) {
      // The range that finishes last merges the pair's S ranges, always in range order, with the
      // merge law: w_r = exp(LSE_r - max LSE), O = sum w_r O_r / sum w_r, LSE = max + ln sum w_r.
      __threadfence();                               // this range's partials, before the count
      ptx::named_bar_sync(1, 256);                   // the eight softmax warps
      const int first = work.w - work.y;             // the pair's first slot (its counter)
      if (threadIdx.x == 0) {
        const int prev = atomicAdd(a.merge_count + (size_t)g.bh * a.n_slots + first, 1);
        bars->merge_last = prev == work.z - 1 ? 1 : 0;
      }
      ptx::named_bar_sync(1, 256);
      if (bars->merge_last != 0 && i < g.N) {
        __threadfence();
        const size_t base = ((size_t)g.bh * a.n_slots + first) * (2 * BM) + (i - g.q0);
        float mx = -INFINITY;
        for (int r = 0; r < work.z; ++r) mx = fmaxf(mx, __ldcg(a.lse_part + base + (size_t)r * (2 * BM)));
        float wsum = 0.f;
        if (mx != -INFINITY)
          for (int r = 0; r < work.z; ++r) {
            const float L = __ldcg(a.lse_part + base + (size_t)r * (2 * BM));
            wsum += L == -INFINITY ? 0.f : ptx::ex2((L - mx) * kLog2e);
          }
        const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll 1
        for (int q4 = 0; q4 < D / 32; ++q4) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
          if (mx != -INFINITY)
            for (int r = 0; r < work.z; ++r) {
              const size_t pr = base + (size_t)r * (2 * BM);
              const float L = __ldcg(a.lse_part + pr);
              if (L == -INFINITY) continue;
              const float w = ptx::ex2((L - mx) * kLog2e);
              const float4* src = reinterpret_cast<const float4*>(a.o_part + pr * D + q4 * 32);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4) {
                const float4 x = __ldcg(src + v4);
                acc[4 * v4 + 0] = fmaf(w, x.x, acc[4 * v4 + 0]);
                acc[4 * v4 + 1] = fmaf(w, x.y, acc[4 * v4 + 1]);
                acc[4 * v4 + 2] = fmaf(w, x.z, acc[4 * v4 + 2]);
                acc[4 * v4 + 3] = fmaf(w, x.w, acc[4 * v4 + 3]);
              }
            }
          uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = ptx::pack2<F16>(acc[8 * v4 + 0] * winv, acc[8 * v4 + 1] * winv);
            w.y = ptx::pack2<F16>(acc[8 * v4 + 2] * winv, acc[8 * v4 + 3] * winv);
            w.z = ptx::pack2<F16>(acc[8 * v4 + 4] * winv, acc[8 * v4 + 5] * winv);
            w.w = ptx::pack2<F16>(acc[8 * v4 + 6] * winv, acc[8 * v4 + 7] * winv);
            dst[v4] = w;
          }
        }
        a.lse[row] = wsum > 0.f ? mx + log2f(wsum) * kLn2 : -INFINITY;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 9) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---- host side -----------------------------------------------------------------------------------

cudaError_t make_map(CUtensorMap* m, const void* base, int D, int N, int BH, bool f16) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tensor_map(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, bool F16, bool kDrop, bool kPlan>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  // token axis and slice count of the tensor maps: per (b, h) slice, or packed per head
  const bool packed = a.cu_seqlens != nullptr;
  const int q_slices = packed ? a.H : a.B * a.H, kv_slices = packed ? a.Hkv : a.B * a.Hkv;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, D, a.rows, q_slices, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, D, packed ? a.rows : a.Nk, kv_slices, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mv, a.v, D, packed ? a.rows : a.Nk, kv_slices, F16)) != cudaSuccess) return e;
  auto kern = fwd_sm103_kernel<D, F16, kDrop, kPlan>;
  // + the live-tile bitmap of a block-sparse mask (one bit per key tile)
  const int smem = Cfg<D, F16>::kSmem + (a.block_mask != nullptr ? ((a.n_tiles + 127) / 128) * 16 : 0);
  // The warp groups re-split the CTA's registers (4 warps down to 88, 8 warps up to 200 per
  // thread); that only completes if the launch holds at least that many registers.
  static LaunchSetup setup;
  int regs = 0;
  if ((e = prepare_launch(setup, kern, smem, &regs)) != cudaSuccess) return e;
  if (regs * kThreads < 128 * 88 + 256 * 200) return cudaErrorInvalidConfiguration;
  dim3 grid(kPlan ? a.plan_entries * a.B * a.H : ((a.N + 2 * BM - 1) / (2 * BM)) * a.B * a.H * a.n_splits);
  kern<<<grid, kThreads, smem, s>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (a.drop.enabled) {
    if (a.plan != nullptr) return cudaErrorInvalidValue;     // no plan with dropout
    if (dt == FA_FP16) return a.d == 64 ? launch<64, true, true, false>(a, s) : launch<128, true, true, false>(a, s);
    return a.d == 64 ? launch<64, false, true, false>(a, s) : launch<128, false, true, false>(a, s);
  }
  if (a.plan != nullptr) {
    // at d = 64 the persistent kernel of fa_fwd_bs_persist_sm103.cu
    if (a.d == 64) return launch_fwd_bs_persist_sm103(a, dt, s);
    return dt == FA_FP16 ? launch<128, true, false, true>(a, s) : launch<128, false, false, true>(a, s);
  }
  // d = 64 without a tile mask, packing or split-KV: the two-CTAs-per-SM kernel of
  // fa_fwd_bn64_sm103.cu (64-key tiles), faster than this one at every length measured.
  if (a.d == 64 && a.block_mask == nullptr && a.cu_seqlens == nullptr && a.n_splits == 1 &&
      a.o_part == nullptr && a.Nk == a.N)
    return launch_fwd_bn64_sm103(a, dt, s);
  if (dt == FA_FP16) return a.d == 64 ? launch<64, true, false, false>(a, s) : launch<128, true, false, false>(a, s);
  return a.d == 64 ? launch<64, false, false, false>(a, s) : launch<128, false, false, false>(a, s);
}

}  // namespace fa
