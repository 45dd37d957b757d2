// Persistent balanced block-sparse attention forward for sm_103a, d = 64 (bf16 or fp16 in, fp32
// accumulate): fa_forward_blocksparse's kernel at that head size.
//
// The method and the per-tile pipeline are those of fa_fwd_sm103.cu ("FlashAttention paper
// story", tiling, online-softmax and block-sparse paragraphs; "FlashAttention：让精确注意力服从内存
// 层次", sections "Online softmax" and its merge law): two 128-row Q tiles per unit, K/V tiles
// through rings, S and O in TMEM, the softmax warpgroups ping-ponging, split ranges merged by the
// last range to finish.  What differs is the execution: one CTA per SM runs unit after unit
// (plan entry x slice), claimed in plan order from a counter in the plan's workspace by the
// producer warp and handed to the other roles through two entries in shared memory (with the
// pair's live-tile bitmap, which the plan's counting kernel wrote); Q has two buffers, ring
// positions and barrier phases count across units, and the split ranges' merge synchronises the
// softmax warps through mbarriers with bounded waits.  So the next unit's copies and first
// products run during the current unit's last tiles and epilogue, which at the block-sparse
// workload's dozen key tiles a unit were about 30 % of a CTA's time.  (Applied to every forward
// launch the same structure measured slower on the short dense shapes, so only this one uses it.)
//
// Inputs as fa_forward_blocksparse takes them: [B, H, N, 64] Q and O, [B, Hkv, N, 64] K and V,
// a tile mask, optional causal mask and key lengths; no packing, dropout or split-KV here.
//
// GB300 layout of one CTA (384 threads): warp 8 producer (Q, K), warp 10 producer (V), warp 9 MMA
// issuer, warps 0-7 softmax; TMEM S_0 [0,128), S_1 [128,256), O_0 [256,320), O_1 [320,384).
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
constexpr int BN = 128;          // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kBarBytes = 320;   // the barrier area; the two unit entries follow

enum : int { kNone = 0, kPartial = 1, kFull = 2 };

template <bool F16>
struct Cfg {
  static constexpr int kTileBytes = BN * D * 2;                 // one K or V tile; one Q tile
  static constexpr int kSlots = 8;                              // K and V slots in all
  static constexpr int kKSlots = 4;                             // K ring: slots [0, kKSlots)
  static constexpr int kVSlots = kSlots - kKSlots;              // V ring: the rest
  static constexpr int kQOff = 0;                               // Q buffer 0 (two Q tiles)
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kQ1Off = kKVOff + kSlots * kTileBytes;   // Q buffer 1
  static constexpr int kBarOff = kQ1Off + 2 * kTileBytes;
  static constexpr int kSmem = kBarOff + kBarBytes + 1024;      // + barriers + alignment slack
  static constexpr uint32_t kIdescS = ptx::idesc_f32acc(BM, BN, false, false, F16);
  static constexpr uint32_t kIdescO = ptx::idesc_f32acc(BM, D, false, true, F16);
};

struct Bars {              // all mbarriers of one CTA (8 bytes each)
  uint64_t q_full[2];      // Q buffer b holds its unit's two Q tiles
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t pv_done[2];
  uint64_t mma_done;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t unit_full[2];   // unit entry e published (by the producer warp)
  uint64_t unit_empty[2];  // unit entry e released (V producer, MMA, 8 softmax warps)
  uint64_t q_free[2];      // every product reading Q buffer b has completed
  uint64_t merge_in;       // the eight softmax warps have written a split unit's partials
  uint64_t merge_out;      // ... and the last-range decision is made
  uint32_t tmem_base;
  int merge_last;          // this CTA merges its pair's ranges
};

static_assert(sizeof(Bars) <= kBarBytes, "the unit entries start kBarBytes after the barriers");

// A unit handed from the producer warp to the others (two entries after the barriers): the unit
// (plan entry x slices + slice; -1 = no more) and its pair's live key tiles, one bit per tile.
struct UnitEntry {
  int unit;
  int pad[3];
  uint32_t bits[4];        // [words] in fact (UnitEntry::bytes)
  static __host__ __device__ int bytes(int words) { return 16 + ((4 * words + 15) / 16) * 16; }
};
constexpr int kUnitEnd = -1;

// One unit's tile geometry: which key tiles exist and how each Q tile must treat them.
struct Geo {
  int bh;          // (b, h) slice: Q/O slice index in the tensor maps
  int ks;          // K/V slice index
  int j0;          // first key tile of this unit's range
  int q0;          // first query row of Q tile 0
  int N, kv_lim;   // keys with j >= kv_lim are masked (padding and tail)
  int causal;
  const uint8_t* bm;
  int T;
  int j_end;       // key tiles [j0, j_end) may be live
  const uint32_t* bits;   // live key tiles of the pair (shared memory), or null: all of [j0, j_end)

  __device__ int kind(int t, int j) const {
    const int r0 = q0 + t * BM;
    if (r0 >= N) return kNone;
    const int r1 = min(r0 + BM, N) - 1;
    const int c0 = j * BN, c1 = c0 + BN - 1;
    if (bm[(size_t)(r0 / BM) * T + j] == 0) return kNone;
    if (c0 >= kv_lim || (causal && c0 > r1)) return kNone;
    if (c1 < kv_lim && (!causal || c1 <= r0)) return kFull;
    return kPartial;
  }
  // the next live key tile at or after j (j_end if none), a bitmap word at a time
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

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bs_persist_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  using C = Cfg<F16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
  const uint32_t sQ = ptx::smem_u32(smem + C::kQOff);
  const uint32_t sQ1 = ptx::smem_u32(smem + C::kQ1Off);
  const uint32_t sKV = ptx::smem_u32(smem + C::kKVOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int BHs = a.B * a.H;
  const int ent_bytes = UnitEntry::bytes(a.bit_words);
  auto entry = [&](int e) {
    return reinterpret_cast<UnitEntry*>(smem + C::kBarOff + kBarBytes + e * ent_bytes);
  };
  auto entry_bits = [&](int e) { return reinterpret_cast<uint32_t*>(smem + C::kBarOff + kBarBytes + e * ent_bytes + 16); };
  // The geometry of unit x, whose plan entry is wk = {pair, range, ranges, slot}: the (b, h)
  // slice varies fastest, then the plan's entries in order (the split ranges first).  With
  // with_range the key tiles are restricted to the unit's range of the pair's live tiles (needs
  // the bitmap `bits`).
  auto make_geo = [&](int x, const int4 wk, const uint32_t* bits, bool with_range) {
    const int bh = x % BHs;
    const int b = bh / a.H, h = bh % a.H;
    Geo g;
    g.bh = bh;
    g.q0 = wk.x * 2 * BM;
    g.N = a.N;
    // grouped-query attention: query head h reads key/value head h / (H / Hkv)
    g.ks = b * a.Hkv + h / (a.H / a.Hkv);
    g.kv_lim = a.kv_lens != nullptr ? max(0, min(a.Nk, (int)a.kv_lens[b])) : a.Nk;
    g.causal = a.causal;
    g.bm = a.block_mask;
    g.T = a.n_tiles;
    int last_key = g.kv_lim;
    if (a.causal) last_key = min(last_key, min(g.q0 + 2 * BM, g.N));
    g.j_end = (last_key + BN - 1) / BN;
    g.j0 = 0;
    g.bits = bits;
    if (with_range && wk.z > 1 && bits != nullptr) {
      // range r of S over the pair's live tiles: live tiles [r c / S, (r + 1) c / S) (the last
      // range to the end), turned into tile indices through the bitmap
      const int words = (g.j_end + 31) / 32;
      int c = 0;
      for (int w = 0; w < words; ++w) c += __popc(bits[w]);
      const int lo = (int)(((long long)wk.y * c) / wk.z);
      const int hi = wk.y == wk.z - 1 ? c : (int)(((long long)(wk.y + 1) * c) / wk.z);
      auto tile_of = [&](int k) {             // tile index of live tile number k (j_end if none)
        for (int w = 0; w < words; ++w) {
          uint32_t word = bits[w];
          const int n = __popc(word);
          if (k < n) {
            for (int i = 0; i < k; ++i) word &= word - 1;
            return w * 32 + __ffs(word) - 1;
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
  // the unit that entry e holds (kUnitEnd: none), after waiting for it to be published
  auto take_unit = [&](int u, int* e, int4* wk, const uint32_t** bits, bool* ok) {
    *e = u & 1;
    *ok = ptx::mbar_wait(ptx::smem_u32(&bars->unit_full[*e]), (u >> 1) & 1, a.dbg.wait_limit_ms, a.err);
    if (!*ok) return kUnitEnd;
    const int x = *reinterpret_cast<volatile const int*>(&entry(*e)->unit);
    if (x == kUnitEnd) return kUnitEnd;
    *wk = a.plan[x / BHs];
    *bits = entry_bits(*e);
    return x;
  };
  const uint32_t lim_ms = a.dbg.wait_limit_ms;

  if (warp == 8 && lane == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->q_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->q_full[1]), 1);
    for (int e = 0; e < 2; ++e) {
      ptx::mbar_init(ptx::smem_u32(&bars->unit_full[e]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->unit_empty[e]), 10);   // V producer, MMA, 8 softmax warps
      ptx::mbar_init(ptx::smem_u32(&bars->q_free[e]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->merge_in), 8);
    ptx::mbar_init(ptx::smem_u32(&bars->merge_out), 1);
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
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
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
    ptx::regs_dec<88>();
    if (warp == 8) {
      // ------------------------------- producer warp ------------------------------------------
      // Claims the units with work in plan order, publishes each with its pair's live tiles
      // (clipped to the unit's key range), then copies its Q (buffers alternate between units)
      // and its K tiles into the ring.
      const int total = a.plan_entries * BHs;
      int u = 0;                                   // units published
      int n = 0;                                   // K tiles issued
      bool ok = true;
      while (ok) {
        int x = 0;
        int4 wk = make_int4(-1, 0, 0, 0);
        do {
          if (lane == 0) x = atomicAdd(a.next_unit, 1);
          x = __shfl_sync(0xffffffffu, x, 0);
          if (x >= total) break;
          wk = a.plan[x / BHs];
        } while (wk.x < 0);
        const bool done = x >= total;
        const int e = u & 1;
        if (lane == 0) ok = ptx::mbar_wait(ptx::smem_u32(&bars->unit_empty[e]), ((u >> 1) & 1) ^ 1, lim_ms, a.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        UnitEntry* ent = entry(e);
        uint32_t* ebits = entry_bits(e);
        if (!done) {
          const Geo g0 = make_geo(x, wk, nullptr, false);
          const uint32_t* src = a.pair_bits + (size_t)wk.x * a.bit_words;
          for (int w = lane; w < a.bit_words; w += 32) {
            uint32_t b = src[w];
            const int lo = w * 32;
            if (lo >= g0.j_end) b = 0u;
            else if (g0.j_end - lo < 32) b &= (1u << (g0.j_end - lo)) - 1u;
            ebits[w] = b;
          }
        }
        __syncwarp();
        if (lane == 0) {
          ent->unit = done ? kUnitEnd : x;
          ptx::mbar_arrive(ptx::smem_u32(&bars->unit_full[e]));
        }
        if (done) break;
        if (lane == 0) {
          const Geo g = make_geo(x, wk, ebits, true);
          const int qb = u & 1;
          // Q buffer qb is free once every product of the unit before last has completed
          if (u >= 2) ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_free[qb]), ((u >> 1) - 1) & 1, lim_ms, a.err);
          if (ok) {
            const uint32_t qbar = ptx::smem_u32(&bars->q_full[qb]);
            const uint32_t qdst = qb ? sQ1 : sQ;
            ptx::mbar_arrive_expect_tx(qbar, 2 * C::kTileBytes);
            for (int t = 0; t < 2; ++t)
              ptx::tma_load_3d(qdst + t * C::kTileBytes, &tmQ, qbar, 0, g.q0 + t * BM, g.bh);
          }
          for (int j = g.next(g.j0); j < g.j_end && ok; j = g.next(j + 1), ++n) {
            const int slot = n % C::kKSlots;
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[slot]), ((n / C::kKSlots) & 1) ^ 1, lim_ms, a.err);
            if (!ok) break;
            const uint32_t fb = ptx::smem_u32(&bars->kv_full[slot]);
            ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
            ptx::tma_load_3d(sKV + slot * C::kTileBytes, &tmK, fb, 0, j * BN, g.ks);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++u;
      }
      // Drain: every copy this warp issued must have landed before shared memory is released.
      if (lane == 0) {
        for (int m = max(0, u - 2); m < u; ++m)
          ptx::mbar_wait(ptx::smem_u32(&bars->q_full[m & 1]), (m >> 1) & 1, lim_ms, a.err);
        for (int m = max(0, n - C::kKSlots); m < n; ++m)
          ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[m % C::kKSlots]), (m / C::kKSlots) & 1, lim_ms, a.err);
      }
    } else if (warp == 10 && lane == 0) {
      // ------------------------------- TMA producer of V ------------------------------------
      // K and V have rings of their own, each with its own producer thread, so a K tile (freed
      // as soon as both S products have read it) is refilled without queueing behind a V slot
      // (freed only after both PV products of the next key tile).
      int u = 0;                                   // units run
      int n = 0;                                   // V tiles issued
      bool ok = true;
      while (ok) {
        int e = 0;
        int4 wk;
        const uint32_t* bits = nullptr;
        const int x = take_unit(u, &e, &wk, &bits, &ok);
        if (x == kUnitEnd) break;
        const Geo g = make_geo(x, wk, bits, true);
        for (int j = g.next(g.j0); j < g.j_end && ok; j = g.next(j + 1), ++n) {
          const int slot = C::kKSlots + n % C::kVSlots;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_empty[slot]), ((n / C::kVSlots) & 1) ^ 1, lim_ms, a.err);
          if (!ok) break;
          const uint32_t fb = ptx::smem_u32(&bars->kv_full[slot]);
          ptx::mbar_arrive_expect_tx(fb, C::kTileBytes);
          ptx::tma_load_3d(sKV + slot * C::kTileBytes, &tmV, fb, 0, j * BN, g.ks);
        }
        ptx::mbar_arrive(ptx::smem_u32(&bars->unit_empty[e]));
        ++u;
      }
      for (int m = max(0, n - C::kVSlots); m < n; ++m)
        ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[C::kKSlots + m % C::kVSlots]), (m / C::kVSlots) & 1, lim_ms, a.err);
    } else if (warp == 9 && lane == 0) {
      // ------------------------------- MMA issuer ---------------------------------------------
      int u = 0;                                   // units run
      int rr = 0;                                  // key tiles run: ring positions and phases
      bool ok = true;
      while (ok) {
        int e = 0;
        int4 wk;
        const uint32_t* bits = nullptr;
        const int x = take_unit(u, &e, &wk, &bits, &ok);
        if (x == kUnitEnd) break;
        const Geo g = make_geo(x, wk, bits, true);
        const int qb = u & 1;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->q_full[qb]), (uint32_t)((u >> 1) & 1), lim_ms, a.err);
        ptx::tc_fence_after();
        const uint32_t sQu = qb ? sQ1 : sQ;
        int idx = 0;
        int prev_v = -1;
        uint32_t prev_vph = 0;
        for (int j = g.next(g.j0); j < g.j_end && ok; j = g.next(j + 1), ++idx, ++rr) {
          const int kslot = rr % C::kKSlots;
          const uint32_t kph = (rr / C::kKSlots) & 1;
          const int vslot = C::kKSlots + rr % C::kVSlots;
          const uint32_t vph = (rr / C::kVSlots) & 1;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[kslot]), kph, lim_ms, a.err);
          if (ok && idx > 0) ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[prev_v]), prev_vph, lim_ms, a.err);
          if (!ok) break;
          ptx::tc_fence_after();
          for (int t = 0; t < 2 && ok; ++t) {
            if (idx > 0) {
              // O_t += P_t V_{j_prev}: P_t of the previous key tile sits in S_t's columns.
              ok = ptx::mbar_wait(ptx::smem_u32(&bars->p_ready[t]), (rr - 1) & 1, lim_ms, a.err);
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
            const uint32_t qbase = sQu + t * C::kTileBytes;
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
          // so the softmax of Q tile 1, on seeing S_1(j), frees both (a commit stalls the tensor
          // pipe for about as long as one MMA).
          prev_v = vslot;
          prev_vph = vph;
        }
        if (ok && idx > 0) {
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->kv_full[prev_v]), prev_vph, lim_ms, a.err);
          ptx::tc_fence_after();
          for (int t = 0; t < 2 && ok; ++t) {
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->p_ready[t]), (rr - 1) & 1, lim_ms, a.err);
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
        // every product of this unit, the last readers of Q buffer qb among them, is issued
        ptx::mma_commit(ptx::smem_u32(&bars->q_free[qb]));
        ptx::mbar_arrive(ptx::smem_u32(&bars->unit_empty[e]));
        ++u;
      }
      // every MMA this thread issued has finished before TMEM and shared memory are released
      ptx::mma_commit(ptx::smem_u32(&bars->mma_done));
      ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, lim_ms, a.err);
    }
  } else {
    // ------------------------------- softmax warpgroups -----------------------------------------
    ptx::regs_inc<200>();
    const int t = warp / 4;
    const int sub = warp % 4;
    const int r = sub * 32 + lane;                  // TMEM lane == row within the Q tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const float c = a.scale * kLog2e;               // scores -> log2 domain
    int u = 0;                                      // units run
    int rr = 0;                                     // key tiles run: barrier phases
    int nv = 0;                                     // units whose O received products
    int ns = 0;                                     // split units merged
    bool ok = true;
    while (ok) {
      int e = 0;
      int4 wk;
      const uint32_t* bits = nullptr;
      const int x = take_unit(u, &e, &wk, &bits, &ok);
      if (x == kUnitEnd) break;
      const Geo g = make_geo(x, wk, bits, true);
      const int i = g.q0 + t * BM + r;              // query row in the head
      int row_lim = g.kv_lim;
      if (a.causal) row_lim = min(row_lim, i + 1);
      float m_run = -INFINITY, l_run = 0.f;
      int idx = 0;
      for (int j = g.next(g.j0); j < g.j_end; j = g.next(j + 1), ++idx, ++rr) {
        // how this Q tile treats key tile j (a read of the mask: issued before the wait for S, so
        // its latency does not delay the loads of S)
        const int kind = g.kind(t, j);
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->s_full[t]), rr & 1, lim_ms, a.err);
        if (!ok) break;
        ptx::tc_fence_after();
        if (t == 1 && sub == 0 && lane == 0) {
          // S_1(j) has completed, and with it every MMA issued before it: both S products of key
          // tile j (K_j's slot is free) and both PV products of the previous tile (V's slot too).
          ptx::mbar_arrive(ptx::smem_u32(&bars->kv_empty[rr % C::kKSlots]));
          if (idx > 0) ptx::mbar_arrive(ptx::smem_u32(&bars->kv_empty[C::kKSlots + (rr - 1) % C::kVSlots]));
        }
        uint32_t pk[32];
        if (kind == kNone) {
#pragma unroll
          for (int q = 0; q < 32; ++q) pk[q] = 0u;
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
              for (int q = 0; q < 32; ++q) s[q4 * 32 + q] = __uint_as_float(raw[q4][q]);
            }
          }
          if (kind == kPartial) {
            const int lim = row_lim - j * BN;
#pragma unroll
            for (int q = 0; q < BN; ++q) s[q] = q < lim ? s[q] : -INFINITY;
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
              for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
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
            for (int q = 0; q < 32; ++q) {
              const float2 y = ptx::fma2(make_float2(s[half * 64 + 2 * q], s[half * 64 + 2 * q + 1]), c2, nm2);
              const float2 pp = make_float2(ptx::ex2(y.x), ptx::ex2(y.y));
              ls[q & 3] = ptx::add2(ls[q & 3], pp);      // the normaliser counts every allowed key
              pk[q] = ptx::pack2<F16>(pp.x, pp.y);
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
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->pv_done[t]), (uint32_t)(nv & 1), lim_ms, a.err);
        ptx::tc_fence_after();
        // both PV products of the unit's last key tile have completed: its V slot is free
        if (t == 1 && sub == 0 && lane == 0)
          ptx::mbar_arrive(ptx::smem_u32(&bars->kv_empty[C::kKSlots + (rr - 1) % C::kVSlots]));
        ++nv;
      }
      const bool any = l_run > 0.f;
      const float inv = any ? 1.f / l_run : 0.f;
      const size_t row = (size_t)g.bh * a.rows + i;      // this query row on its axis
      uint16_t* orow = static_cast<uint16_t*>(a.o) + row * D;
      // a split pair: this range's normalised partial output (fp32) and log-sum-exp
      const bool split = wk.z > 1;
      const size_t prow = ((size_t)g.bh * a.n_slots + wk.w) * (2 * BM) + (i - g.q0);
      float* porow = split ? a.o_part + prow * D : nullptr;
#pragma unroll 1
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t o[32];
        if (have_o && ok) {
          ptx::tmem_ld32(tO + q4 * 32, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence(o);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = 0u;
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
      if (split) {
        // The range that finishes last merges the pair's S ranges, always in range order, with the
        // merge law: w_r = exp(LSE_r - max LSE), O = sum w_r O_r / sum w_r, LSE = max + ln sum w_r.
        // The eight softmax warps meet through barriers with bounded waits (a warp that gave up
        // on a unit must not leave the others blocked).
        __threadfence();                               // this range's partials, before the count
        const int first = wk.w - wk.y;                 // the pair's first slot (its counter)
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->merge_in));
        if (threadIdx.x == 0) {
          ptx::mbar_wait(ptx::smem_u32(&bars->merge_in), ns & 1, lim_ms, a.err);
          const int prev = atomicAdd(a.merge_count + (size_t)g.bh * a.n_slots + first, 1);
          bars->merge_last = prev == wk.z - 1 ? 1 : 0;
          ptx::mbar_arrive(ptx::smem_u32(&bars->merge_out));
        }
        ptx::mbar_wait(ptx::smem_u32(&bars->merge_out), ns & 1, lim_ms, a.err);
        ++ns;
        if (bars->merge_last != 0 && i < g.N) {
          __threadfence();
          const size_t base = ((size_t)g.bh * a.n_slots + first) * (2 * BM) + (i - g.q0);
          float mx = -INFINITY;
          for (int k = 0; k < wk.z; ++k) mx = fmaxf(mx, __ldcg(a.lse_part + base + (size_t)k * (2 * BM)));
          float wsum = 0.f;
          if (mx != -INFINITY)
            for (int k = 0; k < wk.z; ++k) {
              const float L = __ldcg(a.lse_part + base + (size_t)k * (2 * BM));
              wsum += L == -INFINITY ? 0.f : ptx::ex2((L - mx) * kLog2e);
            }
          const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll 1
          for (int q4 = 0; q4 < D / 32; ++q4) {
            float acc[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = 0.f;
            if (mx != -INFINITY)
              for (int k = 0; k < wk.z; ++k) {
                const size_t pr = base + (size_t)k * (2 * BM);
                const float L = __ldcg(a.lse_part + pr);
                if (L == -INFINITY) continue;
                const float w = ptx::ex2((L - mx) * kLog2e);
                const float4* src = reinterpret_cast<const float4*>(a.o_part + pr * D + q4 * 32);
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4) {
                  const float4 y = __ldcg(src + v4);
                  acc[4 * v4 + 0] = fmaf(w, y.x, acc[4 * v4 + 0]);
                  acc[4 * v4 + 1] = fmaf(w, y.y, acc[4 * v4 + 1]);
                  acc[4 * v4 + 2] = fmaf(w, y.z, acc[4 * v4 + 2]);
                  acc[4 * v4 + 3] = fmaf(w, y.w, acc[4 * v4 + 3]);
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
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->unit_empty[e]));
      ++u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 9) ptx::tmem_dealloc(tmem, kTmemCols);
}

cudaError_t make_map(CUtensorMap* m, const void* base, int N, int BH, bool f16) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tensor_map(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool F16>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_map(&mq, a.q, a.rows, a.B * a.H, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mk, a.k, a.Nk, a.B * a.Hkv, F16)) != cudaSuccess) return e;
  if ((e = make_map(&mv, a.v, a.Nk, a.B * a.Hkv, F16)) != cudaSuccess) return e;
  auto kern = fwd_bs_persist_sm103_kernel<F16>;
  // + the two unit entries (each with the pair's live-tile bitmap)
  const int smem = Cfg<F16>::kSmem + 2 * UnitEntry::bytes(a.bit_words);
  // The warp groups re-split the CTA's registers (4 warps down to 88, 8 warps up to 200 per
  // thread); that only completes if the launch holds at least that many registers.
  static LaunchSetup setup;
  int regs = 0;
  if ((e = prepare_launch(setup, kern, smem, &regs)) != cudaSuccess) return e;
  if (regs * kThreads < 128 * 88 + 256 * 200) return cudaErrorInvalidConfiguration;
  int sms = 0;                                     // one CTA per SM, at most one per unit
  if ((e = sm_count(&sms)) != cudaSuccess) return e;
  const int units = min(a.plan_entries * a.B * a.H, max(1, sms));
  fwd_bs_persist_sm103_kernel<F16><<<units, kThreads, smem, s>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bs_persist_sm103(const FwdArgs& a, fa_dtype dt, cudaStream_t s) {
  if (a.plan == nullptr || a.d != 64 || a.drop.enabled || a.cu_seqlens != nullptr || a.n_splits > 1 ||
      a.block_mask == nullptr || a.next_unit == nullptr || a.pair_bits == nullptr || a.o_part == nullptr)
    return cudaErrorInvalidValue;
  return dt == FA_FP16 ? launch<true>(a, s) : launch<false>(a, s);
}

}  // namespace fa
