// Dropout mask of the attention probabilities, regenerated wherever it is needed (forward, both
// backward passes) from a counter-based generator instead of being stored: the "dropout RNG" and
// its replay that "FlashAttention：让精确注意力服从内存层次" lists among the production semantics.
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011), written from that paper: ten rounds of two 32x32->64-bit products of counter
// words 0 and 2 by fixed odd multipliers, the high halves xored with the other two counter words
// and the key, the key advanced by two Weyl increments between rounds.
//
// Layout: one call covers a 4 x 4 block of one (b, h) slice's score matrix; counter =
// (j / 4, i / 4, b*H + h, offset), key = (seed low word, seed high word).  Byte (j mod 4) of
// output word (i mod 4) is the 8-bit uniform of element (i, j); the element is kept iff that
// byte is below k8 (keep probability k8 / 256), and kept probabilities are scaled by 256 / k8.
#pragma once

#include <stdint.h>

#include "fa_internal.cuh"

namespace fa {

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)c0 * 0xD2511F53u;
    const uint64_t p1 = (uint64_t)c2 * 0xCD9E8D57u;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Keep bits of the four bytes of one 32-bit word (bit k <-> byte k).
__device__ __forceinline__ uint32_t keep4(uint32_t w, uint32_t k8) {
  return ((w & 0xFFu) < k8 ? 1u : 0u) | (((w >> 8) & 0xFFu) < k8 ? 2u : 0u) |
         (((w >> 16) & 0xFFu) < k8 ? 4u : 0u) | ((w >> 24) < k8 ? 8u : 0u);
}

// The four lanes of a quad (lanes 4m .. 4m+3) own four consecutive rows (or columns) of the score
// matrix, so one call serves all four.  Each lane computes a quarter of the calls and the quad
// exchanges the words: a 4 x 4 transpose across the quad, lane t holding row t of the input and
// receiving column t (element t of every lane's row; element s of the result comes from lane s).
__device__ __forceinline__ uint4 quad_transpose(uint4 w, uint32_t t) {
  auto pick = [&](uint32_t k) { return k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w; };
  const uint32_t own = pick(t);
  const uint32_t r1 = __shfl_xor_sync(0xffffffffu, pick(t ^ 1u), 1);
  const uint32_t r2 = __shfl_xor_sync(0xffffffffu, pick(t ^ 2u), 2);
  const uint32_t r3 = __shfl_xor_sync(0xffffffffu, pick(t ^ 3u), 3);
  auto from = [&](uint32_t s) {          // element t of lane s's row
    const uint32_t k = s ^ t;
    return k == 0 ? own : k == 1 ? r1 : k == 2 ? r2 : r3;
  };
  return make_uint4(from(0), from(1), from(2), from(3));
}

// Query row i over 64 consecutive keys j0 .. j0+63 (j0 a multiple of 4): bit c of the result
// is the keep bit of key j0 + c.  The quad's lanes must own rows i0 .. i0+3 (i = i0 + lane % 4).
__device__ __forceinline__ uint64_t keep_row64(const DropoutArgs& d, uint32_t bh, int i, int j0) {
  const uint32_t t = (uint32_t)i & 3u;
  uint64_t bits = 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    // this lane's call: key group 4m + t; after the exchange, element s = word t (this row) of
    // the call for key group 4m + s
    const uint4 r = philox4x32_10((uint32_t)(j0 >> 2) + 4u * m + t, (uint32_t)i >> 2, bh, d.offset,
                                  d.seed_lo, d.seed_hi);
    const uint4 c = quad_transpose(r, t);
    const uint32_t k8 = (uint32_t)d.k8;
    bits |= (uint64_t)(keep4(c.x, k8) | (keep4(c.y, k8) << 4) | (keep4(c.z, k8) << 8) |
                       (keep4(c.w, k8) << 12)) << (16 * m);
  }
  return bits;
}

// The same bits computed by each lane on its own (16 calls per 64 elements, no exchange): in the
// backward passes, whose warps have less slack to hide the exchange's latency, this measured
// faster than the shared form.
__device__ __forceinline__ uint64_t keep_row64_own(const DropoutArgs& d, uint32_t bh, int i, int j0) {
  uint64_t bits = 0;
  const uint32_t sel = (uint32_t)i & 3u;
#pragma unroll 4
  for (int g = 0; g < 16; ++g) {
    const uint4 r = philox4x32_10((uint32_t)(j0 >> 2) + g, (uint32_t)i >> 2, bh, d.offset, d.seed_lo,
                                  d.seed_hi);
    const uint32_t w = sel == 0 ? r.x : sel == 1 ? r.y : sel == 2 ? r.z : r.w;
    bits |= (uint64_t)keep4(w, (uint32_t)d.k8) << (4 * g);
  }
  return bits;
}

// Key j over 64 consecutive queries i0 .. i0+63 (i0 a multiple of 4): bit c of the result is
// the keep bit of query i0 + c (each lane on its own).
__device__ __forceinline__ uint64_t keep_col64_own(const DropoutArgs& d, uint32_t bh, int i0, int j) {
  uint64_t bits = 0;
  const uint32_t sh = 8u * ((uint32_t)j & 3u);
  const uint32_t k8 = (uint32_t)d.k8;
#pragma unroll 4
  for (int g = 0; g < 16; ++g) {
    const uint4 r = philox4x32_10((uint32_t)j >> 2, (uint32_t)(i0 >> 2) + g, bh, d.offset, d.seed_lo,
                                  d.seed_hi);
    const uint32_t k4 = (((r.x >> sh) & 0xFFu) < k8 ? 1u : 0u) | (((r.y >> sh) & 0xFFu) < k8 ? 2u : 0u) |
                        (((r.z >> sh) & 0xFFu) < k8 ? 4u : 0u) | (((r.w >> sh) & 0xFFu) < k8 ? 8u : 0u);
    bits |= (uint64_t)k4 << (4 * g);
  }
  return bits;
}

// 32-element forms of the two above (each lane on its own, 8 calls): a query over keys
// j0 .. j0+31, a key over queries i0 .. i0+31.
__device__ __forceinline__ uint64_t keep_row32_own(const DropoutArgs& d, uint32_t bh, int i, int j0) {
  uint64_t bits = 0;
  const uint32_t sel = (uint32_t)i & 3u;
#pragma unroll 4
  for (int g = 0; g < 8; ++g) {
    const uint4 r = philox4x32_10((uint32_t)(j0 >> 2) + g, (uint32_t)i >> 2, bh, d.offset, d.seed_lo,
                                  d.seed_hi);
    const uint32_t w = sel == 0 ? r.x : sel == 1 ? r.y : sel == 2 ? r.z : r.w;
    bits |= (uint64_t)keep4(w, (uint32_t)d.k8) << (4 * g);
  }
  return bits;
}
__device__ __forceinline__ uint64_t keep_col32_own(const DropoutArgs& d, uint32_t bh, int i0, int j) {
  uint64_t bits = 0;
  const uint32_t sh = 8u * ((uint32_t)j & 3u);
  const uint32_t k8 = (uint32_t)d.k8;
#pragma unroll 4
  for (int g = 0; g < 8; ++g) {
    const uint4 r = philox4x32_10((uint32_t)j >> 2, (uint32_t)(i0 >> 2) + g, bh, d.offset, d.seed_lo,
                                  d.seed_hi);
    const uint32_t k4 = (((r.x >> sh) & 0xFFu) < k8 ? 1u : 0u) | (((r.y >> sh) & 0xFFu) < k8 ? 2u : 0u) |
                        (((r.z >> sh) & 0xFFu) < k8 ? 4u : 0u) | (((r.w >> sh) & 0xFFu) < k8 ? 8u : 0u);
    bits |= (uint64_t)k4 << (4 * g);
  }
  return bits;
}

}  // namespace fa
