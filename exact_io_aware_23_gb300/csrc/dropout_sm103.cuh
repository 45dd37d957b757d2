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

// The key of round r is (seed low + r * 0x9E3779B9, seed high + r * 0xBB67AE85) mod 2^32; the
// host computes the ten pairs once (DropoutArgs::rk0, rk1), so a round's key is an operand of
// the xor instead of two additions per round and call.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const DropoutArgs& d) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)c0 * 0xD2511F53u;
    const uint64_t p1 = (uint64_t)c2 * 0xCD9E8D57u;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    c0 = hi1 ^ c1 ^ d.rk0[r];
    c1 = lo1;
    c2 = hi0 ^ c3 ^ d.rk1[r];
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// ---- drop flags ----------------------------------------------------------------------------------
// Every kernel that needs the mask reads it as flags: bit 7 of a byte set iff that element is
// dropped (its uniform is >= k8).  A flag is applied to a packed bf16/fp16 pair or to an fp32
// value by one byte permute that copies bit 7 over the element's bytes (the prmt "replicate the
// sign" selector) and one and-not.

struct DropTest {
  uint32_t lo7;   // low seven bits of 256 - k8, in every byte
  uint32_t hi;    // bit 7 of 256 - k8, in every byte
  uint32_t all;   // every flag set when k8 == 0 (nothing is kept)
};

__device__ __forceinline__ DropTest drop_test(const DropoutArgs& d) {
  const uint32_t K = (uint32_t)(256 - d.k8) & 0xFFu;
  DropTest t;
  t.lo7 = (K & 0x7Fu) * 0x01010101u;
  t.hi = (K & 0x80u) * 0x01010101u;
  t.all = d.k8 == 0 ? ~0u : 0u;
  return t;
}

__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) { return (a & m) | (b & ~m); }
__device__ __forceinline__ uint32_t rotl(uint32_t x, uint32_t n) { return __funnelshift_l(x, x, n); }
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Flags of a word's four uniforms (bit 7 of byte b <-> byte b; the other bits are undefined).
// byte >= k8  <=>  byte + (256 - k8) carries out of bit 7.  The low seven bits of each byte are
// added on their own (at most 254: nothing crosses into the next byte), which gives the carry
// into bit 7; the carry out is the majority of it and the two operands' bit 7.
__device__ __forceinline__ uint32_t drop_flags(uint32_t w, const DropTest& c) {
  const uint32_t s = (w & 0x7F7F7F7Fu) + c.lo7;
  return (w & c.hi) | (w & s) | (c.hi & s);
}

// One call's sixteen flags in one word: bit 7 - r of byte b = flag of (row r of the call's 4 x 4
// block, i.e. output word r; column b, i.e. byte b).  Bits 3..0 of each byte are undefined.
__device__ __forceinline__ uint32_t pack_flags(const uint4& r, const DropTest& c) {
  uint32_t x = bitsel(drop_flags(r.x, c), drop_flags(r.y, c) >> 1, 0x80808080u);
  x = bitsel(x, drop_flags(r.z, c) >> 2, 0xC0C0C0C0u);
  x = bitsel(x, drop_flags(r.w, c) >> 3, 0xE0E0E0E0u);
  return x | c.all;
}

// Sharing one quad's calls.  The four lanes 4q .. 4q+3 of a warp own four consecutive rows (or
// columns) of the score matrix, the ones a call covers; lane u computes and packs the call of
// group 4m + u along the other axis, so the quad makes four calls for 64 elements a lane instead
// of sixteen.  The packed words are exchanged once (three shuffles) and gathered into one word
// per lane:

// Row-owning lanes (lane t holds row t of the block: the forward, the dQ pass).  Result: bit
// 7 - k of byte b = flag of (this row, column b of group 4m + (t ^ k)).  Group u's four flags are
// brought to bit 7 of the bytes by a left shift of u ^ t.
__device__ __forceinline__ uint32_t gather_row_flags(uint32_t P, uint32_t t) {
  const uint32_t r1 = __shfl_xor_sync(0xffffffffu, P, 1);
  const uint32_t r2 = __shfl_xor_sync(0xffffffffu, P, 2);
  const uint32_t r3 = __shfl_xor_sync(0xffffffffu, P, 3);
  // lane t ^ k's word holds this row at bit 7 - t; rotate it to bit 7 - k
  uint32_t g = bitsel(rotl(P, t), rotl(r1, t - 1u), 0x80808080u);
  g = bitsel(g, rotl(r2, t - 2u), 0xC0C0C0C0u);
  return bitsel(g, rotl(r3, t - 3u), 0xE0E0E0E0u);
}

// Column-owning lanes (lane s holds column s of the block: the dK/dV pass).  Result: byte k =
// the flags of (group 4m + (s ^ k) along the rows, this column), row r at bit 7 - r.
__device__ __forceinline__ uint32_t gather_col_flags(uint32_t P, uint32_t s) {
  const uint32_t r1 = __shfl_xor_sync(0xffffffffu, P, 1);
  const uint32_t r2 = __shfl_xor_sync(0xffffffffu, P, 2);
  const uint32_t r3 = __shfl_xor_sync(0xffffffffu, P, 3);
  const uint32_t sel = s | ((s + 4u) << 4);       // byte s of the first word, byte s of the second
  return prmt(prmt(P, r1, sel), prmt(r2, r3, sel), 0x5410u);
}

// Masks (all ones over a dropped element) from gathered flags.
// Row form: x = gathered word << (u ^ t) for group u; pair h = elements (2h, 2h+1) of the group.
__device__ __forceinline__ uint32_t row_pair_mask(uint32_t x, int h) {
  return prmt(x, 0u, h ? 0xBBAAu : 0x9988u);
}
// Row form, element b of the group (fp32).
__device__ __forceinline__ uint32_t row_elem_mask(uint32_t x, int b) {
  return prmt(x, 0u, (uint32_t)(8 | b) * 0x1111u);
}
// Column form, group u with k = u ^ s: rows (2h, 2h+1) of the group as a pair.
__device__ __forceinline__ uint32_t col_pair_mask(uint32_t g, int h, uint32_t k) {
  return prmt(g << (2 * h), g << (2 * h + 1), ((8u | k) * 0x11u) | ((12u | k) * 0x1100u));
}
// Column form, row r of group u (k = u ^ s), fp32.
__device__ __forceinline__ uint32_t col_elem_mask(uint32_t g, int r, uint32_t k) {
  return prmt(g << r, 0u, (8u | k) * 0x1111u);
}

}  // namespace fa
