// Counter-based random draws for fused dropout.
//
// Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): a keyed bijection of
// a 128-bit counter, ten rounds of two 32 x 32 -> 64-bit products whose halves
// are mixed with the other two counter words and the round key. Because a draw
// is a pure function of (counter, key), the backward pass regenerates exactly
// the keep decisions of the forward pass from the element's indices, and the
// dropout mask never exists in memory.
//
// Element (b, h, i, j) of a problem with H heads uses byte j mod 16 (byte
// j mod 4 of word (j mod 16) / 4, little-endian) of the block at counter
// (j / 16, i, b*H + h, offset); it is kept iff that byte >= t, t = round(256 p).
#pragma once

#include <cstdint>

namespace fa {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;  // round multipliers
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;  // key increments

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c0;  // one wide multiply each
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c2;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k1;
    c1 = static_cast<uint32_t>(p1);
    c3 = static_cast<uint32_t>(p0);
    c0 = n0;
    c2 = n2;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Sign bit of each byte of the result = [byte of w >= byte of t4] (t4: the
// threshold replicated into the four bytes); the other bits are garbage.
// c4 = 0x80808080 - (t4 & 0x7f7f7f7f). Bytes are compared without carries
// between them: (w & 0x7f) + 0x80 - (t & 0x7f) has its top bit set iff the
// low seven bits of w are >= those of t, which decides where the top bits of
// w and t agree; where they differ, the top bit of w decides.
__device__ __forceinline__ uint32_t keep_msb(uint32_t w, uint32_t t4, uint32_t c4) {
  const uint32_t d = (w & 0x7f7f7f7fu) + c4;
  return (w & ~t4) | (~(w ^ t4) & d);
}

// The keep decisions of 32 consecutive keys (two Philox blocks: key e takes
// byte e mod 4 of word e / 4 of {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}) in
// one word: key e = 4 w + b at bit 8 b + 7 - w, so that shifting the word
// left by w brings the decisions of keys 4 w .. 4 w + 3 to the sign bits of
// bytes 0..3.
__device__ __forceinline__ uint32_t keep_bits32(const uint4& a, const uint4& b, uint32_t t4, uint32_t c4) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) r |= (keep_msb(w[i], t4, c4) & 0x80808080u) >> i;
  return r;
}

// Mask for the packed bf16 pair of keys (2 c, 2 c + 1), c = 0..15, of a word
// made by keep_bits32: 0xffff over each kept half, 0 over a dropped one
// (prmt with the sign-replicating selector: 8 + i copies the sign of byte i).
__device__ __forceinline__ uint32_t pair_mask_bits(uint32_t bits, int c) {
  const uint32_t s = bits << (c >> 1);
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(s), "r"((c & 1) ? 0xBBAAu : 0x9988u));
  return r;
}

// Decision for key e (0..31) of a word made by keep_bits32.
__device__ __forceinline__ bool keep_bit(uint32_t bits, int e) {
  return (bits >> (8 * (e & 3) + 7 - (e >> 2))) & 1u;
}

// 16 x 16 byte transpose across the 16 lanes of a half-warp. Lane p holds row
// p in w (byte k of the row = byte k mod 4 of w[k / 4]); afterwards it holds
// column p. Four butterfly stages (lane distance 8, 4, 2, 1): at distance s a
// lane whose bit s is clear trades its row bytes whose index has bit s set
// for the partner's bytes whose index has bit s clear. Bytes are moved in
// 32-bit words, two shuffles per stage.
__device__ __forceinline__ void transpose16_bytes(uint32_t (&w)[4], int lane) {
  {  // distance 8: words {2,3} <-> partner's words {0,1}
    const bool up = lane & 8;
    const uint32_t s0 = up ? w[0] : w[2], s1 = up ? w[1] : w[3];
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 8);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 8);
    if (up) { w[0] = r0; w[1] = r1; } else { w[2] = r0; w[3] = r1; }
  }
  {  // distance 4: words {1,3} <-> partner's words {0,2}
    const bool up = lane & 4;
    const uint32_t s0 = up ? w[0] : w[1], s1 = up ? w[2] : w[3];
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 4);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 4);
    if (up) { w[0] = r0; w[2] = r1; } else { w[1] = r0; w[3] = r1; }
  }
  {  // distance 2: upper 16-bit halves <-> partner's lower halves
    const bool up = lane & 2;
    const uint32_t pick = up ? 0x5410u : 0x7632u;      // halves sent from (w[a], w[a+1])
    const uint32_t put0 = up ? 0x3254u : 0x5410u;      // merge into w[a]
    const uint32_t put1 = up ? 0x3276u : 0x7610u;      // merge into w[a+1]
#pragma unroll
    for (int a = 0; a < 4; a += 2) {
      const uint32_t r = __shfl_xor_sync(0xffffffffu, __byte_perm(w[a], w[a + 1], pick), 2);
      w[a] = __byte_perm(w[a], r, put0);
      w[a + 1] = __byte_perm(w[a + 1], r, put1);
    }
  }
  {  // distance 1: odd bytes <-> partner's even bytes
    const bool up = lane & 1;
    const uint32_t pick = up ? 0x6420u : 0x7531u;
    const uint32_t put0 = up ? 0x3514u : 0x5240u;
    const uint32_t put1 = up ? 0x3716u : 0x7260u;
#pragma unroll
    for (int a = 0; a < 4; a += 2) {
      const uint32_t r = __shfl_xor_sync(0xffffffffu, __byte_perm(w[a], w[a + 1], pick), 1);
      w[a] = __byte_perm(w[a], r, put0);
      w[a + 1] = __byte_perm(w[a + 1], r, put1);
    }
  }
}

}  // namespace fa
