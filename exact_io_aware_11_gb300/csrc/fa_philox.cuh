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

// 0xff in each byte of `w` that is >= the byte threshold (replicated in t4), else 0x00.
__device__ __forceinline__ uint32_t keep_bytes(uint32_t w, uint32_t t4) { return __vcmpgeu4(w, t4); }

// For a pair of elements whose keep bytes are bytes (2 s, 2 s + 1) of `m`
// (s = 0 or 1): a mask that clears the dropped bf16 halves of a packed pair.
__device__ __forceinline__ uint32_t pair_mask(uint32_t m, int s) {
  return __byte_perm(m, 0u, s ? 0x3322u : 0x1100u);
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

// Four keep bytes (0xff / 0x00) -> four bits, byte b -> bit b.
__device__ __forceinline__ uint32_t keep_nibble(uint32_t m) {
  return ((m & 0x01010101u) * 0x01020408u) >> 24;
}

}  // namespace fa
