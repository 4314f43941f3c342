// fa_philox.cuh -- the random bytes behind attention dropout, on the device.
//
// Dropout ("Flash Attention, From First Principles", "Honesty time -- the
// confession list", item 4: the extra lines of the paper's algorithm 2) keeps
// probability p_rk of query r and key k with a factor 256/(256 - t), or drops
// it, t = round(256 p).  The decision comes from the counter-based generator
// Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), so that the backward
// pass regenerates exactly the forward's mask instead of storing it: with
// key (seed low word, seed high word) and counter (k/4, r/4, head, 0), byte
// k%4 of output word r%4 belongs to (r, k), and the entry is kept iff that
// byte is >= t.  One call serves a 4 x 4 patch of (query, key) pairs.
//
// Philox4x32-10 itself: ten rounds over four 32-bit words; a round forms the
// full 64-bit products of words 0 and 2 with two fixed odd multipliers,
// moves the low halves to positions 3 and 1 and the high halves, each XORed
// with a neighbouring input word and one round-key word, to positions 0 and
// 2; the round key advances by two fixed Weyl increments between rounds.
#pragma once
#include <cstdint>

#include "fa_internal.h"  // DropSpec

namespace fa {

struct Philox4 {
  uint32_t x[4];
};

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;  // multiplier of word 0
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;  // multiplier of word 2
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;  // key increment, word 0
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;  // key increment, word 1

// One call: the four output words at counter (c0, c1, c2, c3) under the key
// (k0, k1).
__host__ __device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1,
                                                          uint32_t c2, uint32_t c3,
                                                          uint32_t k0, uint32_t k1) {
  uint32_t x0 = c0, x1 = c1, x2 = c2, x3 = c3;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)kPhiloxM0 * x0;
    const uint64_t p1 = (uint64_t)kPhiloxM1 * x2;
    const uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
    const uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
    x1 = (uint32_t)p1;
    x3 = (uint32_t)p0;
    x0 = y0;
    x2 = y2;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return Philox4{{x0, x1, x2, x3}};
}

// 0xFF in every byte of w that is >= t, 0x00 in the others (any t).
__device__ __forceinline__ uint32_t keep_bytes(uint32_t w, uint32_t t4) {
  return __vcmpgeu4(w, t4);
}

// The same decisions in three operations, for t >= 1: bit 7 of byte j of the
// result is set iff byte j of w is >= t, i.e. iff w_j + (256 - t) carries out
// of the byte.  s holds the sums of the low seven bits, so its bit 7 is the
// carry into bit 7; the carry out is the majority of that carry and the two
// top bits.  The other bits of the result are meaningless.
__device__ __forceinline__ uint32_t keep_flags(uint32_t w, const DropSpec& d) {
  const uint32_t s = (w & 0x7F7F7F7Fu) + d.c7;
  return (w & d.c4) | ((w | d.c4) & s);
}

// Byte selection: four bytes taken from the pair (a, b) by the 16-bit selector
// s (nibble i picks result byte i: 0-3 from a, 4-7 from b).
__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(s));
  return r;
}

// 4 x 4 word transpose across the four lanes of a quad: on entry lane q holds
// a[j] for j = 0..3 (row q of the block), on return it holds the former a[q]
// of lanes 0..3 (column q).  Two exchange steps (partners q^1, then q^2),
// two shuffles each.
__device__ __forceinline__ void quad_transpose(uint32_t (&a)[4], int lane) {
  const bool b0 = lane & 1, b1 = (lane >> 1) & 1;
  {
    const uint32_t s0 = b0 ? a[0] : a[1], s1 = b0 ? a[2] : a[3];
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
    if (b0) { a[0] = r0; a[2] = r1; } else { a[1] = r0; a[3] = r1; }
  }
  {
    const uint32_t s0 = b1 ? a[0] : a[2], s1 = b1 ? a[1] : a[3];
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 2);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
    if (b1) { a[0] = r0; a[1] = r1; } else { a[2] = r0; a[3] = r1; }
  }
}

// 4 x 4 byte transpose inside one thread: byte b of w[j] becomes byte j of
// w[b].
__device__ __forceinline__ void byte_transpose(uint32_t (&w)[4]) {
  const uint32_t lo01 = byte_perm(w[0], w[1], 0x5140u);  // w0.b0 w1.b0 w0.b1 w1.b1
  const uint32_t hi01 = byte_perm(w[0], w[1], 0x7362u);  // w0.b2 w1.b2 w0.b3 w1.b3
  const uint32_t lo23 = byte_perm(w[2], w[3], 0x5140u);
  const uint32_t hi23 = byte_perm(w[2], w[3], 0x7362u);
  w[0] = byte_perm(lo01, lo23, 0x5410u);
  w[1] = byte_perm(lo01, lo23, 0x7632u);
  w[2] = byte_perm(hi01, hi23, 0x5410u);
  w[3] = byte_perm(hi01, hi23, 0x7632u);
}

// Keep mask (0xFFFF per kept element) of the bf16 pair at elements 2i, 2i+1
// of a keep_flags word (elements 0-3 = its bytes): selector nibbles 8-15 copy
// the top bit of a byte into all eight bits.
__device__ __forceinline__ uint32_t pair_mask(uint32_t kf, int i) {
  return byte_perm(kf, 0u, (i & 1) ? 0xBBAAu : 0x9988u);
}

// Keep mask (all ones when kept) of element e (0..3) of a keep_flags word.
__device__ __forceinline__ uint32_t elem_mask(uint32_t kf, int e) {
  return byte_perm(kf, 0u, 0x8888u | (0x1111u * (uint32_t)e));
}

// The decision for one (head bh, query r, key k), one Philox call per entry
// (for the CUDA-core kernels, whose threads hold single entries).
__device__ __forceinline__ bool keep_one(const DropSpec& d, int bh, int r, int k) {
  const Philox4 o = philox4x32_10((uint32_t)k >> 2, (uint32_t)r >> 2, (uint32_t)bh,
                                  0u, d.k0, d.k1);
  const uint32_t w01 = (r & 1) ? o.x[1] : o.x[0];
  const uint32_t w23 = (r & 1) ? o.x[3] : o.x[2];
  const uint32_t w = (r & 2) ? w23 : w01;
  return ((w >> (8 * (k & 3))) & 0xFFu) >= (d.t4 & 0xFFu);
}

}  // namespace fa
