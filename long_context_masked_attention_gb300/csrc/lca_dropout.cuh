// lca_dropout.cuh — attention dropout inside the fused kernels.
//
// The FlashAttention review page ("长上下文能力：FlashAttention vs.
// RingAttention", FlashAttention-1 核心优化, 算子融合) lists dropout among
// the operations fused with the matmuls, the mask and the softmax.  Here it
// is inverted dropout on the attention probabilities: with keep probability
// kp, O = (P * Z / kp) V where Z_ij in {0, 1}; LSE stays that of P.
//
// Random bits come from Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011), a counter-based
// generator, so every kernel regenerates the same Z_ij from its indices alone:
// one call per (query head h, global query row i, 16 consecutive keys of the
// row's segment), counter (j / 16, i, h, 0), key (seed low word, seed high
// word).  Key j takes byte j % 4 of output word (j % 16) / 4 and is kept when
// that byte is >= t, t = floor(256 p + 1/2) for drop probability p, so
// kp = (256 - t) / 256.
#pragma once
#include <cstdint>

namespace lca {

// The key of each of the ten rounds: the seed words advanced by the Weyl
// constants, k[2r] = seed_lo + r 0x9E3779B9, k[2r+1] = seed_hi + r 0xBB67AE85
// (mod 2^32).  The host fills them into the kernel arguments, so every round
// reads its key as a constant operand.
struct PhiloxKeys {
  uint32_t k[20];
};

inline PhiloxKeys philox_round_keys(uint64_t seed) {
  PhiloxKeys r;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    r.k[2 * i] = k0;
    r.k[2 * i + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return r;
}

struct DropCtx {
  uint32_t tlo;  // (t & 0x7F) in every byte
  uint32_t nt;   // ~t in every byte
};

__host__ __device__ __forceinline__ DropCtx make_drop_ctx(int t) {
  DropCtx d;
  d.tlo = static_cast<uint32_t>(t & 0x7F) * 0x01010101u;
  d.nt = ~(static_cast<uint32_t>(t & 0xFF) * 0x01010101u);
  return d;
}

// Ten rounds; each multiplies counter words 0 and 2 by the round constants
// (one 32 x 32 -> 64-bit product each) and crosses the product halves over,
// mixing in the round key.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const PhiloxKeys& key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t w0 = static_cast<uint64_t>(c0) * 0xD2511F53u;
    const uint64_t w1 = static_cast<uint64_t>(c2) * 0xCD9E8D57u;
    c0 = static_cast<uint32_t>(w1 >> 32) ^ c1 ^ key.k[2 * r];
    c1 = static_cast<uint32_t>(w1);
    c2 = static_cast<uint32_t>(w0 >> 32) ^ c3 ^ key.k[2 * r + 1];
    c3 = static_cast<uint32_t>(w0);
  }
  return make_uint4(c0, c1, c2, c3);
}

// Bit 7 of byte b of the result = (byte b of w >= t), for the four bytes at
// once: the low seven bits compare through one subtraction with a
// borrow-free guard bit, and the top bits decide where they differ (majority
// of w, ~t and the difference).  Other bits are garbage.
__device__ __forceinline__ uint32_t keep_signs(uint32_t w, const DropCtx& d) {
  const uint32_t diff = (w | 0x80808080u) - d.tlo;
  return (w & d.nt) | (w & diff) | (d.nt & diff);
}

// Bit b (0..3) = byte b of w >= t: the four sign bits gathered from bits 7,
// 15, 23, 31 by a multiply.
__device__ __forceinline__ uint32_t keep4(uint32_t w, const DropCtx& d) {
  return ((keep_signs(w, d) & 0x80808080u) * 0x00204081u) >> 28;
}

// 0xFFFF in the low half iff byte 2h keeps, in the high half iff byte 2h+1
// keeps (h = 0 or 1), from keep_signs: a byte permute that replicates the
// selected bytes' sign bits.
template <int h>
__device__ __forceinline__ uint32_t keep_halves(uint32_t signs) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(signs), "n"(h ? 0xBBAA : 0x9988));
  return r;
}

// Keep bits of 32 consecutive keys 16 g .. 16 g + 31 of query row `row` (bit e
// = key 16 g + e), from the two Philox calls of key groups g and g + 1.
__device__ __forceinline__ uint32_t keep32(const DropCtx& d, const PhiloxKeys& key, uint32_t row, uint32_t head,
                                           uint32_t g) {
  const uint4 a = philox4x32_10(g, row, head, 0u, key);
  const uint4 b = philox4x32_10(g + 1u, row, head, 0u, key);
  return keep4(a.x, d) | (keep4(a.y, d) << 4) | (keep4(a.z, d) << 8) | (keep4(a.w, d) << 12) |
         (keep4(b.x, d) << 16) | (keep4(b.y, d) << 20) | (keep4(b.z, d) << 24) | (keep4(b.w, d) << 28);
}

// Transpose of the 32 x 32 bit matrix whose row r is lane r's x: returns, in
// lane c, the word whose bit r is bit c of lane r's x.  Five stages swap the
// off-diagonal s x s blocks for s = 16, 8, 4, 2, 1.
__device__ __forceinline__ uint32_t warp_transpose_bits(uint32_t x, int lane) {
  const uint32_t lowmask[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const int s = 16 >> i;
    const uint32_t m = lowmask[i];
    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, s);
    x = (lane & s) ? ((x & ~m) | ((y >> s) & m)) : ((x & m) | ((y & m) << s));
  }
  return x;
}

}  // namespace lca
