// Exact key-product features of the tensor-core moments stage (bf16 inputs, d = 64).
//
// The second key moment sum_j p_j k_j k_j^T is a contraction of the weights P with the features
// k_a * k_b (a <= b) of every key. A product of two bf16 values has 16 significant bits, so it is
// split exactly into hi = bf16(k_a k_b) and lo = k_a k_b - hi (both exact bf16: one packed
// multiply and one packed fused multiply-add); both parts are contracted into the same fp32
// accumulator. Rounding the products instead would break the Gram structure of the moments (the
// ridge system could become indefinite); rounding the weights only perturbs them consistently.
//
// Feature order (2208 slots = 1104 pairs of two bf16 features, the layout of a moment row): the
// upper triangle of kt kt^T for the augmented key kt = [k_0..k_63, 1, 0], row by row: for row a,
// the pairs (a, b), (a, b+1) for even b from a (even a) or a + 1 (odd a) up to 64 -- so one operand
// of each packed product is a key word exactly as loaded -- then the 16 pairs of odd diagonal
// entries (4u+1, 4u+1), (4u+3, 4u+3). Slot (a, 64) holds sum p k_a, slots (a, 65) are zero
// padding. Pairs at and beyond kFeaturePairs are zero (padding of a wider pass layout).
#pragma once

#include <cstdint>

namespace lla {
namespace feat {

struct PairSpec { int a, b; bool diag, pad; };
constexpr int kRowPairs = 1088;
constexpr int kFeaturePairs = kRowPairs + 16;   // 1104
constexpr int kFeatureSlots = 2 * kFeaturePairs;  // 2208, the row stride of a moment row

__host__ __device__ constexpr PairSpec pair_spec(int p) {
  if (p >= kFeaturePairs) return PairSpec{0, 0, false, true};
  if (p >= kRowPairs) return PairSpec{p - kRowPairs, 0, true, false};
  int a = 0;
  while (true) {
    const int cnt = (a % 2 == 0) ? 33 - a / 2 : 32 - (a - 1) / 2;
    if (p < cnt) return PairSpec{a, (a % 2 == 0 ? a : a + 1) + 2 * p, false, false};
    p -= cnt;
    ++a;
  }
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t x, uint32_t y, uint32_t z) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(z));
  return r;
}

// Feature pair P (a compile-time index) of one key: its hi and lo words (two bf16 each).
// kw[t] = k[2t] | k[2t+1] << 16 for t < 32; kw[32] = bf16(1) | 0 << 16 (constant feature, pad).
template <int P>
__device__ __forceinline__ void pair_product(const uint32_t (&kw)[33], uint32_t& hi, uint32_t& lo) {
  constexpr PairSpec ps = pair_spec(P);
  if constexpr (ps.pad) {
    hi = 0u;
    lo = 0u;
  } else {
    uint32_t x, y;
    if constexpr (ps.diag) {  // (k[4u+1], k[4u+3]) squared
      x = __byte_perm(kw[2 * ps.a], kw[2 * ps.a + 1], 0x7632);
      y = x;
    } else {                  // (k[a], k[a]) times (k[b], k[b+1])
      x = __byte_perm(kw[ps.a >> 1], 0u, (ps.a & 1) ? 0x3232 : 0x1010);
      y = kw[ps.b >> 1];
    }
    hi = bf16x2_mul(x, y);
    lo = bf16x2_fma(x, y, hi ^ 0x80008000u);
  }
}

// One group of 8 feature slots (pairs P0..P0+3) of one key, stored as one 16-byte row of the
// group's core matrix in the hi and in the lo tile.
template <int P0>
__device__ __forceinline__ void feature_group(const uint32_t (&kw)[33], uint8_t* hi_row,
                                              uint8_t* lo_row) {
  uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
  pair_product<P0 + 0>(kw, h0, l0);
  pair_product<P0 + 1>(kw, h1, l1);
  pair_product<P0 + 2>(kw, h2, l2);
  pair_product<P0 + 3>(kw, h3, l3);
  *reinterpret_cast<uint4*>(hi_row) = make_uint4(h0, h1, h2, h3);
  *reinterpret_cast<uint4*>(lo_row) = make_uint4(l0, l1, l2, l3);
}

}  // namespace feat
}  // namespace lla
