// 2:4 top-2-of-4 selection of one group of bf16 activations ("RT-Lynx" page,
// Method: "Top-K based 2:4 activation selection").
#pragma once
#include <cstdint>

namespace lynx {

// Kept pair of one group of four bf16 values (given as raw bits in lo = x1:x0,
// hi = x3:x2).  A tournament finds the two largest magnitudes with four
// comparisons, every one of them resolving ties towards the lower index:
// W1/L1 = winner/loser of (x0, x1), W2/L2 = of (x2, x3).  If |W1| >= |W2| the
// top entry is W1 and the runner-up is the better of L1 and W2 (L2 cannot
// beat W2); otherwise the top entry is W2 and the runner-up is the better of
// W1 and L2.  The kept pair is therefore (0,1), (W1,W2) or (2,3).  Returns
// the metadata nibble i0 | i1 << 2 (i0 < i1), writes the kept bf16 pair
// (i0 in the low half) and the group's fp32 sums of x^2 and of kept x^2.
// The squares of bf16 values are exact in fp32, so when the dropped entries
// are zero both sums add the same two terms in the same order and are equal
// bit for bit (s = 1 exactly for an input that is already 2:4).
__device__ __forceinline__ uint32_t select_group(uint32_t lo, uint32_t hi, uint32_t& kept, float& q_all,
                                                 float& q_kept) {
  const float x0 = __uint_as_float(lo << 16), x1 = __uint_as_float(lo & 0xFFFF0000u);
  const float x2 = __uint_as_float(hi << 16), x3 = __uint_as_float(hi & 0xFFFF0000u);
  const float a0 = fabsf(x0), a1 = fabsf(x1), a2 = fabsf(x2), a3 = fabsf(x3);
  const bool p = a0 >= a1;  // W1 = x0 (ties go to x0)
  const bool q = a2 >= a3;  // W2 = x2
  const float mx01 = fmaxf(a0, a1), mn01 = fminf(a0, a1);
  const float mx23 = fmaxf(a2, a3), mn23 = fminf(a2, a3);
  const bool r = mx01 >= mx23;                          // top entry is W1
  const bool c = r ? (mn01 >= mx23) : (mx01 >= mn23);  // runner-up is L1 (r) / W1 (!r)
  const uint32_t w = (p ? 0u : 1u) | (q ? 8u : 12u);   // nibble of (W1, W2)
  const uint32_t nib = r ? (c ? 0x4u : w) : (c ? w : 0xEu);
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  // bytes 2i, 2i+1 of hi:lo hold entry i
  kept = __byte_perm(lo, hi, (i0 * 0x22u + 0x10u) | ((i1 * 0x22u + 0x10u) << 8));
  q_all = fmaf(x1, x1, x0 * x0) + fmaf(x3, x3, x2 * x2);
  const float k0 = __uint_as_float(kept << 16), k1 = __uint_as_float(kept & 0xFFFF0000u);
  q_kept = fmaf(k1, k1, k0 * k0);
  return nib;
}

}  // namespace lynx
