// 2:4 top-2-of-4 selection of one group of bf16 activations ("RT-Lynx" page,
// Method: "Top-K based 2:4 activation selection").
#pragma once
#include <cstdint>

namespace lynx {

// Top-2-of-4 decision table.  Index bit b is one pairwise comparison of the four magnitudes,
// c_ij = (|x_i| >= |x_j|) for i < j:  bit 0 c02, 1 c13, 2 c03, 3 c12, 4 c01, 5 c23.  Entry i is kept when at
// most one other entry beats it (j beats i if |x_j| > |x_i|, or |x_j| == |x_i| and j < i); for comparisons
// that come from real magnitudes exactly two entries qualify.  An entry holds the byte_perm selector that
// moves the kept pair (lower index first) out of hi:lo in bits 0-15 and the metadata nibble i0 | i1 << 2 in
// bits 16-19; the index patterns no set of magnitudes produces map to the pair (0, 1).
struct SelectTable {
  uint32_t e[64];
};
__host__ __device__ constexpr SelectTable make_select_table() {
  SelectTable t{};
  for (int idx = 0; idx < 64; ++idx) {
    const int c02 = idx & 1, c13 = (idx >> 1) & 1, c03 = (idx >> 2) & 1, c12 = (idx >> 3) & 1;
    const int c01 = (idx >> 4) & 1, c23 = (idx >> 5) & 1;
    const int loss[4] = {(1 - c01) + (1 - c02) + (1 - c03), c01 + (1 - c12) + (1 - c13), c02 + c12 + (1 - c23),
                         c03 + c13 + c23};
    int kept[2] = {0, 1}, n = 0;
    for (int i = 0; i < 4; ++i)
      if (loss[i] <= 1 && n < 2) kept[n++] = i;
    if (n != 2) {
      kept[0] = 0;
      kept[1] = 1;
    }
    const uint32_t i0 = static_cast<uint32_t>(kept[0]), i1 = static_cast<uint32_t>(kept[1]);
    t.e[idx] = ((i0 * 0x22u + 0x10u) | ((i1 * 0x22u + 0x10u) << 8)) | ((i0 | (i1 << 2)) << 16);
  }
  return t;
}

__device__ __forceinline__ uint32_t set_ge_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;  // per 16-bit half: bf16 1.0 where a >= b, else 0.0
  asm("set.ge.bf16x2.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// acc + x * x for a bf16 x (the low 16 bits of `bits`) in one fused multiply-add with fp32 accumulation:
// the product of two bf16 values is exact in fp32, so this equals fmaf(float(x), float(x), acc).
__device__ __forceinline__ float fma_sq_bf16(uint32_t bits, float acc) {
  float d;
  asm("{ .reg .b16 h; cvt.u16.u32 h, %1; fma.rn.f32.bf16 %0, h, h, %2; }" : "=f"(d) : "r"(bits), "f"(acc));
  return d;
}

// Kept pair of one group of four bf16 values (raw bits lo = x1:x0, hi = x3:x2).  The six comparisons run
// as three packed bf16x2 compares of the sign-cleared values (the bit patterns of |x| order like the
// magnitudes; +0 and -0 compare equal); a packed multiply-add turns their 1.0 / 0.0 results into the table
// index (small integers, exact in bf16: lane 0 holds 128 + c02 + 4 c03 + 16 c01, lane 1 holds
// 2 c13 + 8 c12 + 32 c23, and the bf16 pattern of their sum, 128 + index, carries the index in its low
// mantissa bits).  `table` is the decision table in shared memory.  Returns the metadata nibble, writes the
// kept bf16 pair (lower index in the low half) and adds the squares to the running fp32 sums: x0^2 .. x3^2
// to sum_all, the kept pair's (lower index first) to sum_kept, one rounding per term.  A dropped zero adds
// +0 and leaves a sum unchanged, so when every dropped entry is zero both sums take the same terms in the
// same order and stay equal bit for bit (s = 1 exactly for an input that is already 2:4).
__device__ __forceinline__ uint32_t select_group(uint32_t lo, uint32_t hi, const uint32_t* table, uint32_t& kept,
                                                 float& sum_all, float& sum_kept) {
  const uint32_t m01 = lo & 0x7FFF7FFFu, m23 = hi & 0x7FFF7FFFu;
  const uint32_t m32 = __byte_perm(m23, 0u, 0x1032u);  // |x3| : |x2| -> |x2| : |x3|
  const uint32_t m02 = __byte_perm(m01, m23, 0x5410u), m13 = __byte_perm(m01, m23, 0x7632u);
  const uint32_t e1 = set_ge_bf16x2(m01, m23);  // c02, c13
  const uint32_t e2 = set_ge_bf16x2(m01, m32);  // c03, c12
  const uint32_t e3 = set_ge_bf16x2(m02, m13);  // c01, c23
  uint32_t w = fma_bf16x2(e1, 0x40003F80u, 0x00004300u);  // weights (1, 2), offset (128, 0)
  w = fma_bf16x2(e2, 0x41004080u, w);                      // weights (4, 8)
  w = fma_bf16x2(e3, 0x42004180u, w);                      // weights (16, 32)
  const uint32_t v = fma_bf16x2(__byte_perm(w, 0u, 0x1032u), 0x3F803F80u, w);  // lane 0: the sum of both lanes
  const uint32_t ent = table[v & 0x3Fu];
  kept = __byte_perm(lo, hi, ent);
  float sa = fma_sq_bf16(lo, sum_all);
  sa = fma_sq_bf16(lo >> 16, sa);
  sa = fma_sq_bf16(hi, sa);
  sum_all = fma_sq_bf16(hi >> 16, sa);
  sum_kept = fma_sq_bf16(kept >> 16, fma_sq_bf16(kept, sum_kept));
  return (ent >> 16) & 0xFu;
}

}  // namespace lynx
