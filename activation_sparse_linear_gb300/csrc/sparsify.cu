// Online 2:4 activation sparsification (RT-Lynx page, Method: "Top-K based 2:4
// activation selection", performed online and handed to the sparse tensor core
// in its own format; Code examples, first formula: s = ||X||_2 / ||X~||_2).
//
// One warp per token row.  Each lane streams 16-byte vectors (8 channels = two
// groups of 4) with the warp covering 256 contiguous channels per step, so
// every load instruction is a fully coalesced 512-byte access.  Per group the
// two largest magnitudes are kept (ties to the lower index) by ranking the four
// 15-bit magnitude keys; the lane emits the two kept bf16 values of each group
// (an 8-byte coalesced store), one metadata byte that four neighbouring lanes
// assemble into a 32-bit word with shuffles (written as two 16-bit halves to
// the TMEM-ordered lanes, see kernels.h), and fp32 partial sums of x^2 and of
// the kept x^2.  The warp reduces the sums and writes s.
#include <cuda_runtime.h>

#include "kernels.h"

namespace lynx {
namespace {

constexpr int kUnroll = 4;

// Kept pair of one group of four bf16 values (given as raw bits): returns the
// 4-bit metadata nibble (i0 | i1 << 2, i0 < i1) and writes the kept values.
__device__ __forceinline__ uint32_t select_group(uint32_t lo, uint32_t hi, uint32_t& kept, float& sx, float& st) {
  const uint32_t b0 = lo & 0xFFFFu, b1 = lo >> 16, b2 = hi & 0xFFFFu, b3 = hi >> 16;
  const uint32_t k0 = b0 & 0x7FFFu, k1 = b1 & 0x7FFFu, k2 = b2 & 0x7FFFu, k3 = b3 & 0x7FFFu;
  // i beats j (i < j) when k_i >= k_j; rank = number of entries that beat this one.
  const uint32_t w01 = k0 >= k1, w02 = k0 >= k2, w03 = k0 >= k3;
  const uint32_t w12 = k1 >= k2, w13 = k1 >= k3, w23 = k2 >= k3;
  const uint32_t r0 = (w01 ^ 1) + (w02 ^ 1) + (w03 ^ 1);
  const uint32_t r1 = w01 + (w12 ^ 1) + (w13 ^ 1);
  const uint32_t r2 = w02 + w12 + (w23 ^ 1);
  const uint32_t r3 = w03 + w13 + w23;
  const uint32_t keep = (r0 < 2) | ((r1 < 2) << 1) | ((r2 < 2) << 2) | ((r3 < 2) << 3);
  // keep mask -> (i0, i1): 0011->(0,1) 0101->(0,2) 1001->(0,3) 0110->(1,2) 1010->(1,3) 1100->(2,3)
  const uint32_t i0 = (keep & 1) ? 0u : ((keep & 2) ? 1u : 2u);
  const uint32_t i1 = (keep & 8) ? 3u : ((keep & 4) ? 2u : 1u);
  const uint32_t c0 = (i0 == 0) ? b0 : ((i0 == 1) ? b1 : b2);
  const uint32_t c1 = (i1 == 3) ? b3 : ((i1 == 2) ? b2 : b1);
  kept = c0 | (c1 << 16);
  const float x0 = __uint_as_float(b0 << 16), x1 = __uint_as_float(b1 << 16);
  const float x2 = __uint_as_float(b2 << 16), x3 = __uint_as_float(b3 << 16);
  sx += x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3;
  const float v0 = __uint_as_float(c0 << 16), v1 = __uint_as_float(c1 << 16);
  st += v0 * v0 + v1 * v1;
  return i0 | (i1 << 2);
}

__global__ void __launch_bounds__(256) sparsify_kernel(const uint4* __restrict__ X, int M, int K, int M_pad,
                                                       int K_pad, uint2* __restrict__ vals,
                                                       uint8_t* __restrict__ meta, float* __restrict__ s) {
  const int lane = threadIdx.x & 31;
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= M_pad) return;  // warp-uniform
  const bool live = row < M;
  const int kv = K / 8;  // 16-byte vectors per row
  const uint4* xr = X + static_cast<int64_t>(row) * kv;
  uint2* vr = vals + static_cast<int64_t>(row) * (K / 8);  // 4 kept values (8 B) per 8 channels
  const int64_t chunks_k = K_pad / kMetaChunkCols;
  // this row's two 16-bit destinations in chunk 0; chunk c adds c * kMetaChunkBytes
  uint16_t* m_lo = reinterpret_cast<uint16_t*>(meta + meta_half_offset(row, 0, 0, chunks_k));
  uint16_t* m_hi = reinterpret_cast<uint16_t*>(meta + meta_half_offset(row, 0, 1, chunks_k));
  float sx = 0.f, st = 0.f;
  for (int base = 0; base < K_pad; base += 256 * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int k = base + u * 256 + lane * 8;
      v[u] = (live && k < K) ? __ldg(xr + k / 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int k = base + u * 256 + lane * 8;
      uint32_t kept0, kept1;
      const uint32_t n0 = select_group(v[u].x, v[u].y, kept0, sx, st);
      const uint32_t n1 = select_group(v[u].z, v[u].w, kept1, sx, st);
      const uint32_t byte = n0 | (n1 << 4);
      uint32_t word = byte;
      word |= __shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8;
      word |= __shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16;
      word |= __shfl_down_sync(0xFFFFFFFFu, byte, 3) << 24;
      if (live && k < K) vr[k / 8] = make_uint2(kept0, kept1);
      if ((lane & 3) == 0 && k < K_pad) {
        const int64_t off = static_cast<int64_t>(k / kMetaChunkCols) * (kMetaChunkBytes / 2);
        m_lo[off] = static_cast<uint16_t>(word & 0xFFFFu);
        m_hi[off] = static_cast<uint16_t>(word >> 16);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sx += __shfl_xor_sync(0xFFFFFFFFu, sx, o);
    st += __shfl_xor_sync(0xFFFFFFFFu, st, o);
  }
  if (lane == 0 && live) s[row] = st > 0.f ? sqrtf(sx / st) : 1.f;
}

}  // namespace

cudaError_t launch_sparsify(const void* X, int M, int K, void* vals, void* meta, float* s, cudaStream_t stream) {
  const int M_pad = static_cast<int>(round_up(M, kMetaRows));
  const int K_pad = static_cast<int>(round_up(K, kMetaKPad));
  const int warps_per_block = 8;
  const int blocks = (M_pad + warps_per_block - 1) / warps_per_block;
  sparsify_kernel<<<blocks, warps_per_block * 32, 0, stream>>>(static_cast<const uint4*>(X), M, K, M_pad, K_pad,
                                                               static_cast<uint2*>(vals),
                                                               static_cast<uint8_t*>(meta), s);
  return cudaGetLastError();
}

}  // namespace lynx
