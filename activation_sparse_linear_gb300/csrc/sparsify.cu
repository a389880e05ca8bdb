// Online 2:4 activation sparsification (RT-Lynx page, Method: "Top-K based 2:4
// activation selection", performed online and handed to the sparse tensor core
// in its own format; Code examples, first formula: s = ||X||_2 / ||X~||_2).
//
// Each thread streams 16-byte vectors (8 channels = two groups of 4).  Per group the
// two largest magnitudes are kept (ties to the lower index); the lane emits the
// two kept bf16 values of each group
// (an 8-byte coalesced store), one metadata byte that four neighbouring lanes
// assemble into a 32-bit word with shuffles (written as two 16-bit halves to
// the TMEM-ordered lanes, see kernels.h), and fp32 partial sums of x^2 and of
// the kept x^2.  The warp reduces the sums and writes s.
#include <cuda_runtime.h>

#include "kernels.h"

namespace lynx {
namespace {

// Kept pair of one group of four bf16 values (given as raw bits in lo = x1:x0,
// hi = x3:x2).  A tournament finds the two largest magnitudes with four
// comparisons, every one of them resolving ties towards the lower index:
// W1/L1 = winner/loser of (x0, x1), W2/L2 = of (x2, x3).  If |W1| >= |W2| the
// top entry is W1 and the runner-up is the better of L1 and W2 (L2 cannot
// beat W2); otherwise the top entry is W2 and the runner-up is the better of
// W1 and L2.  The kept pair is therefore (0,1), (W1,W2) or (2,3).  Returns
// the metadata nibble i0 | i1 << 2 (i0 < i1), writes the kept bf16 pair
// (i0 in the low half) and accumulates x^2 and kept x^2 in fp32.
__device__ __forceinline__ uint32_t select_group(uint32_t lo, uint32_t hi, uint32_t& kept, float& sx, float& st) {
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
  sx = fmaf(x0, x0, sx);
  sx = fmaf(x1, x1, sx);
  sx = fmaf(x2, x2, sx);
  sx = fmaf(x3, x3, sx);
  const float k0 = __uint_as_float(kept << 16), k1 = __uint_as_float(kept & 0xFFFF0000u);
  st = fmaf(k0, k0, st);
  st = fmaf(k1, k1, st);
  return nib;
}

// A persistent CTA of kThreads threads walks token rows blockIdx.x,
// blockIdx.x + gridDim.x, ...: thread t handles the 16-byte vectors t,
// t + kThreads, ... of a row, so every load instruction of a warp is one
// coalesced 512-byte access.  kLoads vectors per thread cover a row in one
// batch (4: K <= 4096, 12: K <= 12288; longer rows take several batches).
// With kPrefetch the loads of the CTA's next row are issued before the
// current row is processed, so a row's selection overlaps the next row's
// memory latency.
constexpr int kThreads = 128;

template <int kLoads, bool kPrefetch>
__global__ void __launch_bounds__(kThreads, kLoads <= 4 ? 6 : 3) sparsify_kernel(const uint4* __restrict__ X, int M, int K, int K_pad,
                                                            int M_pad, uint2* __restrict__ vals,
                                                            uint8_t* __restrict__ meta, float* __restrict__ s) {
  __shared__ float red[2][2][kThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int V = K_pad / 8;  // vectors per (padded) row
  const int Vx = K / 8;     // vectors that exist in X
  const int64_t blocks_k = K_pad / kMetaBlockCols;

  auto load_row = [&](int row, int base, uint4 (&v)[kLoads]) {
    const bool live = row < M;
    const uint4* xr = X + static_cast<int64_t>(row) * Vx;
#pragma unroll
    for (int l = 0; l < kLoads; ++l) {
      const int i = base + l * kThreads + t;
      v[l] = (live && i < Vx) ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
    }
  };

  uint4 cur[kLoads], nxt[kLoads];
  int row = blockIdx.x;
  if (kPrefetch && row < M_pad) load_row(row, 0, cur);
  for (int parity = 0; row < M_pad; row += gridDim.x, parity ^= 1) {
    const bool live = row < M;
    uint2* vr = vals + static_cast<int64_t>(row) * Vx;  // 4 kept values (8 B) per 8 channels
    uint8_t* m_lo = meta + meta_half_offset(row, 0, 0, blocks_k);
    uint8_t* m_hi = meta + meta_half_offset(row, 0, 1, blocks_k);
    float sx = 0.f, st = 0.f;
    for (int base = 0; base < V; base += kThreads * kLoads) {
      if (kPrefetch) {
        if (row + static_cast<int>(gridDim.x) < M_pad) load_row(row + gridDim.x, 0, nxt);
      } else {
        load_row(row, base, cur);
      }
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
        const int i = base + l * kThreads + t;
        if (base + l * kThreads >= V) break;  // uniform across the CTA: every lane reaches the shuffles
        uint32_t kept0, kept1;
        const uint32_t n0 = select_group(cur[l].x, cur[l].y, kept0, sx, st);
        const uint32_t n1 = select_group(cur[l].z, cur[l].w, kept1, sx, st);
        const uint32_t byte = n0 | (n1 << 4);
        uint32_t word = byte;
        word |= __shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8;
        word |= __shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16;
        word |= __shfl_down_sync(0xFFFFFFFFu, byte, 3) << 24;
        if (live && i < Vx) vr[i] = make_uint2(kept0, kept1);
        if ((lane & 3) == 0 && i < V) {
          const int c = i / 4;  // 4 vectors per 32-channel chunk
          const int64_t off = static_cast<int64_t>(c / 4) * kMetaChunkBytes + (c % 4) * 4;
          *reinterpret_cast<uint16_t*>(m_lo + off) = static_cast<uint16_t>(word & 0xFFFFu);
          *reinterpret_cast<uint16_t*>(m_hi + off) = static_cast<uint16_t>(word >> 16);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sx += __shfl_xor_sync(0xFFFFFFFFu, sx, o);
      st += __shfl_xor_sync(0xFFFFFFFFu, st, o);
    }
    if (lane == 0) {
      red[parity][0][warp] = sx;
      red[parity][1][warp] = st;
    }
    __syncthreads();  // red[parity] complete; red[parity ^ 1] was read before this barrier
    if (t == 0 && live) {
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) {
        a += red[parity][0][w];
        b += red[parity][1][w];
      }
      s[row] = b > 0.f ? sqrtf(a / b) : 1.f;
    }
    if (kPrefetch) {
#pragma unroll
      for (int l = 0; l < kLoads; ++l) cur[l] = nxt[l];
    }
  }
}

}  // namespace

cudaError_t launch_sparsify(const void* X, int M, int K, void* vals, void* meta, float* s, cudaStream_t stream) {
  const int M_pad = static_cast<int>(round_up(M, kMetaRowPad));
  const int K_pad = static_cast<int>(round_up(K, kMetaBlockCols));
  const bool short_rows = K_pad / 8 <= 4 * kThreads;
  auto* k = short_rows ? sparsify_kernel<4, true> : sparsify_kernel<12, false>;
  static int per_sm[2][64] = {};  // resident CTAs per SM, per kernel variant and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int& occ = per_sm[short_rows ? 0 : 1][dev];
  if (!occ) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, 0) != cudaSuccess || n < 1) n = 1;
    occ = n;
  }
  int grid = sm_count() * occ;
  if (grid > M_pad) grid = M_pad;
  k<<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(X), M, K, K_pad, M_pad, static_cast<uint2*>(vals),
                                   static_cast<uint8_t*>(meta), s);
  return cudaGetLastError();
}

}  // namespace lynx
