// Tensor-core rate microbenchmark: back-to-back tcgen05.mma (dense) or
// tcgen05.mma.sp (2:4 sparse A) of shape M=128, N=256 from operands resident in
// shared memory, one CTA per SM, no global-memory traffic.  It measures the
// peak the sparse GEMM is held against (the 2:4 rate relative to dense).
#include <cuda_runtime.h>

#include "../../include/lynx.h"
#include "kernels.h"

namespace lynx {
namespace {

constexpr int kN = 256;

__device__ unsigned long long g_rate_cycles;
__device__ int g_rate_error;

// mode 0: dense; 1: sparse, metadata resident in TMEM; 2: sparse, each MMA
// preceded by a tcgen05.cp.128x128b of its 2 KiB metadata chunk into one of
// eight 32-column slots; 3: sparse with a tcgen05.commit after every two
// MMAs (one pipeline stage of 64 channels); 4: sparse with two commits after
// every four MMAs; 5: sparse with A in the 64-byte swizzle of 64-byte rows.
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int mode, int iters, DevCtl ctl,
                                                          unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* A = smem;               // 128 rows x 128 B, 128-byte swizzle
  uint8_t* B = smem + 128 * 128;   // 256 rows x 128 B
  uint8_t* E = B + kN * 128;       // 2 KiB metadata chunk: 128 lanes x 16 B
  __shared__ __align__(8) uint64_t bar;
  __shared__ __align__(8) uint64_t stage_bar[8];
  __shared__ uint32_t slot;
  const int t = threadIdx.x, warp = t >> 5;
  // small finite operands: 1.0 in every bf16 slot of A and B
  for (int i = t; i < (128 + kN) * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0x3F803F80u;
  for (int i = t; i < 128 * 4; i += blockDim.x) reinterpret_cast<uint32_t*>(E)[i] = 0x44444444u;
  if (t == 0) {
    mbar_init(&bar, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&stage_bar[i], 1);
    fence_mbar_init();
  }
  fence_proxy_async();
  if (warp == 0) {
    tmem_alloc(&slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = slot;
  // metadata column 256 (32-column aligned): every group keeps positions 0 and 1
  tc_st_32x32b_x1(tm + (static_cast<uint32_t>(warp * 32) << 16) + 256, 0x44444444u);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t == 0) {
    constexpr uint32_t ID = idesc_bf16(128, kN, false), IDS = idesc_bf16(128, kN, true);
    const uint64_t t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const uint32_t k = i & 3;
      if (mode == 2) {
        const uint32_t slot_col = tm + 256 + (i & 7) * 32;
        tc_cp_128x128b(slot_col, sdesc(smem_u32(E), 128, 128, SWZ_NONE));
        tc_mma_sp(tm, sdesc(smem_u32(A) + (k & 1) * 32, 16, 1024, SWZ_128B),
                  sdesc(smem_u32(B) + (k & 1) * 64, 16, 1024, SWZ_128B), slot_col, IDS, i != 0);
      } else if (mode == 5) {
        tc_mma_sp(tm, sdesc(smem_u32(A) + (k & 1) * 32, 16, 512, SWZ_64B),
                  sdesc(smem_u32(B) + (k & 1) * 64, 16, 1024, SWZ_128B), tm + 256, IDS, i != 0);
      } else if (mode >= 1) {
        tc_mma_sp(tm, sdesc(smem_u32(A) + (k & 1) * 32, 16, 1024, SWZ_128B),
                  sdesc(smem_u32(B) + (k & 1) * 64, 16, 1024, SWZ_128B), tm + 256, IDS, i != 0);
        if (mode == 3 && (i & 1)) tc_commit(&stage_bar[(i >> 1) & 7]);
        if (mode == 4 && (i & 3) == 3) {
          tc_commit(&stage_bar[(i >> 1) & 7]);
          tc_commit(&stage_bar[((i >> 1) + 1) & 7]);
        }
      }
      else
        tc_mma(tm, sdesc(smem_u32(A) + k * 32, 16, 1024, SWZ_128B), sdesc(smem_u32(B) + k * 32, 16, 1024, SWZ_128B),
               ID, i != 0);
    }
    tc_commit(&bar);
    const bool ok = mbar_wait(&bar, 0, ctl, 5);
    const uint64_t t1 = clock64();
    if (ok) atomicMax(cycles, static_cast<unsigned long long>(t1 - t0));
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// CTA-pair variant: modes 6 (sparse, A 128-byte swizzle), 7 (sparse, A 64-byte swizzle), 8 (dense);
// M = 256 across the pair, N = 256 (each CTA holds 128 rows of B).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    mma_rate_pair_kernel(int mode, int iters, DevCtl ctl, unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* A = smem;              // 128 rows x 128 B
  uint8_t* B = smem + 128 * 128;  // 128 rows x 128 B (this CTA's half of N = 256)
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  const int t = threadIdx.x, warp = t >> 5;
  const bool leader = cluster_ctarank() == 0;
  for (int i = t; i < 256 * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0x3F803F80u;
  if (t == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  fence_proxy_async();
  if (warp == 0) {
    tmem_alloc_pair(&slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tm = slot;
  for (int col = 256; col < 288; ++col) tc_st_32x32b_x1(tm + (static_cast<uint32_t>(warp * 32) << 16) + col, 0x44444444u);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (t == 0 && leader) {
    constexpr uint32_t ID = idesc_bf16(256, 256, false), IDS = idesc_bf16(256, 256, true);
    const uint64_t t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const uint32_t k = i & 3;
      if (mode == 6)
        tc_mma_sp_pair(tm, sdesc(smem_u32(A) + (k & 1) * 32, 16, 1024, SWZ_128B),
                       sdesc(smem_u32(B) + (k & 1) * 64, 16, 1024, SWZ_128B), tm + 256, IDS, i != 0);
      else if (mode == 7)
        tc_mma_sp_pair(tm, sdesc(smem_u32(A) + (k & 1) * 32, 16, 512, SWZ_64B),
                       sdesc(smem_u32(B) + (k & 1) * 64, 16, 1024, SWZ_128B), tm + 256, IDS, i != 0);
      else
        tc_mma_pair(tm, sdesc(smem_u32(A) + k * 32, 16, 1024, SWZ_128B),
                    sdesc(smem_u32(B) + k * 32, 16, 1024, SWZ_128B), ID, i != 0);
    }
    tc_commit_pair(&bar, 0x3);
    const bool ok = mbar_wait(&bar, 0, ctl, 6);
    const uint64_t t1 = clock64();
    if (ok) atomicMax(cycles, static_cast<unsigned long long>(t1 - t0));
  }
  __syncwarp();
  if (!leader) mbar_wait(&bar, 0, ctl, 7);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tm, 512);
  }
}

}  // namespace
}  // namespace lynx

using namespace lynx;

extern "C" int lynx_mma_rate(int mode, int iters, double* tflops, double* macs_per_clock, void* stream) {
  if (mode < 0 || mode > 8) return LYNX_ERR_UNSUPPORTED;
  const bool pair = mode >= 6;
  const int sparse = mode != 0;
  if (!tflops || !macs_per_clock) return LYNX_ERR_NULL;
  if (iters < 1 || iters > (1 << 24)) return LYNX_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // operands need 48 KiB; asking for 150 KiB keeps one CTA (and one 512-column TMEM owner) per SM
  const int smem = 150 * 1024;
  if (cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(mma_rate_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return LYNX_ERR_CUDA;
  unsigned long long* cyc = nullptr;
  int* err = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&cyc), g_rate_cycles) != cudaSuccess ||
      cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_rate_error) != cudaSuccess)
    return LYNX_ERR_CUDA;
  cudaMemsetAsync(cyc, 0, sizeof(unsigned long long), st);
  cudaMemsetAsync(err, 0, sizeof(int), st);
  DevCtl ctl{err, 2000000000ull, 0};
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  const int grid = pair ? sm_count() / 2 * 2 : sm_count();
  for (int rep = 0; rep < 2; ++rep) {  // warm-up, then the timed launch
    if (rep == 1) cudaEventRecord(e0, st);
    if (pair)
      mma_rate_pair_kernel<<<grid, 128, smem, st>>>(mode, iters, ctl, cyc);
    else
      mma_rate_kernel<<<grid, 128, smem, st>>>(mode, iters, ctl, cyc);
  }
  cudaEventRecord(e1, st);
  unsigned long long hc = 0;
  int herr = 0;
  cudaMemcpyAsync(&hc, cyc, sizeof(hc), cudaMemcpyDeviceToHost, st);
  cudaMemcpyAsync(&herr, err, sizeof(herr), cudaMemcpyDeviceToHost, st);
  const cudaError_t e = cudaStreamSynchronize(st);
  float ms = 0.f;
  cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return LYNX_ERR_CUDA;
  if (herr) return LYNX_ERR_TIMEOUT;
  // dense-equivalent work per MMA and SM: 128 rows x 256 x K with K = 16 (dense) or 32 logical (sparse);
  // a pair MMA covers 256 rows on two SMs
  const bool sp = mode != 0 && mode != 8;
  const double macs = static_cast<double>(grid) * iters * 128.0 * kN * (sp ? 32.0 : 16.0);
  *tflops = 2.0 * macs / (ms * 1e-3) / 1e12;
  *macs_per_clock = hc ? static_cast<double>(iters) * 128.0 * kN * (sp ? 32.0 : 16.0) / static_cast<double>(hc)
                       : 0.0;
  return LYNX_OK;
}
