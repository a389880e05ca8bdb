// Dense tcgen05 projection GEMM: Y = bf16(rowscale o (A . B^T)), used for the
// LoRA down-projection T' = (X LB^T) / s on its own ("RT-Lynx" page, Method:
// Yr = X (LA LB)^T computed as (X LB^T) LA^T) and for the dense layer's
// low-rank branch.
//
// A persistent CTA walks 128 x BN output tiles with a 128 x BN fp32
// accumulator in tensor memory (TMEM).  Warp 0 (one lane) is the TMA producer,
// warp 1 (one lane) issues tcgen05.mma, warps 2-5 drain TMEM through
// tcgen05.ld into registers, hand the accumulator back to the MMA warp, then
// apply the per-row scale and store bf16 while the next tile's mainloop runs.
// Per pipeline stage (64 input channels): A 128 rows x 64 bf16 and B BN rows x
// 64 bf16, both 128-byte rows with the 128-byte swizzle.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kernels.h"

namespace lynx {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_SLOT = BM * 128;

enum Site : int { SITE_PRODUCER = 1, SITE_MMA = 2, SITE_EPILOGUE = 3, SITE_DRAIN = 4 };

template <int BN>
struct Cfg {
  static constexpr int B_SLOT = BN * 128;
  static constexpr int STAGE = A_SLOT + B_SLOT;
  static constexpr int NST = BN <= 64 ? 8 : 4;
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int THREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = NST * STAGE + BAR_BYTES + 1024;
  static_assert(STAGE % 1024 == 0, "stage slots must keep 1 KiB alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Persistent: CTA b processes tiles b, b + gridDim.x, ...; tile t covers rows
// (t % num_m) * 128 and columns (t / num_m) * BN, so the CTAs in flight share
// the B (weight) tiles they stream and the small A operand stays in L2.
template <int BN>
__global__ void __launch_bounds__(192, 1) gemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE);
  uint64_t* empty = full + C::NST;
  uint64_t* acc_full = empty + C::NST;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* consumed_sh = abort_flag + 1;
  volatile int* issued_sh = abort_flag + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (a.M + BM - 1) / BM;
  const int num_n = (a.N + BN - 1) / BN;
  const int ntiles = num_m * num_n;
  const int nk = (a.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *consumed_sh = 0;
    *issued_sh = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmA);
    prefetch_tmap(&a.tmB);
  }
  if (warp == 1) {
    tmem_alloc(tslot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int g = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
        const int m0 = (tile % num_m) * BM, n0 = (tile / num_m) * BN;
        for (int it = 0; it < nk; ++it) {
          const int st = g % C::NST;
          const uint32_t ph = (g / C::NST) & 1;
          if (!mbar_wait(&empty[st], ph ^ 1, a.ctl, SITE_PRODUCER) || *abort_flag) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* sA = smem + st * C::STAGE;
          if (a.ctl.inject == 1 && g == 0) {  // test hook: this stage never arrives
            ++g;
            continue;
          }
          mbar_arrive_expect_tx(&full[st], A_SLOT + C::B_SLOT);
          tma_load_2d(sA, &a.tmA, &full[st], it * BK, m0);
          tma_load_2d(sA + A_SLOT, &a.tmB, &full[st], it * BK, n0);
          ++g;
        }
      }
      *issued_sh = g;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC = idesc_bf16(BM, BN, false);
      int g = 0, tcount = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x, ++tcount) {
        if (!mbar_wait(acc_empty, (tcount & 1) ^ 1, a.ctl, SITE_MMA)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int it = 0; it < nk; ++it) {
          const int st = g % C::NST;
          const uint32_t ph = (g / C::NST) & 1;
          if (!mbar_wait(&full[st], ph, a.ctl, SITE_MMA)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + st * C::STAGE);
          const uint32_t sB = sA + A_SLOT;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(tmem, sdesc(sA + j * 32, 16, 1024, SWZ_128B), sdesc(sB + j * 32, 16, 1024, SWZ_128B), IDESC,
                   !(it == 0 && j == 0));
          tc_commit(&empty[st]);
          ++g;
        }
        if (!stop) tc_commit(acc_full);
      }
      *consumed_sh = g;
      tc_commit(drain);  // every MMA this CTA issued has completed once this fires
      mbar_wait(drain, 0, a.ctl, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const bool vec_ok = (a.ldy % 8) == 0;
    const bool divide = a.scale_mode == SCALE_DIV;
    int tcount = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tcount) {
      bool ok = mbar_wait(acc_full, tcount & 1, a.ctl, SITE_EPILOGUE);
      ok = __all_sync(0xFFFFFFFFu, ok) && !*abort_flag;
      if (!ok) break;
      tc_fence_after();
      const int m0 = (tile % num_m) * BM, n0 = (tile / num_m) * BN;
      const int row = m0 + q * 32 + lane;
      float sc = 1.f;
      if (a.scale_mode != SCALE_NONE && row < a.M) sc = a.rowscale[row];
      uint32_t packed[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 32, r);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x0 = __uint_as_float(r[2 * j]), x1 = __uint_as_float(r[2 * j + 1]);
          if (divide) {
            x0 = x0 / sc;
            x1 = x1 / sc;
          } else {
            x0 *= sc;
            x1 *= sc;
          }
          __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
          packed[c * 16 + j] = *reinterpret_cast<uint32_t*>(&h);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);  // the accumulator may be overwritten now
      if (row < a.M) {
        __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(a.Y) + static_cast<int64_t>(row) * a.ldy;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          const int col0 = n0 + c * 32;
          if (vec_ok && col0 + 32 <= a.N) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + col0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[c * 16 + 4 * v], packed[c * 16 + 4 * v + 1], packed[c * 16 + 4 * v + 2],
                                  packed[c * 16 + 4 * v + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (col0 + j < a.N) {
                const uint32_t w = packed[c * 16 + j / 2];
                const uint16_t b = (j & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFFu);
                reinterpret_cast<uint16_t*>(yrow)[col0 + j] = b;
              }
            }
          }
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();

  if (*abort_flag && warp == 0 && lane == 0) {
    // Let every copy this CTA started land before its shared memory is released.
    const int issued = *issued_sh;
    for (int g = *consumed_sh; g < issued; ++g) {
      if (a.ctl.inject == 1 && g == 0) continue;
      if (!mbar_wait(&full[g % C::NST], (g / C::NST) & 1, a.ctl, SITE_DRAIN)) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

int sm_count() {
  static std::atomic<int> counts[64] = {};  // per device; racing first calls store the same value
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = counts[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

template <int BN>
cudaError_t launch(const GemmArgs& a, cudaStream_t st) {
  using C = Cfg<BN>;
  auto* k = gemm_kernel<BN>;
  static std::atomic<bool> attr_set[64] = {};  // per device; setting it twice from racing threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int ntiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = ntiles < sm_count() ? ntiles : sm_count();
  k<<<grid, C::THREADS, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_proj_gemm(const GemmArgs& a, cudaStream_t st) {
  if (a.N != kRankLB) return cudaErrorInvalidValue;
  return launch<kRankLB>(a, st);
}

}  // namespace lynx
