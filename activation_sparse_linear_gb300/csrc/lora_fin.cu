// The rest of the sparse layer's first half when its input H was produced -- and already sparsified -- by the
// previous layer's GELU epilogue (the MLP pair; "RT-Lynx" page, CUDA kernel optimisation: one execution path for
// the online sparsification):
//   T  = H LB^T on the tensor core (the LoRA down-projection of the dense input, Method: Yr = X (LA LB)^T),
//   s  = sqrt(sum h^2 / sum kept h^2) per row (Code examples, first formula), from the epilogue's per-slot
//        partial sums added in slot order, 1 when the kept sum is zero,
//   T' = bf16(T * (1 / s)), the intermediate the sparse GEMM's LoRA stage reads.
//
// Work units are (128-row tile, k-split) pairs.  A CTA runs units one after another: warp 0 issues the TMA
// loads of H (128 x 64, 128-byte swizzle) and LB (64 x 64) into a ring of stages, warp 1 issues four
// tcgen05.mma (M = 128, N = 64, K = 16) per stage into a 64-column TMEM accumulator, warps 2-5 drain it.  With
// more than one split every unit writes its fp32 partial (128 x 64) to global memory and the unit that takes
// the tile's last arrival ticket adds the partials in split order, so the result does not depend on which
// unit finishes last; no unit waits for another.  Every mbarrier wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kernels.h"

namespace lynx {
namespace {

constexpr int F_ROWS = 128;
constexpr int F_NST = 8;
constexpr int F_AT = F_ROWS * 128;           // H tile: 128 rows x 64 channels
constexpr int F_BT = kRankLB * 128;          // LB tile: 64 ranks x 64 channels
constexpr int F_STAGE = F_AT + F_BT;
constexpr int F_THREADS = 192;               // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int F_SMEM = F_NST * F_STAGE + 256 + 1024;
constexpr int F_MAX_SPLIT = 8;
static_assert(F_SMEM <= 232448, "shared memory budget");

enum Site : int { SITE_F_PRODUCER = 31, SITE_F_MMA = 32, SITE_F_EPILOGUE = 33, SITE_F_DRAIN = 34 };

__global__ void __launch_bounds__(F_THREADS, 1) lora_fin_kernel(const __grid_constant__ FinArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + F_NST * F_STAGE);
  uint64_t* empty = full + F_NST;
  uint64_t* acc_full = empty + F_NST;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* epi_bar = drain + 1;   // every epilogue warp has written its share of the partial
  uint64_t* epi_bar2 = drain + 2;  // the unit's arrival ticket is known
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* consumed_sh = abort_flag + 1;
  volatile int* issued_sh = abort_flag + 2;
  volatile int* last_flag = abort_flag + 3;
  static_assert(8 * (2 * F_NST + 5) + 20 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (a.M + F_ROWS - 1) / F_ROWS;
  const int nk = (a.K + 63) / 64;
  const int S = a.splits;
  const int nunits = num_m * S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < F_NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    mbar_init(epi_bar, 4);
    mbar_init(epi_bar2, 1);
    *abort_flag = 0;
    *consumed_sh = 0;
    *issued_sh = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmH);
    prefetch_tmap(&a.tmLB);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  pdl_launch_dependents();
  pdl_wait();  // H and the norm partials come from the previous kernel

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int g = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < nunits && !stop; u += gridDim.x) {
        const int mt = u % num_m, ks = u / num_m;
        const int kbeg = ks * nk / S, kend = (ks + 1) * nk / S;
        for (int kk = kbeg; kk < kend; ++kk, ++g) {
          const int st = g % F_NST;
          if (!mbar_wait(&empty[st], ((g / F_NST) & 1) ^ 1, a.ctl, SITE_F_PRODUCER) || *abort_flag) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* sA = smem + st * F_STAGE;
          mbar_arrive_expect_tx(&full[st], F_STAGE);
          tma_load_2d(sA, &a.tmH, &full[st], kk * 64, mt * F_ROWS);
          tma_load_2d(sA + F_AT, &a.tmLB, &full[st], kk * 64, 0);
        }
      }
      *issued_sh = g;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC = idesc_bf16(F_ROWS, kRankLB, false);
      constexpr uint64_t STEP = F_STAGE >> 4;
      const uint64_t a0 = sdesc(smem_u32(smem), 16, 1024, SWZ_128B);
      const uint64_t b0 = sdesc(smem_u32(smem) + F_AT, 16, 1024, SWZ_128B);
      int g = 0, tcount = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < nunits && !stop; u += gridDim.x, ++tcount) {
        const int ks = u / num_m;
        const int kbeg = ks * nk / S, kend = (ks + 1) * nk / S;
        if (!mbar_wait(acc_empty, (tcount & 1) ^ 1, a.ctl, SITE_F_MMA)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int kk = kbeg; kk < kend; ++kk, ++g) {
          const int st = g % F_NST;
          if (!mbar_wait(&full[st], (g / F_NST) & 1, a.ctl, SITE_F_MMA)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a0 + st * STEP, bd = b0 + st * STEP;
          tc_mma(tmem, ad, bd, IDESC, kk != kbeg);
          tc_mma(tmem, ad + 2, bd + 2, IDESC, 1);
          tc_mma(tmem, ad + 4, bd + 4, IDESC, 1);
          tc_mma(tmem, ad + 6, bd + 6, IDESC, 1);
          tc_commit(&empty[st]);
        }
        if (!stop) tc_commit(acc_full);
      }
      *consumed_sh = g;
      tc_commit(drain);
      mbar_wait(drain, 0, a.ctl, SITE_F_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- epilogue: one row per lane
    const int q = warp & 3;
    int tcount = 0, nsplit = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++tcount) {
      const int mt = u % num_m, ks = u / num_m;
      const int rloc = q * 32 + lane, row = mt * F_ROWS + rloc;
      bool ok = mbar_wait(acc_full, tcount & 1, a.ctl, SITE_F_EPILOGUE);
      ok = __all_sync(0xFFFFFFFFu, ok) && !*abort_flag;
      if (!ok) break;
      tc_fence_after();
      float t[64];
      {
        uint32_t r0[32], r1[32];
        tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16), r0);
        tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + 32, r1);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          t[j] = __uint_as_float(r0[j]);
          t[32 + j] = __uint_as_float(r1[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);  // the accumulator may be overwritten now
      bool finish = true;
      if (S > 1) {
        float4* mine = reinterpret_cast<float4*>(a.partials + ((static_cast<int64_t>(mt) * S + ks) * F_ROWS + rloc) * kRankLB);
#pragma unroll
        for (int v = 0; v < 16; ++v) mine[v] = make_float4(t[4 * v], t[4 * v + 1], t[4 * v + 2], t[4 * v + 3]);
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_bar);
        ok = mbar_wait(epi_bar, nsplit & 1, a.ctl, SITE_F_EPILOGUE);
        if (ok && warp == 2 && lane == 0) {
          unsigned int ticket;
          asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(a.counters + mt) : "memory");
          *last_flag = ticket == static_cast<unsigned int>(S - 1);
          mbar_arrive(epi_bar2);
        }
        ok = ok && mbar_wait(epi_bar2, nsplit & 1, a.ctl, SITE_F_EPILOGUE);
        ok = __all_sync(0xFFFFFFFFu, ok);
        ++nsplit;
        if (!ok) break;
        finish = *last_flag != 0;
        if (finish) {
          __threadfence();
          // add the partials in split order, four columns at a time; every split's load of a group is issued
          // before the group is added, so the L2 round trips overlap
          const float4* src = reinterpret_cast<const float4*>(a.partials + (static_cast<int64_t>(mt) * S * F_ROWS + rloc) * kRankLB);
          const int64_t sstride = static_cast<int64_t>(F_ROWS) * kRankLB / 4;  // float4s between splits
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            float4 p[F_MAX_SPLIT];
#pragma unroll
            for (int s2 = 0; s2 < F_MAX_SPLIT; ++s2)
              if (s2 < S) p[s2] = __ldcg(src + s2 * sstride + v);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int s2 = 0; s2 < F_MAX_SPLIT; ++s2)
              if (s2 < S) {
                acc.x += p[s2].x;
                acc.y += p[s2].y;
                acc.z += p[s2].z;
                acc.w += p[s2].w;
              }
            t[4 * v] = acc.x;
            t[4 * v + 1] = acc.y;
            t[4 * v + 2] = acc.z;
            t[4 * v + 3] = acc.w;
          }
        }
      }
      if (finish && row < a.M) {
        float nx = 0.f, nkept = 0.f;
        const float2* hn = a.hnorm + static_cast<int64_t>(row) * a.slots;
        for (int j = 0; j < a.slots; ++j) {  // slot order
          const float2 p = hn[j];
          nx += p.x;
          nkept += p.y;
        }
        const float sv = nkept > 0.f ? sqrtf(nx / nkept) : 1.f;
        const float inv = 1.f / sv;  // T' = T * (1 / s): one division per row
        a.s[row] = sv;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.T) + static_cast<int64_t>(row) * kRankLB);
#pragma unroll
        for (int v8 = 0; v8 < 8; ++v8) {
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(t[8 * v8 + 2 * j] * inv, t[8 * v8 + 2 * j + 1] * inv);
            pk[j] = *reinterpret_cast<uint32_t*>(&b2);
          }
          dst[v8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();

  if (*abort_flag && warp == 0 && lane == 0) {
    // Let every copy this CTA started land before its shared memory is released.
    const int issued = *issued_sh;
    for (int g = *consumed_sh; g < issued; ++g)
      if (!mbar_wait(&full[g % F_NST], (g / F_NST) & 1, a.ctl, SITE_F_DRAIN)) break;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

// k-splits: enough units for half of the SMs (their loads already outrun HBM), at most F_MAX_SPLIT, at least two
// 64-channel steps per unit.
int lora_fin_splits(int M, int K) {
  const int num_m = (M + F_ROWS - 1) / F_ROWS;
  const int nk = (K + 63) / 64;
  int s = (sm_count() / 2 + num_m - 1) / num_m;
  if (s > F_MAX_SPLIT) s = F_MAX_SPLIT;
  if (s > nk / 2) s = nk / 2;
  return s < 1 ? 1 : s;
}

size_t lora_fin_partial_bytes(int M, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>((M + F_ROWS - 1) / F_ROWS) * splits * F_ROWS * kRankLB * 4;
}

int lora_fin_counters(int M) { return (M + F_ROWS - 1) / F_ROWS; }

cudaError_t launch_lora_fin(const FinArgs& a, cudaStream_t st) {
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(lora_fin_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int nunits = ((a.M + F_ROWS - 1) / F_ROWS) * a.splits;
  const int grid = nunits < sm_count() ? nunits : sm_count();
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(F_THREADS);
  cfg.dynamicSmemBytes = F_SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lora_fin_kernel, a);
}

}  // namespace lynx
