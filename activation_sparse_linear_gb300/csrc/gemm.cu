// tcgen05 GEMM for the RT-Lynx linear layer: Y = rowscale o (A_op . B^T) [+ T'. LA^T]
//
// One CTA computes a 128 x BN output tile with a 128 x BN fp32 accumulator in
// tensor memory (TMEM).  Warp 0 (one lane) is the TMA producer, warp 1 (one
// lane) issues tcgen05.mma; afterwards all four warps drain TMEM through
// tcgen05.ld, apply the per-row scale and store bf16.
//
// Operand staging per pipeline stage (64 logical input channels):
//   * dense A: 128 rows x 64 bf16 (128 B rows, 128-byte swizzle)       16 KiB
//   * sparse A: 128 rows x 32 kept bf16 (64 B rows, 64-byte swizzle)     8 KiB
//   * B: BN rows x 64 bf16 (128 B rows, 128-byte swizzle)               BN*128 B
//   * sparse metadata: two 2 KiB chunks (one per tcgen05.mma.sp, 128 lanes x
//     16 B, word 0 used); tcgen05.cp.128x128b moves each chunk to its own TMEM
//     slot, 8 slots on 32-column boundaries after the accumulator, and the MMA
//     reads the slot's first column.
// The LoRA-up branch ("RT-Lynx" page, CUDA kernel optimisation: Yr is produced
// on chip and accumulated into Ys) is one extra stage: A = T' (128 x R), B = LA
// (BN x R), four dense K=16 MMAs into the same accumulator.  Because the
// epilogue multiplies the whole tile by s, T' holds (X LB^T)/s.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace lynx {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_SLOT = BM * 128;
constexpr int META_SLOT = 2 * kMetaChunkBytes;  // two MMAs per stage
constexpr int META_RING = 8;                     // TMEM metadata slots
constexpr int META_SLOT_COLS = 32;               // slot pitch in TMEM columns

enum Site : int { SITE_PRODUCER = 1, SITE_MMA = 2, SITE_EPILOGUE = 3, SITE_DRAIN = 4 };

template <int BN, bool SPARSE, bool LORA>
struct Cfg {
  static constexpr int B_SLOT = BN * 128;
  static constexpr int STAGE = A_SLOT + B_SLOT + (SPARSE ? META_SLOT : 0);
  static constexpr int NST = BN <= 64 ? 8 : 4;
  static constexpr int TMEM_COLS = SPARSE ? 512 : (BN < 32 ? 32 : BN);
  static constexpr int META_COL = BN;  // first TMEM column of the metadata ring
  static_assert(META_COL + (SPARSE ? META_RING * META_SLOT_COLS : 0) <= TMEM_COLS, "TMEM budget");
  static_assert(!SPARSE || 2 * NST <= META_RING, "a slot must outlive the stages in flight");
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = NST * STAGE + BAR_BYTES + 1024;
  static_assert(STAGE % 1024 == 0, "stage slots must keep 1 KiB alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int BN, bool SPARSE, bool LORA>
__global__ void __launch_bounds__(128, 1) gemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = Cfg<BN, SPARSE, LORA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE);
  uint64_t* empty = full + C::NST;
  uint64_t* accb = empty + C::NST;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* consumed_sh = abort_flag + 1;
  volatile int* issued_sh = abort_flag + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int nk = (a.K + BK - 1) / BK;
  const int iters = nk + (LORA ? 1 : 0);
  const int64_t chunks_k = meta_chunks_k(a.K);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    *consumed_sh = 0;
    *issued_sh = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmA);
    prefetch_tmap(&a.tmB);
    if (LORA) {
      prefetch_tmap(&a.tmT);
      prefetch_tmap(&a.tmLA);
    }
  }
  if (warp == 1) {
    tmem_alloc(tslot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    int issued = 0;
    for (int it = 0; it < iters; ++it) {
      const int st = it % C::NST;
      const uint32_t ph = (it / C::NST) & 1;
      if (!mbar_wait(&empty[st], ph ^ 1, a.ctl, SITE_PRODUCER) || *abort_flag) {
        *abort_flag = 1;
        break;
      }
      uint8_t* sA = smem + st * C::STAGE;
      uint8_t* sB = sA + A_SLOT;
      uint8_t* sM = sB + C::B_SLOT;
      if (a.ctl.inject == 1 && it == 0) continue;  // test hook: this stage never arrives
      if (it < nk) {
        const uint32_t bytes = (SPARSE ? BM * 64 : A_SLOT) + C::B_SLOT + (SPARSE ? META_SLOT : 0);
        mbar_arrive_expect_tx(&full[st], bytes);
        tma_load_2d(sA, &a.tmA, &full[st], SPARSE ? it * (BK / 2) : it * BK, m0);
        tma_load_2d(sB, &a.tmB, &full[st], it * BK, n0);
        if (SPARSE)
          bulk_load(sM, a.meta + (static_cast<int64_t>(blockIdx.y) * chunks_k + 2 * it) * kMetaChunkBytes,
                    META_SLOT, &full[st]);
      } else {
        mbar_arrive_expect_tx(&full[st], A_SLOT + C::B_SLOT);
        tma_load_2d(sA, &a.tmT, &full[st], 0, m0);
        tma_load_2d(sB, &a.tmLA, &full[st], 0, n0);
      }
      issued = it + 1;
    }
    *issued_sh = issued;
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC = idesc_bf16(BM, BN, false);
    constexpr uint32_t IDESC_SP = idesc_bf16(BM, BN, true);
    int consumed = 0;
    for (int it = 0; it < iters; ++it) {
      const int st = it % C::NST;
      const uint32_t ph = (it / C::NST) & 1;
      if (!mbar_wait(&full[st], ph, a.ctl, SITE_MMA)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t sA = smem_u32(smem + st * C::STAGE);
      const uint32_t sB = sA + A_SLOT;
      if (it < nk) {
        if constexpr (SPARSE) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t mcol = tmem + C::META_COL + ((2 * it + j) % META_RING) * META_SLOT_COLS;
            tc_cp_128x128b(mcol, sdesc(sB + C::B_SLOT + j * kMetaChunkBytes, 128, 128, SWZ_NONE));
            tc_mma_sp(tmem, sdesc(sA + j * 32, 16, 512, SWZ_64B), sdesc(sB + j * 64, 16, 1024, SWZ_128B), mcol,
                      IDESC_SP, (it | j) != 0);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(tmem, sdesc(sA + j * 32, 16, 1024, SWZ_128B), sdesc(sB + j * 32, 16, 1024, SWZ_128B), IDESC,
                   (it | j) != 0);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc_mma(tmem, sdesc(sA + j * 32, 16, 1024, SWZ_128B), sdesc(sB + j * 32, 16, 1024, SWZ_128B), IDESC, 1);
      }
      tc_commit(&empty[st]);
      consumed = it + 1;
    }
    tc_commit(accb);  // fires once every issued MMA has completed (also after an abort)
    *consumed_sh = consumed;
  }
  __syncwarp();
  __syncthreads();
  const bool aborted = *abort_flag != 0;

  if (aborted && warp == 0 && lane == 0) {
    // Let every copy this CTA started land before its shared memory is released.
    const int issued = *issued_sh;
    for (int it = *consumed_sh; it < issued; ++it) {
      if (a.ctl.inject == 1 && it == 0) continue;
      if (!mbar_wait(&full[it % C::NST], (it / C::NST) & 1, a.ctl, SITE_DRAIN)) break;
    }
  }

  // ---------------------------------------------------------------- epilogue
  bool ok = mbar_wait(accb, 0, a.ctl, SITE_EPILOGUE);
  ok = __all_sync(0xFFFFFFFFu, ok) && !aborted;
  tc_fence_after();
  if (ok) {
    const int row = m0 + warp * 32 + lane;
    float sc = 1.f;
    if (a.scale_mode != SCALE_NONE && row < a.M) sc = a.rowscale[row];
    const bool divide = a.scale_mode == SCALE_DIV;
    __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(a.Y) + static_cast<int64_t>(row) * a.ldy;
    const bool vec_ok = (a.ldy % 8) == 0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, r);
      tc_wait_ld();
      if (row < a.M) {
        const int col0 = n0 + c * 32;
        __nv_bfloat162 o[16];
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
          o[j] = __floats2bfloat162_rn(x0, x1);
        }
        if (vec_ok && col0 + 32 <= a.N) {
          uint4* dst = reinterpret_cast<uint4*>(yrow + col0);
          const uint4* src = reinterpret_cast<const uint4*>(o);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = src[q];
        } else {
          const __nv_bfloat16* ob = reinterpret_cast<const __nv_bfloat16*>(o);
          for (int j = 0; j < 32; ++j)
            if (col0 + j < a.N) yrow[col0 + j] = ob[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN, bool SPARSE, bool LORA>
cudaError_t launch(const GemmArgs& a, cudaStream_t st) {
  using C = Cfg<BN, SPARSE, LORA>;
  auto* k = gemm_kernel<BN, SPARSE, LORA>;
  static bool attr_set[64] = {};  // per device; setting it twice from racing threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM);
  k<<<grid, 128, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(int kind, const GemmArgs& a, cudaStream_t st) {
  switch (kind) {
    case 0: return launch<256, false, false>(a, st);
    case 1: return launch<256, false, true>(a, st);
    case 2: return launch<256, true, true>(a, st);
    case 3: return launch<256, true, false>(a, st);
    case 4: return launch<64, false, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lynx
