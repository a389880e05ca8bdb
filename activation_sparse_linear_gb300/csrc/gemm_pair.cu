// CTA-pair (cta_group::2) tcgen05 GEMM for the RT-Lynx linear layer:
//   Y[256 x 256 tile] = rowscale o (A_op . W^T) [+ T' . LA^T]
//
// Two CTAs of a cluster share one 256 x 256 output tile.  CTA r of the pair
// owns rows 128r..128r+127 of the tile (its TMEM holds their 128 x 256 fp32
// accumulator) and stages, per step, its own 128 rows of A and its half (128
// columns) of the W tile; one tcgen05.mma.cta_group::2 issued by the leader
// CTA (rank 0) multiplies the whole 256 x 256 x K step, reading A and W from
// both CTAs' shared memory, so each CTA stages half of the weight bytes a
// single-CTA 128 x 256 tile would need.
//
// Sparse A (compressed values, 128-byte swizzle) goes through
// tcgen05.mma.sp.cta_group::2 in steps of 128 channels: every stage carries
// each CTA's 2 KiB metadata chunk of those channels, which the leader copies
// into both TMEMs with one tcgen05.cp.cta_group::2 (each CTA's own shared
// memory into its own TMEM); MMA j of the stage reads the even column pair
// (j & 2) with the sparsity selector j & 1.
//
// The LoRA-up branch ("RT-Lynx" page, CUDA kernel optimisation: Yr is produced
// on chip and accumulated into Ys) is one extra stage: A = T' (128 x 64),
// B = this CTA's half of LA; four dense MMAs into the same accumulator.
// Because the epilogue multiplies the tile by s, T' holds (X LB^T)/s.
//
// Roles per CTA: warp 0 lane 0 TMA producer (both CTAs), warp 1 lane 0 MMA
// issuer (leader only), warps 2-9 epilogue (two warps per TMEM lane quarter,
// 128 columns each: TMEM -> registers -> scale -> bf16 -> global).  Every
// mbarrier wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace lynx {
namespace {

constexpr int ROWS = 128;          // rows per CTA
constexpr int TN = 256;            // output columns per pair tile (MMA N)
constexpr int HALF_N = TN / 2;     // W rows staged per CTA
constexpr int META_RING = 8;       // TMEM metadata groups
constexpr int META_GROUP_COLS = 4;
constexpr int META_COL = TN;       // first metadata column (after the accumulator)
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int SUB = HALF_N * 128;  // one 64-channel W sub-tile of this CTA (128 rows x 128 B)

enum Site : int { SITE_PRODUCER = 11, SITE_MMA = 12, SITE_EPILOGUE = 13, SITE_DRAIN = 14 };

// Per stage and CTA: sparse = 128 channels (A: 64 kept values per row, 128-byte rows; W: two 64-channel
// sub-tiles; one metadata chunk) feeding four tcgen05.mma.sp; dense = 64 channels feeding four tcgen05.mma.
// Four MMAs per barrier round keep the single issuing thread ahead of the tensor pipe.
template <bool SPARSE>
struct PairCfg {
  static constexpr int BK = SPARSE ? 128 : 64;
  static constexpr int A_SLOT = ROWS * 128;
  static constexpr int B_SLOT = SPARSE ? 2 * SUB : SUB;
  static constexpr int M_SLOT = SPARSE ? kMetaChunkBytes : 0;
  static constexpr int STAGE = A_SLOT + B_SLOT + M_SLOT;
  static constexpr int NST = SPARSE ? 4 : 6;
  static constexpr int SMEM = NST * STAGE + 256 + 1024;
  static_assert(STAGE % 1024 == 0, "stage slots keep 1 KiB alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NST <= META_RING, "a metadata group must outlive the stages in flight");
};

template <bool SPARSE, bool LORA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ PairArgs a) {
  using C = PairCfg<SPARSE>;
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
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int num_mp = (a.M + 2 * ROWS - 1) / (2 * ROWS);
  const int num_n = (a.N + TN - 1) / TN;
  const int ntiles = num_mp * num_n;
  const int nk = (a.K + C::BK - 1) / C::BK;
  const int nstages = nk + (LORA ? 1 : 0);
  const int64_t blocks_k = meta_blocks_k(a.K);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * EPI_WARPS);  // every epilogue warp of both CTAs of the pair
    mbar_init(drain, 1);
    *abort_flag = 0;
    *consumed_sh = 0;
    *issued_sh = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmA);
    prefetch_tmap(&a.tmB);
    if (SPARSE) prefetch_tmap(&a.tmMeta);
    if (LORA) {
      prefetch_tmap(&a.tmT);
      prefetch_tmap(&a.tmLA);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tslot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      constexpr uint32_t STAGE_BYTES = C::A_SLOT + C::B_SLOT + C::M_SLOT;
      constexpr uint32_t LORA_BYTES = C::A_SLOT + SUB;
      const uint32_t full_leader0 = mapa_shared(&full[0], 0);  // the leader's full barriers, 8 B apart
      int g = 0, st = 0;
      uint32_t ph = 0;
      bool stop = false;
      for (int tile = cluster; tile < ntiles && !stop; tile += nclusters) {
        const int mp = tile % num_mp, nb = tile / num_mp;
        const int m0 = mp * 2 * ROWS + static_cast<int>(rank) * ROWS;
        const int n0 = nb * TN + static_cast<int>(rank) * HALF_N;
        const int meta_row = static_cast<int>(2 * ((mp * 2 + static_cast<int>(rank)) * blocks_k));
        for (int it = 0; it < nstages; ++it) {
          if (!mbar_wait(&empty[st], ph ^ 1, a.ctl, SITE_PRODUCER) || *abort_flag) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* sA = smem + st * C::STAGE;
          uint8_t* sB = sA + C::A_SLOT;
          const uint32_t fb = full_leader0 + 8 * st;
          if (!(a.ctl.inject == 1 && g == 0)) {  // test hook: the first stage never arrives
            if (it < nk) {
              if (leader) mbar_arrive_expect_tx(&full[st], 2 * STAGE_BYTES);
              if constexpr (SPARSE) {
                tma_load_2d_pair(sA, &a.tmA, fb, it * 64, m0);
                tma_load_2d_pair(sB, &a.tmB, fb, it * 128, n0);
                tma_load_2d_pair(sB + SUB, &a.tmB, fb, it * 128 + 64, n0);
                tma_load_2d_pair(sB + C::B_SLOT, &a.tmMeta, fb, 0, meta_row + 2 * it);
              } else {
                tma_load_2d_pair(sA, &a.tmA, fb, it * 64, m0);
                tma_load_2d_pair(sB, &a.tmB, fb, it * 64, n0);
              }
            } else {
              if (leader) mbar_arrive_expect_tx(&full[st], 2 * LORA_BYTES);
              tma_load_2d_pair(sA, &a.tmT, fb, 0, m0);
              tma_load_2d_pair(sB, &a.tmLA, fb, 0, n0);
            }
          }
          ++g;
          if (++st == C::NST) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      *issued_sh = g;
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (leader)
      // Descriptors and TMEM addresses are built once; each stage only adds offsets, so the issuing
      // thread's work per MMA stays well under the MMA's own duration.
      constexpr uint32_t IDESC = idesc_bf16(2 * ROWS, TN, false);
      constexpr uint32_t IDESC_SP = idesc_bf16(2 * ROWS, TN, true);
      constexpr uint64_t STEP = C::STAGE >> 4;  // descriptor start-address units per stage
      const uint32_t s0 = smem_u32(smem);
      const uint64_t a0 = sdesc(s0, 16, 1024, SWZ_128B);
      const uint64_t b0 = sdesc(s0 + C::A_SLOT, 16, 1024, SWZ_128B);
      const uint64_t e0 = sdesc(s0 + C::A_SLOT + C::B_SLOT, 128, 128, SWZ_NONE);
      const uint32_t meta0 = tmem + META_COL;
      int g = 0, st = 0, tcount = 0;
      uint32_t ph = 0;
      bool stop = false;
      for (int tile = cluster; tile < ntiles && !stop; tile += nclusters, ++tcount) {
        if (!mbar_wait(acc_empty, (tcount & 1) ^ 1, a.ctl, SITE_MMA)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int it = 0; it < nstages; ++it) {
          if (!mbar_wait(&full[st], ph, a.ctl, SITE_MMA)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a0 + st * STEP, bd = b0 + st * STEP;
          const uint32_t acc0 = it != 0;
          if (it < nk) {
            if constexpr (SPARSE) {
              const uint32_t grp = meta0 + (it & (META_RING - 1)) * META_GROUP_COLS;
              tc_cp_pair_128x128b(grp, e0 + st * STEP);
              // MMA j: A bytes 32j of the 128-byte rows; W sub-tile j/2 at byte 64 (j%2);
              // metadata column pair j/2 with selector j%2
              tc_mma_sp_pair(tmem, ad, bd, grp, IDESC_SP, acc0);
              tc_mma_sp_pair(tmem, ad + 2, bd + 4, grp, IDESC_SP | 1u, 1);
              tc_mma_sp_pair(tmem, ad + 4, bd + (SUB >> 4), grp + 2, IDESC_SP, 1);
              tc_mma_sp_pair(tmem, ad + 6, bd + (SUB >> 4) + 4, grp + 2, IDESC_SP | 1u, 1);
            } else {
              tc_mma_pair(tmem, ad, bd, IDESC, acc0);
              tc_mma_pair(tmem, ad + 2, bd + 2, IDESC, 1);
              tc_mma_pair(tmem, ad + 4, bd + 4, IDESC, 1);
              tc_mma_pair(tmem, ad + 6, bd + 6, IDESC, 1);
            }
          } else {  // LoRA-up: T' (128 x 64) against this CTA's half of LA, four K = 16 steps
            tc_mma_pair(tmem, ad, bd, IDESC, 1);
            tc_mma_pair(tmem, ad + 2, bd + 2, IDESC, 1);
            tc_mma_pair(tmem, ad + 4, bd + 4, IDESC, 1);
            tc_mma_pair(tmem, ad + 6, bd + 6, IDESC, 1);
          }
          tc_commit_pair(&empty[st], 0x3);
          ++g;
          if (++st == C::NST) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!stop) tc_commit_pair(acc_full, 0x3);
      }
      *consumed_sh = g;
      tc_commit_pair(drain, 0x1);  // every MMA this pair issued has completed once this fires
      mbar_wait(drain, 0, a.ctl, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;          // which 128 of the 256 columns
    constexpr int COLS = TN / 2;
    const bool vec_ok = (a.ldy % 8) == 0;
    const bool scaled = a.scale_mode == SCALE_MUL;
    const uint32_t acc_empty_leader = mapa_shared(acc_empty, 0);
    int tcount = 0;
    for (int tile = cluster; tile < ntiles; tile += nclusters, ++tcount) {
      bool ok = mbar_wait(acc_full, tcount & 1, a.ctl, SITE_EPILOGUE);
      ok = __all_sync(0xFFFFFFFFu, ok) && !*abort_flag;
      if (!ok) break;
      tc_fence_after();
      const int mp = tile % num_mp, nb = tile / num_mp;
      const int row = mp * 2 * ROWS + static_cast<int>(rank) * ROWS + q * 32 + lane;
      const int n0 = nb * TN + half * COLS;
      const float sc = (scaled && row < a.M) ? a.rowscale[row] : 1.f;
      uint32_t packed[COLS / 2];
#pragma unroll
      for (int c = 0; c < COLS / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + half * COLS + c * 32, r);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * sc, __uint_as_float(r[2 * j + 1]) * sc);
          packed[c * 16 + j] = *reinterpret_cast<uint32_t*>(&h);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);  // the pair's accumulator may be overwritten
      if (row < a.M) {
        __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(a.Y) + static_cast<int64_t>(row) * a.ldy;
#pragma unroll
        for (int c = 0; c < COLS / 32; ++c) {
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
                reinterpret_cast<uint16_t*>(yrow)[col0 + j] =
                    (j & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFFu);
              }
            }
          }
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();

  if (*abort_flag && leader && warp == 0 && lane == 0) {
    // Let every copy of this stage sequence land (both CTAs signal the leader's barriers).
    const int issued = *issued_sh;
    for (int g = *consumed_sh; g < issued; ++g) {
      if (a.ctl.inject == 1 && g == 0) continue;
      if (!mbar_wait(&full[g % C::NST], (g / C::NST) & 1, a.ctl, SITE_DRAIN)) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still read its shared memory or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <bool SPARSE, bool LORA>
cudaError_t launch(const PairArgs& a, cudaStream_t st) {
  using C = PairCfg<SPARSE>;
  auto* k = gemm_pair_kernel<SPARSE, LORA>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int ntiles = ((a.M + 2 * ROWS - 1) / (2 * ROWS)) * ((a.N + TN - 1) / TN);
  int clusters = sm_count() / 2;
  if (clusters > ntiles) clusters = ntiles;
  if (clusters < 1) clusters = 1;
  k<<<2 * clusters, THREADS, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_pair(bool sparse, bool lora, const PairArgs& a, cudaStream_t st) {
  if (sparse) return lora ? launch<true, true>(a, st) : launch<true, false>(a, st);
  return lora ? launch<false, true>(a, st) : launch<false, false>(a, st);
}

}  // namespace lynx
