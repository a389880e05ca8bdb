// tcgen05 GEMM for the RT-Lynx linear layer: Y = rowscale o (A_op . B^T) [+ T'. LA^T]
//
// A persistent CTA walks 128 x BN output tiles with a 128 x BN fp32
// accumulator in tensor memory (TMEM).  Warp 0 (one lane) is the TMA producer,
// warp 1 (one lane) issues tcgen05.mma, warps 2-5 drain TMEM through
// tcgen05.ld into registers, hand the accumulator back to the MMA warp, then
// apply the per-row scale and store bf16 while the next tile's mainloop runs.
//
// Operand staging per pipeline stage (64 logical input channels):
//   * dense A: 128 rows x 64 bf16 (128 B rows, 128-byte swizzle)       16 KiB
//   * sparse A: 128 rows x 32 kept bf16 (64 B rows, 64-byte swizzle)     8 KiB
//   * B: BN rows x 64 bf16 (128 B rows, 128-byte swizzle)               BN*128 B
//   * sparse metadata: every second stage carries the 2 KiB chunk of the next
//     128 channels (128 lanes x 16 B = four MMAs' words); tcgen05.cp.128x128b
//     moves it to a 4-column group of an 8-group TMEM ring after the
//     accumulator, and MMA j of the chunk reads column pair (j & 2) with the
//     sparsity selector j & 1.
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
constexpr int META_SLOT = kMetaChunkBytes;  // one chunk per two stages
constexpr int META_RING = 8;                // TMEM metadata groups
constexpr int META_GROUP_COLS = 4;          // columns per group (four MMAs)

enum Site : int { SITE_PRODUCER = 1, SITE_MMA = 2, SITE_EPILOGUE = 3, SITE_DRAIN = 4 };

template <int BN, bool SPARSE, bool LORA>
struct Cfg {
  static constexpr int B_SLOT = BN * 128;
  static constexpr int STAGE = A_SLOT + B_SLOT + (SPARSE ? META_SLOT : 0);
  static constexpr int NST = BN <= 64 ? 8 : 4;
  static constexpr int TMEM_COLS = SPARSE ? 512 : (BN < 32 ? 32 : BN);
  static constexpr int META_COL = BN;  // first TMEM column of the metadata ring
  static constexpr int THREADS = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = NST * STAGE + BAR_BYTES + 1024;
  static_assert(STAGE % 1024 == 0, "stage slots must keep 1 KiB alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(META_COL + (SPARSE ? META_RING * META_GROUP_COLS : 0) <= TMEM_COLS, "TMEM budget");
  static_assert(!SPARSE || NST <= 2 * META_RING, "a metadata group must outlive the stages in flight");
};

// Persistent: CTA b processes tiles b, b + gridDim.x, ...; tile t covers rows
// (t % num_m) * 128 and columns (t / num_m) * BN, so the CTAs in flight share
// the B (weight) tiles they stream and the small A operand stays in L2.
template <int BN, bool SPARSE, bool LORA>
__global__ void __launch_bounds__(192, 1) gemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = Cfg<BN, SPARSE, LORA>;
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
  const int S = a.splits;
  const int ntiles = num_m * num_n * S;
  const int nk = (a.K + BK - 1) / BK;
  // tile t -> row block t % num_m, split (t / num_m) % S, column block t / (num_m * S)
  auto kb_begin = [&](int tile) { return ((tile / num_m) % S) * nk / S; };
  auto kb_end = [&](int tile) { return ((tile / num_m) % S + 1) * nk / S; };
  const int64_t blocks_k = meta_blocks_k(a.K);

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

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int g = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
        const int m0 = (tile % num_m) * BM, n0 = (tile / (num_m * S)) * BN;
        const int k_end = kb_end(tile);
        for (int it = kb_begin(tile); it < k_end + (LORA ? 1 : 0); ++it) {
          const int st = g % C::NST;
          const uint32_t ph = (g / C::NST) & 1;
          if (!mbar_wait(&empty[st], ph ^ 1, a.ctl, SITE_PRODUCER) || *abort_flag) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* sA = smem + st * C::STAGE;
          uint8_t* sB = sA + A_SLOT;
          uint8_t* sM = sB + C::B_SLOT;
          if (a.ctl.inject == 1 && g == 0) {  // test hook: this stage never arrives
            ++g;
            continue;
          }
          if (it < k_end) {
            const bool meta_stage = SPARSE && (it % 2 == 0 || it == kb_begin(tile));
            const uint32_t bytes = (SPARSE ? BM * 64 : A_SLOT) + C::B_SLOT + (meta_stage ? META_SLOT : 0);
            mbar_arrive_expect_tx(&full[st], bytes);
            tma_load_2d(sA, &a.tmA, &full[st], SPARSE ? it * (BK / 2) : it * BK, m0);
            tma_load_2d(sB, &a.tmB, &full[st], it * BK, n0);
            if (meta_stage)
              bulk_load(sM, a.meta + (static_cast<int64_t>(m0 / BM) * blocks_k + it / 2) * kMetaChunkBytes,
                        META_SLOT, &full[st]);
          } else {
            mbar_arrive_expect_tx(&full[st], A_SLOT + C::B_SLOT);
            tma_load_2d(sA, &a.tmT, &full[st], 0, m0);
            tma_load_2d(sB, &a.tmLA, &full[st], 0, n0);
          }
          ++g;
        }
      }
      *issued_sh = g;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_SP = idesc_bf16(BM, BN, true);
      int g = 0, tcount = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x, ++tcount) {
        if (!mbar_wait(acc_empty, (tcount & 1) ^ 1, a.ctl, SITE_MMA)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int k_begin = kb_begin(tile), k_end = kb_end(tile);
        for (int it = k_begin; it < k_end + (LORA ? 1 : 0); ++it) {
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
          const uint32_t first = (it == k_begin);
          if (it < k_end) {
            if constexpr (SPARSE) {
              const uint32_t group = tmem + C::META_COL + ((it / 2) % META_RING) * META_GROUP_COLS;
              if (it % 2 == 0 || first) tc_cp_128x128b(group, sdesc(sB + C::B_SLOT, 128, 128, SWZ_NONE));
#pragma unroll
              for (int j = 0; j < 2; ++j)  // MMA 2*(it%2)+j of the chunk: column pair it%2, selector j
                tc_mma_sp(tmem, sdesc(sA + j * 32, 16, 512, SWZ_64B), sdesc(sB + j * 64, 16, 1024, SWZ_128B),
                          group + 2 * (it % 2), IDESC_SP | j, !(first && j == 0));
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tc_mma(tmem, sdesc(sA + j * 32, 16, 1024, SWZ_128B), sdesc(sB + j * 32, 16, 1024, SWZ_128B),
                       IDESC, !(first && j == 0));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tc_mma(tmem, sdesc(sA + j * 32, 16, 1024, SWZ_128B), sdesc(sB + j * 32, 16, 1024, SWZ_128B), IDESC,
                     1);
          }
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
      const int m0 = (tile % num_m) * BM, n0 = (tile / (num_m * S)) * BN;
      const int row = m0 + q * 32 + lane;
      if (a.partial) {
        // split-K: fp32 partial sums, unscaled, to partial[split][row][col]
        float* prow = a.partial + (static_cast<int64_t>((tile / num_m) % S) * a.M + row) * a.N;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 32, r);
          tc_wait_ld();
          const int col0 = n0 + c * 32;
          if (row < a.M) {
            if (col0 + 32 <= a.N && (a.N % 4) == 0) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                reinterpret_cast<uint4*>(prow + col0)[v] = make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
            } else {
              for (int j = 0; j < 32; ++j)
                if (col0 + j < a.N) prow[col0 + j] = __uint_as_float(r[j]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        continue;
      }
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
  static int counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!counts[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    counts[dev] = n;
  }
  return counts[dev];
}

namespace {

__global__ void lora_finalize_kernel(const float4* __restrict__ partial, int splits, const float* __restrict__ s,
                                     uint2* __restrict__ T, int M, int R4) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // one float4 of T per thread
  if (i >= M * R4) return;
  const int m = i / R4;
  float4 acc = partial[i];
  for (int k = 1; k < splits; ++k) {
    const float4 p = partial[static_cast<int64_t>(k) * M * R4 + i];
    acc.x += p.x;
    acc.y += p.y;
    acc.z += p.z;
    acc.w += p.w;
  }
  const float sc = s ? s[m] : 1.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x / sc, acc.y / sc);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z / sc, acc.w / sc);
  T[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
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
  const int ntiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN) * a.splits;
  const int grid = ntiles < sm_count() ? ntiles : sm_count();
  k<<<grid, C::THREADS, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lora_finalize(const float* partial, int splits, const float* s, void* T, int M, int R,
                                 cudaStream_t st) {
  const int n = M * (R / 4);
  lora_finalize_kernel<<<(n + 255) / 256, 256, 0, st>>>(reinterpret_cast<const float4*>(partial), splits, s,
                                                       static_cast<uint2*>(T), M, R / 4);
  return cudaGetLastError();
}

cudaError_t launch_gemm(int kind, const GemmArgs& a, cudaStream_t st) {
  if (a.splits < 1 || (a.splits > 1 && (!a.partial || kind != 4))) return cudaErrorInvalidValue;
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
