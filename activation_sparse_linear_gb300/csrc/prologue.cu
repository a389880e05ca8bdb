// Fused first half of the RT-Lynx linear layer: one pass over X produces
//   - the 2:4 compressed activations and their metadata ("RT-Lynx" page,
//     Method: top-2-of-4 activation selection, online, in the sparse tensor
//     core's own format),
//   - the row scale s = ||X||_2 / ||X~||_2 (Code examples, first formula),
//   - T' = (X LB^T) / s, the LoRA down-projection (CUDA kernel optimisation:
//     the low-rank branch is computed from the same X tile).
//
// CTA (rb, sp) handles rows 128 rb .. 128 rb + 127 and the sp-th share of the
// 128-channel blocks.  Per 64-channel stage, TMA brings the X tile (128 x 64,
// 128-byte swizzle) and, with the LoRA branch, the LB tile (64 x 64) into a
// ring of shared-memory stages.  One thread issues four tcgen05.mma
// (M = 128, N = 64, K = 16) per stage into a 64-column TMEM accumulator, while
// sixteen selection warps (four threads per row, 16 channels each) read the same
// X tile, keep the top two of every four channels, and store the kept values
// (16 bytes per thread and stage) and the metadata words (32 bits per thread
// and 128-channel block) straight to global memory.  Rows of X are therefore
// read from HBM once for both branches.
//
// The channel blocks of a row block are split over a cluster of `split` CTAs
// so that the grid covers the GPU.  Each row has an owner CTA in the cluster;
// every CTA stores its fp32 shares of a row (x^2, kept x^2, and its share of
// X LB^T) straight into the owner's shared memory (distributed shared memory,
// one slot per sending CTA), and after one cluster barrier the owner adds the
// slots of its rows in rank order and writes s and T'.  With split = 1 the CTA
// writes s and T' itself.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kernels.h"
#include "select.cuh"

namespace lynx {
namespace {

constexpr int P_ROWS = 128;                       // rows per CTA = TMEM lanes
constexpr int P_NST = 7;                          // pipeline stages
constexpr int P_WORKERS = 16;                     // selection warps: four threads per row
constexpr int P_TPR = 32 * P_WORKERS / 128;       // threads per row (16 of each stage's 64 channels each)
constexpr int P_DRAIN0 = 2 + P_WORKERS;           // warps 18, 19: with warps 0 and 1, the T drain in cluster mode
constexpr int P_THREADS = 64 + 32 * P_WORKERS + 64;  // warp 0 TMA, warp 1 MMA, warps 2..17 selection, 18..19 drain
static_assert(P_DRAIN0 % 4 == 2, "warps 0, 1, 18, 19 cover the four TMEM lane quarters");
static_assert(P_TPR == 4, "the selection code below assumes four threads per row");
constexpr int P_XT = P_ROWS * 128;                // X tile: 128 rows x 64 channels (16 KiB)
constexpr int P_LBT = kRankLB * 128;              // LB tile: 64 ranks x 64 channels (8 KiB)
constexpr int P_STAGE = P_XT + P_LBT;
constexpr int P_SMALL = 2048;                     // barriers, s of the rows, norm shares of the rows
constexpr int P_TSTRIDE = 68;                     // floats per row of a T' share (272 B: conflict-free rows)
// Receive slots of the cluster reduction: split x ceil(128 / split) rows (at most 143 for split <= 16), each an
// X LB^T share row and a (x^2, kept x^2) pair.
constexpr int P_RECV_ROWS = 144;
constexpr int P_RECV = P_RECV_ROWS * (P_TSTRIDE * 4 + 8);
constexpr int P_SMEM = P_NST * P_STAGE + P_SMALL + P_RECV + 1024;  // + alignment
static_assert(P_RECV_ROWS >= P_ROWS + kMaxPrologueSplit - 1, "receive slots for every cluster size");
static_assert(P_SMEM <= 232448, "shared memory budget");

__constant__ SelectTable c_select_table = make_select_table();

enum Site : int { SITE_P_PRODUCER = 21, SITE_P_MMA = 22, SITE_P_WORKER = 23, SITE_P_ACC = 24 };

__device__ __forceinline__ void named_sync_workers() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * P_WORKERS) : "memory");
}

template <bool LORA>
__global__ void __launch_bounds__(P_THREADS, 1) prologue_kernel(const __grid_constant__ ProArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_NST * P_STAGE);
  uint64_t* empty = full + P_NST;
  uint64_t* acc_full = empty + P_NST;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_full + 1);
  float* s_sh = reinterpret_cast<float*>(tslot + 4);  // direct mode: s of the CTA's rows (128 floats)
  uint32_t* sel_table = reinterpret_cast<uint32_t*>(s_sh + 3 * P_ROWS);  // the top-2-of-4 decision table
  float* recv_t = reinterpret_cast<float*>(smem + P_NST * P_STAGE + P_SMALL);  // cluster mode: T shares received
  float2* recv_n = reinterpret_cast<float2*>(recv_t + P_RECV_ROWS * P_TSTRIDE);  // ... and norm shares
  static_assert(8 * (2 * P_NST + 1) + 16 + 12 * P_ROWS + 64 * 4 <= P_SMALL, "small-state area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = blockIdx.x / a.split, sp = blockIdx.x % a.split;
  const int r0 = rb * P_ROWS;
  const int kb0 = static_cast<int>(static_cast<int64_t>(sp) * a.nkb / a.split);
  const int kb1 = static_cast<int>(static_cast<int64_t>(sp + 1) * a.nkb / a.split);
  const int nstages = 2 * (kb1 - kb0);  // >= 2: the host keeps split <= nkb

  if (threadIdx.x == 0) {
    for (int i = 0; i < P_NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], P_WORKERS + (LORA ? 1 : 0));
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 64) sel_table[threadIdx.x] = c_select_table.e[threadIdx.x];
  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmX);
    if (LORA) prefetch_tmap(&a.tmLB);
  }
  if (LORA && warp == 1) {
    tmem_alloc(tslot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = LORA ? *tslot : 0u;
  // Cluster mode: each row has an owner CTA, rows [ceil(128 j / split), ceil(128 (j + 1) / split)) for rank j; a
  // share sent by rank p lands in the owner's slot p * rmax + (row - first row of the owner).  The barrier phase
  // opened here tells every thread, before its first store into a peer, that all CTAs of the cluster have started.
  const int rmax = (P_ROWS + a.split - 1) / a.split;
  auto owner_slot = [&](int r, int& o) {
    o = r * a.split / P_ROWS;
    return sp * rmax + r - (P_ROWS * o + a.split - 1) / a.split;
  };
  // Cluster mode: warp w of {0, 1, 18, 19} reads TMEM lane quarter w % 4 of X LB^T as soon as the last MMA has
  // completed and stores its rows' shares into the owners' slots, while the selection warps still work on the
  // last channel block; the CTA's start-up barrier phase is waited for first (every CTA of the cluster started).
  auto push_t_shares = [&](bool ok) {
    const int q = warp & 3;
    bool got = ok && mbar_wait(acc_full, 0, a.ctl, SITE_P_ACC);
    got = __all_sync(0xFFFFFFFFu, got);
    cluster_wait();
    if (!got) return;
    tc_fence_after();
    uint32_t t0[32], t1[32];
    tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16), t0);
    tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + 32, t1);
    tc_wait_ld();
    int o;
    const int slot = owner_slot(q * 32 + lane, o);  // 272-byte rows
    const uint32_t dst = mapa_shared(recv_t + slot * P_TSTRIDE, o);
#pragma unroll
    for (int v4 = 0; v4 < 16; ++v4) {
      const uint32_t* src = v4 < 8 ? t0 + 4 * v4 : t1 + 4 * (v4 - 8);
      st_cluster_f32x4(dst + 16 * v4, make_float4(__uint_as_float(src[0]), __uint_as_float(src[1]),
                                                  __uint_as_float(src[2]), __uint_as_float(src[3])));
    }
  };
  const bool drain_warp = LORA && a.split > 1 && (warp < 2 || warp >= P_DRAIN0);
  if (a.split > 1) cluster_arrive_relaxed();
  // The set-up above may overlap the previous kernel; nothing below touches global memory before it is done.
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0)  // the arrival counters of the split-K GEMM that follows start at zero
    for (int i = threadIdx.x; i < a.nzero; i += P_THREADS) a.zero[i] = 0u;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------------- TMA producer
      int it = 0;
      for (; it < nstages; ++it) {
        const int st = it % P_NST;
        if (!mbar_wait(&empty[st], ((it / P_NST) & 1) ^ 1, a.ctl, SITE_P_PRODUCER)) break;
        // the first loads go out three at a time: stage it waits for stage it - 3, so that each CTA's first
        // tiles are not queued behind every CTA's whole ring (about 3% per launch)
        if (it >= 3 && it < P_NST && !mbar_wait(&full[it - 3], 0, a.ctl, SITE_P_PRODUCER)) break;
        uint8_t* sx = smem + st * P_STAGE;
        const int ch = kb0 * kMetaBlockCols + it * 64;
        if (!(a.ctl.inject == 1 && it == 0)) {  // test hook: the first stage never arrives
          mbar_arrive_expect_tx(&full[st], P_XT + (LORA ? P_LBT : 0));
          tma_load_2d(sx, &a.tmX, &full[st], ch, r0);
          if (LORA) tma_load_2d(sx + P_XT, &a.tmLB, &full[st], ch, 0);
        }
      }
      // Every load issued must land before the CTA exits (after a timeout the consumers stop early).
      // A slot holds at most one outstanding load: the last one issued into it, phase n - 1.
      for (int st = 0; st < P_NST; ++st) {
        int n = it > st ? (it - st + P_NST - 1) / P_NST : 0;
        if (a.ctl.inject == 1 && st == 0 && n > 0) --n;  // stage 0 was never loaded
        if (n > 0) mbar_wait(&full[st], (n - 1) & 1, a.ctl, SITE_P_PRODUCER);
      }
    }
    __syncwarp();
    if (drain_warp) push_t_shares(true);
  } else if (warp == 1) {
    if (LORA && lane == 0) {
      // -------------------------------------------------------------- MMA issuer: T += X_tile LB_tile^T
      constexpr uint32_t IDESC = idesc_bf16(P_ROWS, kRankLB, false);
      constexpr uint64_t STEP = P_STAGE >> 4;
      const uint64_t a0 = sdesc(smem_u32(smem), 16, 1024, SWZ_128B);
      const uint64_t b0 = sdesc(smem_u32(smem) + P_XT, 16, 1024, SWZ_128B);
      bool ok = true;
      for (int it = 0; it < nstages && ok; ++it) {
        const int st = it % P_NST;
        ok = mbar_wait(&full[st], (it / P_NST) & 1, a.ctl, SITE_P_MMA);
        if (!ok) break;
        tc_fence_after();
        const uint64_t ad = a0 + st * STEP, bd = b0 + st * STEP;
        tc_mma(tmem, ad, bd, IDESC, it != 0);
        tc_mma(tmem, ad + 2, bd + 2, IDESC, 1);
        tc_mma(tmem, ad + 4, bd + 4, IDESC, 1);
        tc_mma(tmem, ad + 6, bd + 6, IDESC, 1);
        tc_commit(&empty[st]);
      }
      tc_commit(acc_full);  // fires once every MMA issued above has completed
      mbar_wait(acc_full, 0, a.ctl, SITE_P_ACC);  // no MMA may still run when TMEM is released
    }
    __syncwarp();
    if (drain_warp) push_t_shares(true);
  } else if (warp >= P_DRAIN0) {
    if (drain_warp) push_t_shares(true);
  } else {
    // ---------------------------------------------------------------- selection warps
    // Warp sw (0..15) takes rows base + i and base + 8 + i (i = 0..3, base = 16 (sw / 2) + 4 (sw % 2)), four
    // neighbouring lanes per row (16 of each stage's 64 channels each).  Rows r and r + 8 of a 16-row group
    // share the tensor-memory lanes of their metadata (low and high 16-bit halves of a word), so both halves
    // of every word are computed inside one warp and one lane stores the whole word.
    const int sw = warp - 2;
    const int qq = lane & 3, hsel = lane >> 4;
    const int r = 16 * (sw >> 1) + 4 * (sw & 1) + 8 * hsel + ((lane >> 2) & 3);
    const int row = r0 + r;
    const bool row_live = row < a.M;
    // this thread's 16-bit metadata half: groups 4 (qq & 1) .. +3 of a 32-channel word, in TMEM lane mlane;
    // lane hsel of the pair (lane, lane ^ 16) stores word 2 hsel + qq / 2 of that lane (4 words of 16 bytes)
    const int mlane = (r / 16) * 16 + (qq & 1) * 8 + (r % 8);
    const int64_t blocks_k = meta_blocks_k(a.K);
    uint8_t* mword = a.meta + static_cast<int64_t>(rb) * blocks_k * kMetaChunkBytes + mlane * 16 + hsel * 8 +
                     (qq >> 1) * 4;
    uint16_t* vrow = a.vals + static_cast<int64_t>(row_live ? row : 0) * (a.K / 2);
    float sx = 0.f, skept = 0.f;  // running sums of x^2 and kept x^2 (terms added in channel order)
    bool ok = true;
    // one 128-channel block (two stages) per iteration: eight groups per thread
    for (int kbl = 0; kbl < nstages / 2; ++kbl) {
      uint4 v[4];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int it = 2 * kbl + sub, st = it % P_NST;
        ok = mbar_wait(&full[st], (it / P_NST) & 1, a.ctl, SITE_P_WORKER);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        const uint8_t* xrow = smem + st * P_STAGE + r * 128;
        v[2 * sub] = *reinterpret_cast<const uint4*>(xrow + (((2 * qq) ^ (r & 7)) << 4));
        v[2 * sub + 1] = *reinterpret_cast<const uint4*>(xrow + (((2 * qq + 1) ^ (r & 7)) << 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp no longer reads the stage
      }
      if (!ok) break;
      uint32_t k[8], half[2];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {  // groups in channel order: both sums see their terms in that order
        const uint4 u0 = v[2 * sub], u1 = v[2 * sub + 1];
        const uint32_t n0 = select_group(u0.x, u0.y, sel_table, k[4 * sub], sx, skept);
        const uint32_t n1 = select_group(u0.z, u0.w, sel_table, k[4 * sub + 1], sx, skept);
        const uint32_t n2 = select_group(u1.x, u1.y, sel_table, k[4 * sub + 2], sx, skept);
        const uint32_t n3 = select_group(u1.z, u1.w, sel_table, k[4 * sub + 3], sx, skept);
        half[sub] = n0 | (n1 << 4) | (n2 << 8) | (n3 << 12);
      }
      const int kb = kb0 + kbl;
      if (row_live) {
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {  // the 8 kept values of this thread's 16 channels: 16 bytes
          const int ch = kb * kMetaBlockCols + sub * 64 + 16 * qq;
          if (ch < a.K)
            *reinterpret_cast<uint4*>(vrow + ch / 2) = make_uint4(k[4 * sub], k[4 * sub + 1], k[4 * sub + 2], k[4 * sub + 3]);
        }
      }
      const uint32_t p0 = __shfl_xor_sync(0xFFFFFFFFu, half[0], 16);  // the partner row's halves
      const uint32_t p1 = __shfl_xor_sync(0xFFFFFFFFu, half[1], 16);
      const uint32_t word = hsel == 0 ? (half[0] | (p0 << 16)) : (p1 | (half[1] << 16));
      *reinterpret_cast<uint32_t*>(mword + static_cast<int64_t>(kb) * kMetaChunkBytes) = word;
    }
    // row sums: the four threads of a row are neighbouring lanes
    sx += __shfl_xor_sync(0xFFFFFFFFu, sx, 1);
    skept += __shfl_xor_sync(0xFFFFFFFFu, skept, 1);
    sx += __shfl_xor_sync(0xFFFFFFFFu, sx, 2);
    skept += __shfl_xor_sync(0xFFFFFFFFu, skept, 2);
    if (a.split > 1) cluster_wait();  // every CTA of the cluster has started
    if (qq == 0) {
      if (a.split == 1) {
        const float sv = skept > 0.f ? sqrtf(sx / skept) : 1.f;
        s_sh[r] = sv;
        if (row < a.M) a.s[row] = sv;
      } else {  // this CTA's norm shares of row r, into the owner's slot
        int o;
        const int slot = owner_slot(r, o);
        st_cluster_f32x2(mapa_shared(&recv_n[slot], o), make_float2(sx, skept));
      }
    }
    if (LORA && a.split == 1) {
      named_sync_workers();  // s_sh complete
      if (warp < 6) {
        // TMEM lane quarter q = warp % 4 holds rows 32 q .. 32 q + 31
        const int q = warp & 3;
        bool got = ok && mbar_wait(acc_full, 0, a.ctl, SITE_P_ACC);
        got = __all_sync(0xFFFFFFFFu, got);
        if (got) {
          tc_fence_after();
          uint32_t t0[32], t1[32];
          tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16), t0);
          tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + 32, t1);
          tc_wait_ld();
          const int trow = q * 32 + lane, grow = r0 + trow;
          if (grow < a.M) {
            const float inv = 1.f / s_sh[trow];  // T' = T * (1 / s): one division per row
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.T) + static_cast<int64_t>(grow) * kRankLB);
#pragma unroll
            for (int v8 = 0; v8 < 8; ++v8) {
              const uint32_t* src = v8 < 4 ? t0 + 8 * v8 : t1 + 8 * (v8 - 4);
              uint32_t pk[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(src[2 * j]) * inv,
                                                          __uint_as_float(src[2 * j + 1]) * inv);
                pk[j] = *reinterpret_cast<uint32_t*>(&b2);
              }
              dst[v8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      }
    }
  }
  // the start-up phase for the warps that have not waited for it above
  if (a.split > 1 && (warp < 2 || warp >= P_DRAIN0) && !drain_warp) cluster_wait();
  tc_fence_before();
  __syncthreads();
  if (a.split > 1) {
    // ---------------------------------------------------------------- cluster reduction of the shares
    // The owner of rows [row_lo, row_hi) adds the slots of the split CTAs in rank order (deterministic) and
    // writes s and T'.  Only local shared memory is read: after the barrier no CTA touches a peer, so no CTA
    // has to wait for the others before it leaves.
    cluster_sync();  // every share is in its owner's shared memory
    const int row_lo = (P_ROWS * sp + a.split - 1) / a.split;
    const int rows = (P_ROWS * (sp + 1) + a.split - 1) / a.split - row_lo;
    if (threadIdx.x < rows) {  // s of the row
      const int rr = row_lo + threadIdx.x, grow = r0 + rr;
      float sxs = 0.f, sks = 0.f;
      for (int p = 0; p < a.split; ++p) {
        const float2 n2 = recv_n[p * rmax + threadIdx.x];
        sxs += n2.x;
        sks += n2.y;
      }
      const float sv = sks > 0.f ? sqrtf(sxs / sks) : 1.f;
      s_sh[rr] = sv;
      if (grow < a.M) a.s[grow] = sv;
    }
    if (LORA) {
      __syncthreads();  // s of the CTA's rows in s_sh
      // T' in items of 4 ranks: 16 per row
      for (int i = threadIdx.x; i < rows * 16; i += P_THREADS) {
        const int rl = i / 16, g = i % 16, rr = row_lo + rl, grow = r0 + rr;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < a.split; ++p) {
          const float4 t4 = *reinterpret_cast<const float4*>(recv_t + (p * rmax + rl) * P_TSTRIDE + 4 * g);
          acc.x += t4.x;
          acc.y += t4.y;
          acc.z += t4.z;
          acc.w += t4.w;
        }
        if (grow < a.M) {
          const float inv = 1.f / s_sh[rr];  // T' = T * (1 / s): one division per row
          __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
          reinterpret_cast<uint2*>(a.T)[static_cast<int64_t>(grow) * (kRankLB / 4) + g] =
              make_uint2(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1));
        }
      }
    }
  }
  if (LORA && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// Kernel attributes, once per device: the dynamic shared memory and, for clusters of 16 CTAs (beyond the
// portable 8), the non-portable cluster size.
cudaError_t set_prologue_attrs() {
  static std::atomic<bool> done[64] = {};  // setting the attributes twice from racing threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  for (auto* k : {prologue_kernel<true>, prologue_kernel<false>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  done[dev] = true;
  return cudaSuccess;
}

}  // namespace

// CTAs per row block: among the cluster sizes (2 .. kMaxPrologueSplit, at most one per channel block) whose
// clusters all fit on the GPU at once and whose grid does not exceed the SM count, the smallest one that gives
// the fewest channel blocks per CTA; 1 when none fits.  Cluster sizes above 8 are non-portable: the GPU
// reports how many of them it holds (a 16-CTA cluster needs 16 SMs of one GPC).
int prologue_split(int M, int K) {
  const int row_blocks = static_cast<int>(round_up(M, kMetaRowPad) / P_ROWS);
  const int nkb = static_cast<int>(meta_blocks_k(K));
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (set_prologue_attrs() != cudaSuccess) return 1;
  static std::atomic<int> fit[64][kMaxPrologueSplit + 1] = {};  // resident clusters per size and device (-1: none)
  int best = 1, best_per = nkb;
  for (int split = 2; split <= kMaxPrologueSplit && split <= nkb; ++split) {
    if (row_blocks * split > sm_count()) break;
    if (!fit[dev][split]) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = split;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(split);
      cfg.blockDim = dim3(P_THREADS);
      cfg.dynamicSmemBytes = P_SMEM;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, prologue_kernel<true>, &cfg) != cudaSuccess) {
        cudaGetLastError();  // an unsupported cluster size is an answer, not an error to keep
        n = 0;
      }
      fit[dev][split] = n > 0 ? n : -1;
    }
    const int per = (nkb + split - 1) / split;
    if (fit[dev][split] >= row_blocks && per < best_per) {
      best = split;
      best_per = per;
    }
  }
  return best;
}

cudaError_t launch_prologue(const ProArgs& args, bool lora, cudaStream_t st) {
  auto* k = lora ? prologue_kernel<true> : prologue_kernel<false>;
  if (cudaError_t e = set_prologue_attrs()) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = args.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the previous kernel ends
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((args.M_pad / P_ROWS) * args.split);
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, args);
}

}  // namespace lynx
