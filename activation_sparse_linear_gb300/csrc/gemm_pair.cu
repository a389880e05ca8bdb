// CTA-pair (cta_group::2) tcgen05 GEMM for the RT-Lynx linear layer:
//   Y = rowscale o (A_op . W^T) [+ T' . LA^T]
//
// Two CTAs of a cluster share one output tile of 256 * MB rows x TN columns.
// CTA r of the pair owns MB blocks of 128 rows (its TMEM holds MB fp32
// accumulators of 128 x TN) and stages, per step, its own rows of A and its
// half (TN/2 rows) of the W tile; each tcgen05.mma.cta_group::2 issued by the
// leader CTA (rank 0) multiplies 256 rows (row block h of both CTAs) by all TN
// columns, reading A and W from both CTAs' shared memory.
//
// The shape is set by the bytes each SM must pull into shared memory per
// multiply-add, which bounds this kernel: per 128-channel step a CTA stages
// MB x 16 KiB of compressed A, TN/2 x 256 B of W and MB x 2 KiB of metadata.
// The sparse path takes MB = 2 with TN = 224 (64 KiB per 7.3 M logical MACs;
// the two accumulators and the metadata ring fill 480 of the 512 TMEM
// columns) or TN = 192 (60 KiB per 6.3 M), or MB = 1, TN = 256 (50 KiB per
// 4.2 M) for few row tiles.  The dense path takes MB = 1 with TN = 256, or
// TN = 448 issued as two 224-column MMAs that read A once through the tensor
// core's A collector (44 KiB per 64-channel step for 3.7 M MACs).
//
// Sparse A (compressed values, 128-byte swizzle) goes through
// tcgen05.mma.sp.cta_group::2 in steps of 128 channels: every stage carries
// each CTA's 2 KiB metadata chunk per row block, which the leader copies into
// both TMEMs with tcgen05.cp.cta_group::2 (each CTA's own shared memory into
// its own TMEM); MMA j of a chunk reads the even column pair (j & 2) with the
// sparsity selector j & 1.
//
// The LoRA-up branch ("RT-Lynx" page, CUDA kernel optimisation: Yr is produced
// on chip and accumulated into Ys) is one extra stage: A = T' (128 x 64 per row
// block), B = this CTA's half of LA; four dense MMAs per row block into the
// same accumulators.  Because the epilogue multiplies the tile by s, T' holds
// (X LB^T)/s.
//
// Roles per CTA: warp 0 TMA producer (both CTAs), warp 1 MMA issuer (leader
// only; with two row blocks warp 10 issues the second block's MMAs); the whole
// warp runs each of these loops and one lane, picked by elect.sync, issues each
// instruction.  Warps 2-9 epilogue (two warps per TMEM lane quarter:
// TMEM -> registers -> scale -> bf16 -> shared staging -> TMA store).  The
// operand ring is as deep as shared memory allows: three stages for the
// 512-row tiles, six for the dense 256 x 256 tile, four for the sparse
// 256 x 256 and the dense 256 x 448 tiles.
// Every mbarrier wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kernels.h"
#include "select.cuh"

namespace lynx {
namespace {

__constant__ SelectTable c_pair_select_table = make_select_table();

__device__ __forceinline__ float tanh_approx(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
  return t;
}
// GELU of the up layer's output, x Phi(x), in the tanh form of Hendrycks and Gimpel ("Gaussian Error Linear
// Units", 2016): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), with the hardware tanh approximation.  Its
// distance from the error-function form is below 1e-3 |x| + 1e-3, under a tenth of a bf16 unit for the
// values that matter, and it costs a handful of instructions instead of an erf evaluation.
__device__ __forceinline__ float gelu_f(float x) {
  const float u = x * fmaf(0.0356774081f, x * x, 0.7978845608f);  // sqrt(2/pi) (x + 0.044715 x^3)
  const float hx = 0.5f * x;
  return fmaf(hx, tanh_approx(u), hx);
}

constexpr int BLOCK = 128;         // rows per TMEM accumulator (one row per lane)
constexpr int kPairMaxSplit = 4;   // k-splits per tile at most (the host's choice and test hook stay within it)
constexpr int kDenseBK = 64;       // channels per stage of the dense path (64 or 128: one or two 64-channel boxes)
constexpr int META_RING = 4;       // TMEM metadata stages
constexpr int META_GROUP_COLS = 4;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int MMA_WARP2 = 2 + EPI_WARPS;         // second MMA issuer (two row blocks per CTA)
constexpr int THREADS = 96 + 32 * EPI_WARPS;
constexpr int SMEM_LIMIT = 232448;
constexpr int Y_BOX = 32;                          // output staging box: 32 rows x 32 columns bf16 (64-byte rows)
constexpr int Y_BUF = Y_BOX * Y_BOX * 2;

enum Site : int { SITE_PRODUCER = 11, SITE_MMA = 12, SITE_EPILOGUE = 13, SITE_DRAIN = 14 };

// Per stage and CTA: sparse = 128 channels (A: 64 kept values per row, 128-byte rows, per row block; W: two
// 64-channel sub-tiles; one metadata chunk per row block) feeding four tcgen05.mma.sp per row block;
// dense = 64 channels feeding four tcgen05.mma per row block.  Several MMAs per barrier round keep the
// issuing warp ahead of the tensor pipe.
// F1 (sparse, one row block): the stage carries the dense X tile (two 64-channel boxes per row block) instead of
// compressed values; the epilogue warps select in registers and write the compressed values over box 0 and the
// metadata chunk into the stage before the MMAs read them.
// WIDE (dense, one row block, TN = 448): a tile is two 224-column halves, one MMA each per K = 16 step, and the
// two MMAs share one shared-memory read of the X tile through the tensor core's A collector (fill, then last
// use): per 64 channels an SM moves 88 KB through shared memory for 3.7 M MACs (24 bytes per thousand MACs)
// instead of 64 KB for 2.1 M (31); a LoRA stage per half.
template <bool SPARSE, int MB, int TN, bool F1 = false>
struct PairCfg {
  static constexpr int ROWS = MB * BLOCK;    // rows per CTA
  static constexpr int HALF_N = TN / 2;      // W rows staged per CTA
  static constexpr bool WIDE = TN > 256;
  static constexpr int NH = WIDE ? 2 : 1;    // MMA column halves per tile
  static constexpr int MN = TN / NH;         // MMA N
  static constexpr int QN = MN / 2;          // W rows per CTA and MMA half
  static constexpr int BK = SPARSE ? 128 : kDenseBK;
  static constexpr int BOXES = SPARSE ? (F1 ? 2 : 1) : kDenseBK / 64;  // 64-channel (128-byte) A boxes per row block and stage
  static constexpr int A_BOX = BLOCK * 128;
  static constexpr int A_BLOCK = BOXES * A_BOX;
  static constexpr int A_SLOT = MB * A_BLOCK;
  static constexpr int SUB = HALF_N * 128;   // one 64-channel W sub-tile of this CTA (WIDE: both halves' rows)
  static constexpr int B_SLOT = SPARSE ? 2 * SUB : BOXES * SUB;
  static constexpr int M_SLOT = SPARSE ? MB * kMetaChunkBytes : 0;
  static constexpr int LORA_LOAD = MB * A_BOX + (WIDE ? QN * 128 : SUB);  // T' and this CTA's LA rows (WIDE: one half's)
  static constexpr int STAGE = A_SLOT + B_SLOT + M_SLOT;
  static constexpr int LOAD_BYTES = F1 ? A_SLOT + B_SLOT : STAGE;  // TMA bytes of a k-step per CTA
  // Output staging boxes per epilogue warp: two, so that a box is refilled while the other is stored; one
  // for the sparse 256 x 256 tile, whose short 128-channel steps need a fourth operand stage in its place
  // (its few row tiles share each W tile between few CTA pairs, so its loads often come from DRAM).
  static constexpr int Y_BOXES = (SPARSE && MB == 1) ? 1 : 2;
  static constexpr int Y_STAGING = EPI_WARPS * Y_BOXES * Y_BUF;
  static constexpr int NST_FIT = (SMEM_LIMIT - 1280 - Y_STAGING) / STAGE;
  static constexpr int NST = (SPARSE && NST_FIT > META_RING) ? META_RING : NST_FIT;
  static constexpr int SMEM = NST * STAGE + Y_STAGING + 256 + 1024;
  // Accumulator buffers: two where they fit in TMEM next to the metadata ring (the dense 256 x 256 tile, the sparse
  // 256 x 192 tile), so that the MMAs of the next tile run into one while the epilogue drains the other.
  static constexpr int META_COLS = SPARSE ? META_RING * MB * META_GROUP_COLS : 0;
  static constexpr int ACC_BUFS = (2 * MB * TN + META_COLS <= TMEM_COLS) ? 2 : 1;
  static constexpr int ACC_STRIDE = MB * TN;  // TMEM columns per accumulator buffer
  static constexpr int META_COL = ACC_BUFS * ACC_STRIDE;  // first metadata column (after the accumulators)
  static_assert(STAGE % 1024 == 0, "stage slots keep 1 KiB alignment");
  static_assert(NST >= 2 && SMEM <= SMEM_LIMIT, "shared memory budget");
  static_assert(TN % 32 == 0 && MN <= 256 && QN % 8 == 0 && (!WIDE || (!SPARSE && MB == 1 && BOXES == 1)), "MMA N");
  static_assert(LORA_LOAD <= STAGE, "a LoRA stage fits a stage slot");
  static_assert(META_COL + META_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(ACC_BUFS * ACC_STRIDE <= TMEM_COLS, "TMEM budget of the accumulator buffers");
  static_assert(8 * (2 * NST + 2 * ACC_BUFS + 3 + (F1 ? 2 * NST + 1 : 0)) + 32 <= 256, "barrier area");
  static_assert(!F1 || (SPARSE && MB == 1), "in-GEMM selection: sparse, one row block");
  static_assert(!SPARSE || NST <= META_RING, "a metadata group must outlive the stages in flight");
};

// Stores 32 bf16 columns (16 packed pairs) of one output row starting at column col0, clipped to N.
__device__ __forceinline__ void store_chunk(__nv_bfloat16* yrow, int col0, int N, bool vec_ok, const uint32_t* p) {
  if (vec_ok && col0 + 32 <= N) {
    uint4* dst = reinterpret_cast<uint4*>(yrow + col0);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (col0 + j < N) {
        const uint32_t w = p[j / 2];
        reinterpret_cast<uint16_t*>(yrow)[col0 + j] =
            (j & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFFu);
      }
    }
  }
}

// Transposed output: this lane's accumulator row is output column `zrow`; its 32 bf16 values (16 packed pairs)
// belong to output rows zcol0 .. zcol0 + 31 (clipped to nz, the output's row count).
__device__ __forceinline__ void store_chunk_t(void* Y, int64_t ldy, int zrow, int zcol0, int nz, const uint32_t* p) {
  uint16_t* y = static_cast<uint16_t*>(Y) + zrow;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (zcol0 + j < nz) {
      const uint32_t w = p[j / 2];
      y[static_cast<int64_t>(zcol0 + j) * ldy] = (j & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w & 0xFFFFu);
    }
  }
}

// TRANS: the accumulator tile is the transpose of the output (the weight-sparse variant multiplies the pruned
// W, as the sparse operand, by X); the epilogue writes it transposed.  SPLIT: the k-steps of every tile are split
// over a.splits work units (few tiles for the GPU's CTA pairs); see the epilogue.  GELU: the output is
// bf16(GELU(bf16(y))) and, with a.hvals, the epilogue also sparsifies it for the next layer (the MLP pair's
// up layer feeding its down layer: "RT-Lynx" page, CUDA kernel optimisation, one execution path for the online
// sparsification).
// F1: the GEMM selects the 2:4 pattern itself ("RT-Lynx" page, CUDA kernel optimisation: 2:4 activations built
// directly in registers): the producer loads dense X tiles; the epilogue warps, before draining a tile, take each
// stage's X rows (two threads per row, 64 channels each), keep the top two of every four in registers, write the
// compressed values and the metadata into the stage, add x^2 and kept x^2 over the tile's whole K, and at the
// LoRA stage write T' = bf16(T / s) of their rows (T = X LB^T, unscaled, from a.lora_t) in place of a loaded T'.
// One work unit: k-steps [kbeg, kend) of a tile, part `seg` of the tile's `nseg` parts (in k order).
struct Unit {
  int tile, kbeg, kend, seg, nseg;
};
// The u-th unit of CTA pair `cluster` of `nclusters`; false past the last.  The tile and split schedules deal
// (tile, split) units out round-robin, tile fastest, each tile cut into S equal k-ranges.  Stream-K gives pair c
// the contiguous range [c T / P, (c + 1) T / P) of all T = ntiles nk k-steps (tile-major order, P pairs): a tile
// is cut wherever a pair's range ends, and the pairs that share it leave partials as split units do (at most
// kPairMaxSplit parts; the host enables it only where ntiles >= P / 2 and nk >= 8, which guarantees that).
__device__ __forceinline__ bool unit_at(int u, int cluster, int nclusters, int ntiles, int nk, int S, bool streamk,
                                        Unit& o) {
  if (!streamk) {
    const int unit = cluster + u * nclusters;
    if (unit >= ntiles * S) return false;
    const int ks = unit / ntiles;
    o.tile = unit % ntiles;
    o.kbeg = ks * nk / S;
    o.kend = (ks + 1) * nk / S;
    o.seg = ks;
    o.nseg = S;
    return true;
  }
  const int64_t T = static_cast<int64_t>(ntiles) * nk;
  const int64_t b0 = cluster * T / nclusters, b1 = (cluster + 1) * T / nclusters;
  const int64_t t = b0 / nk + u;
  if (b0 >= b1 || t * nk >= b1) return false;
  // the pair whose range holds k-step s: the last c with c T / P <= s
  auto owner = [&](int64_t st) { return static_cast<int>(((st + 1) * nclusters - 1) / T); };
  o.tile = static_cast<int>(t);
  o.kbeg = static_cast<int>(b0 > t * nk ? b0 - t * nk : 0);
  o.kend = static_cast<int>(b1 < (t + 1) * nk ? b1 - t * nk : nk);
  const int first = owner(t * nk);
  o.seg = cluster - first;
  o.nseg = owner(t * nk + nk - 1) - first + 1;
  return true;
}

template <bool SPARSE, bool LORA, int MB, int TN, bool TRANS, bool SPLIT, bool GELU, bool F1 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ PairArgs a) {
  using C = PairCfg<SPARSE, MB, TN, F1>;
  static_assert(!F1 || (LORA && !TRANS && !SPLIT && !GELU), "in-GEMM selection variant");
  static_assert(!C::WIDE || (!TRANS && !SPLIT), "the 448-column tile: whole tiles, not transposed");
  // With two row blocks, two threads issue the MMAs (one row block each): while one waits on a barrier or
  // does its per-stage bookkeeping, the other's queued MMAs keep the tensor pipe busy.
  constexpr int NISS = MB >= 2 ? 2 : 1;
  static_assert(MB % NISS == 0, "row blocks split evenly between the issuers");
  static_assert(!(GELU && (SPLIT || TRANS)), "the GELU epilogue runs on whole, untransposed tiles");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ystage = smem + C::NST * C::STAGE;  // 1 KiB aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(ystage + C::Y_STAGING);
  uint64_t* empty = full + C::NST;
  uint64_t* acc_full = empty + C::NST;        // [ACC_BUFS]
  uint64_t* acc_empty = acc_full + C::ACC_BUFS;  // [ACC_BUFS]
  uint64_t* drain = acc_empty + C::ACC_BUFS;
  uint64_t* epi_bar = drain + 1;   // split-K: every epilogue warp of this CTA has written its partial
  uint64_t* epi_bar2 = drain + 2;  // split-K: the unit's arrival order is known
  uint64_t* conv_full = drain + 3;          // F1 [NST] (leader): both CTAs' selection of the stage is in place
  uint64_t* xfull = conv_full + C::NST;     // F1 [NST]: this CTA's X tile of the stage has landed
  uint64_t* s_bar = xfull + C::NST;         // F1: every epilogue warp of this CTA has written its rows' s
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 3 + (F1 ? 2 * C::NST + 1 : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* consumed_sh = abort_flag + 1;  // one count per MMA issuer
  volatile int* issued_sh = abort_flag + 3;
  volatile int* last_flag = abort_flag + 4;   // split-K: this CTA reduces the unit's tile
  uint32_t* sel_table = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(full) + 256);  // GELU, F1: 64 entries
  float* s_sh = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);  // F1: s of the CTA's rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int num_mp = (a.M + 2 * C::ROWS - 1) / (2 * C::ROWS);
  const int num_n = (a.N + TN - 1) / TN;
  const int ntiles = num_mp * num_n;
  const int nk = (a.K + C::BK - 1) / C::BK;
  // Work units: (tile, k-split) pairs, tile fastest; split ks covers k-steps [ks nk / S, (ks + 1) nk / S) and
  // the last split also the LoRA stage.  With S > 1 each unit leaves an fp32 partial in global memory and the
  // last unit of a tile to finish adds the S partials in split order (see the epilogue).
  const int S = SPLIT ? a.splits : 1;
  const bool streamk = SPLIT && a.stream_k != 0;  // stream-K: S is the partials' stride, kPairMaxSplit
  const bool krot = SPARSE && MB == 2 && !TRANS && !SPLIT && !F1;  // staggered k order (producer)
  const int64_t blocks_k = meta_blocks_k(a.K);
  const int meta_rowblocks = static_cast<int>(round_up(a.M, kMetaRowPad) / kMetaRows);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NISS);  // one commit per MMA issuer
    }
    for (int b = 0; b < C::ACC_BUFS; ++b) {
      mbar_init(&acc_full[b], NISS);
      mbar_init(&acc_empty[b], 2 * EPI_WARPS);  // every epilogue warp of both CTAs of the pair
    }
    mbar_init(drain, NISS);
    mbar_init(epi_bar, EPI_WARPS);
    mbar_init(epi_bar2, 1);
    if constexpr (F1)
      for (int i = 0; i < C::NST; ++i) {
        mbar_init(&conv_full[i], 2 * EPI_WARPS);  // every epilogue warp of both CTAs
        mbar_init(&xfull[i], 1);                  // this CTA's producer (expect_tx)
      }
    if constexpr (F1) mbar_init(s_bar, EPI_WARPS);
    *abort_flag = 0;
    consumed_sh[0] = 0;
    consumed_sh[1] = 0;
    *issued_sh = 0;
    fence_mbar_init();
  }
  if ((GELU || F1) && threadIdx.x < 64) sel_table[threadIdx.x] = c_pair_select_table.e[threadIdx.x];
  if (threadIdx.x == 32) {
    prefetch_tmap(&a.tmA);
    prefetch_tmap(&a.tmB);
    if (SPARSE && !F1) prefetch_tmap(&a.tmMeta);
    if (LORA) {
      if (!F1) prefetch_tmap(&a.tmT);
      prefetch_tmap(&a.tmLA);
    }
    if (a.y_tma) prefetch_tmap(&a.tmY);
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
  // The set-up above may overlap the previous kernel; nothing below touches global memory before it is done.
  pdl_launch_dependents();
  pdl_wait();
  if (a.zero && blockIdx.x == 0)  // the next kernel's arrival counters start at zero
    for (int i = threadIdx.x; i < a.nzero; i += THREADS) a.zero[i] = 0u;

  if (warp == 0) {
    {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      // The whole warp runs the loop and one elected lane issues each copy (see the warp-wide helpers).
      constexpr uint32_t STAGE_BYTES = C::LOAD_BYTES;
      constexpr uint32_t LORA_BYTES = MB * C::A_BOX + C::SUB;  // T' (one box per row block) and this CTA's LA half
      const uint32_t full_leader0 = mapa_shared(&full[0], 0);  // the leader's full barriers, 8 B apart
      int g = 0, st = 0;
      uint32_t ph = 0;
      bool stop = false;
      Unit un;
      for (int u = 0; !stop && unit_at(u, cluster, nclusters, ntiles, nk, S, streamk, un); ++u) {
        const int tile = un.tile, kbeg = un.kbeg, kend = un.kend;
        const int nst_u = kend - kbeg + ((LORA && kend == nk) ? C::NH : 0);
        const int mp = tile % num_mp, nb = tile / num_mp;
        const int m0 = mp * 2 * C::ROWS + static_cast<int>(rank) * C::ROWS;
        const int n0 = nb * TN + static_cast<int>(rank) * C::HALF_N;
        int meta_row[MB];  // first 1 KiB row of each row block's metadata chunks
#pragma unroll
        for (int h = 0; h < MB; ++h) {
          int rb = m0 / BLOCK + h;
          if (rb >= meta_rowblocks) rb = meta_rowblocks - 1;  // rows past the padded M: never stored
          meta_row[h] = static_cast<int>(2 * (rb * blocks_k));
        }
        // Staggered k order: the pairs that share a W column tile (same nb) or a row tile (same mp) would
        // otherwise load the same slice at the same moment and all wait for one DRAM fetch.  Pair (mp, nb) starts
        // at offset (mp + nb) mod G of G = min(8, row tiles) steps spread over at most 24 k-steps, so one pair's
        // load brings each slice into L2 for the others; the window bounds how long a slice has to stay there.
        // Measured on the sparse two-row-block tiles (QKV and MLP up -3 to -5%, MLP down -2%, M = 16384 -3%);
        // the one-row-block tiles measured slower and keep the plain order.
        const int nk_u = kend - kbeg, G = num_mp < 8 ? num_mp : 8;
        const int rot = krot ? (((mp + nb) % G) * (nk_u < 24 ? nk_u : 24)) / G : 0;
        for (int it = 0; it < nst_u; ++it) {
          const int kk = it < nk_u ? kbeg + (it + rot) % nk_u : kbeg + it;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ph ^ 1, a.ctl, SITE_PRODUCER)) || *abort_flag) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* sA = smem + st * C::STAGE;
          uint8_t* sB = sA + C::A_SLOT;
          const uint32_t fb = full_leader0 + 8 * st;
          if (!(a.ctl.inject == 1 && g == 0)) {  // test hook: the first stage never arrives
            if constexpr (C::WIDE) {
              // the CTA's X rows and its rows of both column halves of W; a LoRA stage per half: T' and the
              // CTA's rows of that half of LA
              const int nw0 = nb * TN + static_cast<int>(rank) * C::QN;
              if (kk < kend) {
                if (leader) mbar_arrive_expect_tx_w(&full[st], 2 * (C::A_SLOT + C::B_SLOT));
                tma_load_2d_pair_w(sA, &a.tmA, fb, kk * C::BK, m0);
                tma_load_2d_pair_w(sB, &a.tmB, fb, kk * C::BK, nw0);
                tma_load_2d_pair_w(sB + C::QN * 128, &a.tmB, fb, kk * C::BK, nw0 + C::MN);
              } else {
                if (leader) mbar_arrive_expect_tx_w(&full[st], 2 * C::LORA_LOAD);
                tma_load_2d_pair_w(sA, &a.tmT, fb, 0, m0);
                tma_load_2d_pair_w(sA + C::A_BOX, &a.tmLA, fb, 0, nw0 + (kk - kend) * C::MN);
              }
            } else if (kk < kend) {
              if constexpr (F1) {  // X (dense, two boxes per row block) lands on this CTA's own barrier
                if (leader) mbar_arrive_expect_tx_w(&full[st], 2 * C::B_SLOT);
                mbar_arrive_expect_tx_w(&xfull[st], C::A_SLOT);
#pragma unroll
                for (int h = 0; h < MB; ++h)
#pragma unroll
                  for (int j = 0; j < C::BOXES; ++j)
                    tma_load_2d_w(sA + h * C::A_BLOCK + j * C::A_BOX, &a.tmA, &xfull[st], kk * 128 + 64 * j, m0 + h * BLOCK);
              } else {
                if (leader) mbar_arrive_expect_tx_w(&full[st], 2 * STAGE_BYTES);
#pragma unroll
                for (int h = 0; h < MB; ++h)
#pragma unroll
                  for (int j = 0; j < C::BOXES; ++j)  // sparse: 64 kept values per row = 128 channels
                    tma_load_2d_pair_w(sA + h * C::A_BLOCK + j * C::A_BOX, &a.tmA, fb,
                                     kk * (SPARSE ? 64 : C::BK) + 64 * j, m0 + h * BLOCK);
              }
              if constexpr (SPARSE) {
                tma_load_2d_pair_w(sB, &a.tmB, fb, kk * 128, n0);
                tma_load_2d_pair_w(sB + C::SUB, &a.tmB, fb, kk * 128 + 64, n0);
                if constexpr (!F1)
#pragma unroll
                  for (int h = 0; h < MB; ++h)
                    tma_load_2d_pair_w(sB + C::B_SLOT + h * kMetaChunkBytes, &a.tmMeta, fb, 0, meta_row[h] + 2 * kk);
              } else {
#pragma unroll
                for (int j = 0; j < C::BOXES; ++j) tma_load_2d_pair_w(sB + j * C::SUB, &a.tmB, fb, kk * C::BK + 64 * j, n0);
              }
            } else {
              if constexpr (F1) {  // T' comes from the epilogue warps; the stage is free for them to write
                if (leader) mbar_arrive_expect_tx_w(&full[st], 2 * C::SUB);
                mbar_arrive_w(&xfull[st]);
              } else {
                if (leader) mbar_arrive_expect_tx_w(&full[st], 2 * LORA_BYTES);
#pragma unroll
                for (int h = 0; h < MB; ++h) tma_load_2d_pair_w(sA + h * C::A_BLOCK, &a.tmT, fb, 0, m0 + h * BLOCK);
              }
              tma_load_2d_pair_w(sB, &a.tmLA, fb, 0, n0);
            }
          }
          ++g;
          if (++st == C::NST) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (lane == 0) *issued_sh = g;
    }
  } else if (warp == 1 || warp == MMA_WARP2) {
    const int k = warp == 1 ? 0 : 1;  // issuer index: row blocks h = k, k + NISS, ...
    if (leader && k < NISS) {
      // ------------------------------------------------------------ MMA issuers (leader)
      // The whole warp runs the loop and one elected lane issues each tcgen05 instruction.
      // Descriptors and TMEM addresses are built once; each stage only adds offsets, so the issuing
      // thread's work per MMA stays well under the MMA's own duration.
      constexpr uint32_t IDESC = idesc_bf16(2 * BLOCK, TN, false);
      constexpr uint32_t IDESC_SP = idesc_bf16(2 * BLOCK, TN, true);
      constexpr uint64_t STEP = C::STAGE >> 4;    // descriptor start-address units per stage
      constexpr uint64_t ABLK = C::A_BLOCK >> 4;  // ... per row block of A
      constexpr uint64_t ABOX = C::A_BOX >> 4;    // ... per 64-channel box of A
      constexpr uint64_t WSUB = C::SUB >> 4;      // ... per W sub-tile
      constexpr uint64_t MCHUNK = kMetaChunkBytes >> 4;
      const uint32_t s0 = smem_u32(smem);
      const uint64_t a0 = sdesc(s0, 16, 1024, SWZ_128B);
      const uint64_t b0 = sdesc(s0 + C::A_SLOT, 16, 1024, SWZ_128B);
      const uint64_t e0 = sdesc(s0 + C::A_SLOT + C::B_SLOT, 128, 128, SWZ_NONE);
      const uint32_t meta0 = tmem + C::META_COL;
      int g = 0, st = 0, tcount = 0, mring = 0;
      uint32_t ph = 0;
      bool stop = false;
      Unit un;
      for (int u = 0; !stop && unit_at(u, cluster, nclusters, ntiles, nk, S, streamk, un); ++u, ++tcount) {
        const int kbeg = un.kbeg, kend = un.kend;
        const int nst_u = kend - kbeg + ((LORA && kend == nk) ? C::NH : 0);
        const int ab = tcount % C::ACC_BUFS;  // accumulator buffer of this unit
        const uint32_t acc_base = tmem + ab * C::ACC_STRIDE;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&acc_empty[ab], ((tcount / C::ACC_BUFS) & 1) ^ 1, a.ctl, SITE_MMA))) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int it = 0; it < nst_u; ++it) {
          const bool ok = mbar_wait(&full[st], ph, a.ctl, SITE_MMA) &&
                          (!F1 || mbar_wait(&conv_full[st], ph, a.ctl, SITE_MMA));
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a0 + st * STEP, bd = b0 + st * STEP;
          const uint32_t acc0 = it != 0;
          if constexpr (C::WIDE) {
            constexpr uint32_t IDESC_W = idesc_bf16(2 * BLOCK, C::MN, false);
            if (kbeg + it < kend) {
              // four K = 16 steps, each one MMA per column half: the first fills the A collector, the second
              // uses it last
              constexpr uint64_t BH = (C::QN * 128) >> 4;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t accj = (it | j) != 0;
                tc_mma_pair_fill_w(acc_base, ad + 2 * j, bd + 2 * j, IDESC_W, accj);
                tc_mma_pair_lastuse_w(acc_base + C::MN, ad + 2 * j, bd + BH + 2 * j, IDESC_W, accj);
              }
            } else {  // LoRA stage of column half L: T' against that half's LA rows (after T' in the slot)
              const uint32_t d = acc_base + (it - (kend - kbeg)) * C::MN;
              const uint64_t lh = a0 + st * STEP + (C::A_BOX >> 4);
#pragma unroll
              for (int j = 0; j < 4; ++j) tc_mma_pair_w(d, ad + 2 * j, lh + 2 * j, IDESC_W, 1);
            }
          } else if (kbeg + it < kend) {
            if constexpr (SPARSE) {
              // metadata group of this stage: the ring rotates with every k-step this issuer runs
              const uint32_t grp0 = meta0 + (mring++ & (META_RING - 1)) * (MB * META_GROUP_COLS);
#pragma unroll
              for (int hh = 0; hh < MB / NISS; ++hh) {
                const int h = k + hh * NISS;
                tc_cp_pair_128x128b_w(grp0 + h * META_GROUP_COLS, e0 + st * STEP + h * MCHUNK);
              }
#pragma unroll
              for (int hh = 0; hh < MB / NISS; ++hh) {
                const int h = k + hh * NISS;
                // MMA j: A bytes 32j of the 128-byte rows of row block h; W sub-tile j/2 at byte 64 (j%2);
                // metadata column pair j/2 of row block h's group with selector j%2
                const uint32_t d = acc_base + h * TN, grp = grp0 + h * META_GROUP_COLS;
                const uint64_t ah = ad + h * ABLK;
                tc_mma_sp_pair_w(d, ah, bd, grp, IDESC_SP, acc0);
                tc_mma_sp_pair_w(d, ah + 2, bd + 4, grp, IDESC_SP | 1u, 1);
                tc_mma_sp_pair_w(d, ah + 4, bd + WSUB, grp + 2, IDESC_SP, 1);
                tc_mma_sp_pair_w(d, ah + 6, bd + WSUB + 4, grp + 2, IDESC_SP | 1u, 1);
              }
            } else {
#pragma unroll
              for (int hh = 0; hh < MB / NISS; ++hh) {
                const int h = k + hh * NISS;
                const uint32_t d = acc_base + h * TN;
                const uint64_t ah = ad + h * ABLK;
#pragma unroll
                for (int j = 0; j < C::BOXES; ++j) {  // box j: A box j and W sub-tile j, four K = 16 steps
                  tc_mma_pair_w(d, ah + j * ABOX, bd + j * WSUB, IDESC, acc0 | j);
                  tc_mma_pair_w(d, ah + j * ABOX + 2, bd + j * WSUB + 2, IDESC, 1);
                  tc_mma_pair_w(d, ah + j * ABOX + 4, bd + j * WSUB + 4, IDESC, 1);
                  tc_mma_pair_w(d, ah + j * ABOX + 6, bd + j * WSUB + 6, IDESC, 1);
                }
              }
            }
          } else {  // LoRA-up: T' (128 x 64 per row block) against this CTA's half of LA, four K = 16 steps
#pragma unroll
            for (int hh = 0; hh < MB / NISS; ++hh) {
              const int h = k + hh * NISS;
              const uint32_t d = acc_base + h * TN;
              const uint64_t ah = ad + h * ABLK;
              tc_mma_pair_w(d, ah, bd, IDESC, 1);
              tc_mma_pair_w(d, ah + 2, bd + 2, IDESC, 1);
              tc_mma_pair_w(d, ah + 4, bd + 4, IDESC, 1);
              tc_mma_pair_w(d, ah + 6, bd + 6, IDESC, 1);
            }
          }
          tc_commit_pair_w(&empty[st], 0x3);
          ++g;
          if (++st == C::NST) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!stop) tc_commit_pair_w(&acc_full[ab], 0x3);
      }
      if (lane == 0) consumed_sh[k] = g;
      tc_commit_pair_w(drain, 0x1);  // every MMA of both issuers has completed once this phase completes
      mbar_wait(drain, 0, a.ctl, SITE_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs, warps 2..9)
    // Two warps per TMEM lane quarter q: with two row blocks each drains one block's 32 rows over all TN
    // columns; with one row block each drains half of the columns.  Chunks of 32 columns are read two at a
    // time; the accumulators are released as soon as the last read has landed.  With y_tma each chunk is
    // written as a bf16 32 x 32 box into this warp's staging buffer (64-byte swizzle, so that the 32 lanes
    // writing one row each hit distinct banks) and stored by TMA; otherwise lanes store their rows directly.
    const int q = warp & 3;
    const int w2 = (warp - 2) / 4;
    const int h = MB == 2 ? w2 : 0;
    constexpr int COLS = MB == 2 ? TN : TN / 2;
    constexpr int NC = COLS / 32;
    const int col_off = MB == 2 ? 0 : w2 * COLS;
    const bool vec_ok = (a.ldy % 8) == 0;
    const bool scaled = a.scale_mode == SCALE_MUL;
    const bool y_tma = a.y_tma != 0;
    uint8_t* ybuf = ystage + (warp - 2) * C::Y_BOXES * Y_BUF;
    const uint32_t acc_empty_leader0 = mapa_shared(acc_empty, 0);  // the leader's acc_empty[0]; [1] is 8 B on
    const uint32_t taddr_warp = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * TN + col_off;
    const int m_pad = static_cast<int>(round_up(a.M, kMetaRowPad));  // GELU: metadata rows written
    int tcount = 0, ybox = 0, nsplit = 0;
    // F1: the selection of one unit's stages (two threads per row, 64 channels each; both in one warp), then s
    // of the rows for the epilogue.  cg counts the stages in the producer's order.
    int cg = 0;
    const uint32_t conv_full_leader0 = mapa_shared(&conv_full[0], 0);
    auto convert_unit = [&](int mp) -> bool {
      const int hf = lane >> 4;
      const int rr = 16 * (warp - 2) + (lane & 15);  // row of this CTA's row block
      const int grow = mp * 2 * C::ROWS + static_cast<int>(rank) * C::ROWS + rr;
      const int tl0 = (rr / 16) * 16 + (rr % 8), hh = (rr % 16) / 8;  // metadata lane base and 16-bit half
      float sx = 0.f, sk = 0.f;  // x^2 and kept x^2 of this thread's channels, over the whole K
      for (int it = 0; it <= nk; ++it, ++cg) {
        const int cst = cg % C::NST;
        bool okc = mbar_wait(&xfull[cst], (cg / C::NST) & 1, a.ctl, SITE_EPILOGUE);
        okc = __all_sync(0xFFFFFFFFu, okc) && !*abort_flag;
        if (!okc) return false;
        uint8_t* stage = smem + cst * C::STAGE;
        uint8_t* arow = stage + rr * 128;  // row rr of box 0: the compressed values, or T'
        if (it < nk) {
          const uint8_t* xr = stage + hf * C::A_BOX + rr * 128;  // channels 64 hf .. 64 hf + 63 of the step
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const uint4*>(xr + ((j ^ (rr & 7)) << 4));
          uint32_t kept[16], w0 = 0, w1 = 0;  // metadata words of 32-channel chunks 2 hf and 2 hf + 1
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t n0g = select_group(v[j].x, v[j].y, sel_table, kept[2 * j], sx, sk);
            const uint32_t n1g = select_group(v[j].z, v[j].w, sel_table, kept[2 * j + 1], sx, sk);
            if (j < 4) w0 |= (n0g | (n1g << 4)) << (8 * j);
            else w1 |= (n0g | (n1g << 4)) << (8 * (j - 4));
          }
          __syncwarp();  // both threads of every row have read box 0
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(arow + (((4 * hf + j) ^ (rr & 7)) << 4)) =
                make_uint4(kept[4 * j], kept[4 * j + 1], kept[4 * j + 2], kept[4 * j + 3]);
          uint8_t* mchunk = stage + C::A_SLOT + C::B_SLOT;  // the stage's metadata chunk, tensor-memory order
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int qh = 0; qh < 2; ++qh)
              *reinterpret_cast<uint16_t*>(mchunk + (tl0 + 8 * qh) * 16 + (2 * hf + cc) * 4 + hh * 2) =
                  static_cast<uint16_t>((cc ? w1 : w0) >> (16 * qh));
        } else {
          // the LoRA stage: s of the row from both threads' sums, then T' = bf16(T * (1 / s)) over box 0
          const float tx = sx + __shfl_xor_sync(0xFFFFFFFFu, sx, 16);
          const float tk = sk + __shfl_xor_sync(0xFFFFFFFFu, sk, 16);
          const float sv = tk > 0.f ? sqrtf(tx / tk) : 1.f;
          const float inv = 1.f / sv;
          const uint4* tsrc = reinterpret_cast<const uint4*>(a.lora_t + static_cast<int64_t>(grow < a.M ? grow : 0) *
                                                                            kRankLB + 32 * hf);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 t4 = grow < a.M ? tsrc[j] : make_uint4(0u, 0u, 0u, 0u);
            uint32_t w[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(w[u] << 16) * inv,
                                                        __uint_as_float(w[u] & 0xFFFF0000u) * inv);
              w[u] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(arow + (((4 * hf + j) ^ (rr & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (hf == 0) s_sh[rr] = sv;
        }
        fence_proxy_async();  // the generic-proxy writes above, before the tensor core reads them
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(conv_full_leader0 + 8 * cst);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(s_bar);  // this warp's rows' s are in s_sh
      bool oks = mbar_wait(s_bar, tcount & 1, a.ctl, SITE_EPILOGUE);
      return __all_sync(0xFFFFFFFFu, oks) && !*abort_flag;
    };
    Unit un;
    for (int u = 0; unit_at(u, cluster, nclusters, ntiles, nk, S, streamk, un); ++u, ++tcount) {
      const int tile = un.tile, ks = un.seg;
      const int mp = tile % num_mp, nb = tile / num_mp;
      const int row0 = mp * 2 * C::ROWS + static_cast<int>(rank) * C::ROWS + h * BLOCK + q * 32;
      const int row = row0 + lane;
      const int n0 = nb * TN + col_off;
      if constexpr (F1)
        if (!convert_unit(mp)) break;
      const float sc = F1 ? s_sh[h * BLOCK + q * 32 + lane]
                          : ((scaled && row < a.M) ? a.rowscale[row] : 1.f);  // issued before the wait
      const int ab = tcount % C::ACC_BUFS;
      bool ok = mbar_wait(&acc_full[ab], (tcount / C::ACC_BUFS) & 1, a.ctl, SITE_EPILOGUE);
      ok = __all_sync(0xFFFFFFFFu, ok) && !*abort_flag;
      if (!ok) break;
      tc_fence_after();
      __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(a.Y) + static_cast<int64_t>(row) * a.ldy;
      const bool live = row < a.M;
      // Drain: the 32 x COLS slice is read into registers (converted to bf16 pairs) before most of it is
      // written out, so the accumulators are released after ceil(NC / 2) TMEM round trips.  At most HOLD
      // chunks stay in registers (the register file holds no more without spilling); the first NC - HOLD
      // chunks are written out as soon as they are converted.
      constexpr int HOLD = TRANS ? 5 : 6;  // the transposed write-out needs a few more registers
      constexpr int EARLY = NC > HOLD ? NC - HOLD : 0;
      static_assert(EARLY == 0 || (EARLY <= 2 && C::Y_BOXES == 2), "early chunks use the warp's two staging boxes");
      uint32_t pk[NC * 16];
      auto write_chunk = [&](int c) {
        const uint32_t* p = pk + c * 16;
        const int col0 = n0 + c * 32;
        if (y_tma) {
          uint8_t* box = ybuf + ((ybox + c) % C::Y_BOXES) * Y_BUF;
          if (lane == 0) {  // the store that last used this box has read it
            if constexpr (C::Y_BOXES == 2) bulk_wait_read_one();
            else bulk_wait_read_all();
          }
          __syncwarp();
          if constexpr (TRANS) {
            // box row i = output row col0 + i (accumulator column); element `lane` of it = output column
            // row0 + lane: byte 2 lane of the 64-byte row, whose 16-byte piece lane / 8 is swizzled by row
            const int piece = lane >> 3, off = (lane & 7) * 2;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int i0 = 2 * j, i1 = 2 * j + 1;
              *reinterpret_cast<uint16_t*>(box + i0 * 64 + ((piece ^ ((i0 >> 1) & 3)) << 4) + off) =
                  static_cast<uint16_t>(p[j] & 0xFFFFu);
              *reinterpret_cast<uint16_t*>(box + i1 * 64 + ((piece ^ ((i1 >> 1) & 3)) << 4) + off) =
                  static_cast<uint16_t>(p[j] >> 16);
            }
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)  // 16-byte piece v of this lane's 64-byte row, 64-byte swizzle
              *reinterpret_cast<uint4*>(box + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            if (col0 < a.N && row0 < a.M) {
              if constexpr (TRANS) tma_store_2d(&a.tmY, box, row0, col0);
              else tma_store_2d(&a.tmY, box, col0, row0);
            }
            bulk_commit();
          }
        } else if (live) {
          if constexpr (TRANS) store_chunk_t(a.Y, a.ldy, row, col0, a.N, p);
          else store_chunk(yrow, col0, a.N, vec_ok, p);
        }
      };
      // GELU epilogue: chunk c becomes h = bf16(GELU(y)) in place; with a.hvals its 8 groups of 4 columns are
      // sparsified as the sparsify pass does (kept pairs to hvals, 16 bytes per row and chunk; the 32-bit
      // metadata word of the row, whose 16-bit halves meet those of row r +- 8 -- lane ^ 8 -- in the tensor
      // memory order of the chunk layout; squares of all and of the kept entries into the row's norm sums).
      float hn_all = 0.f, hn_kept = 0.f;
      auto finish_chunk = [&](int c) {
        if constexpr (GELU) {
          uint32_t* p = pk + c * 16;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float y0 = __uint_as_float(p[j] << 16), y1 = __uint_as_float(p[j] & 0xFFFF0000u);
            __nv_bfloat162 hv = __floats2bfloat162_rn(gelu_f(y0), gelu_f(y1));
            p[j] = *reinterpret_cast<uint32_t*>(&hv);
          }
          if (a.hvals) {
            const int col0 = n0 + c * 32;
            uint32_t kept[8], word = 0;
#pragma unroll
            for (int g = 0; g < 8; ++g)
              word |= select_group(p[2 * g], p[2 * g + 1], sel_table, kept[g], hn_all, hn_kept) << (4 * g);
            if (live && col0 < a.N) {
              uint4* dst = reinterpret_cast<uint4*>(a.hvals + static_cast<int64_t>(row) * (a.N / 2) + col0 / 2);
              dst[0] = make_uint4(kept[0], kept[1], kept[2], kept[3]);
              dst[1] = make_uint4(kept[4], kept[5], kept[6], kept[7]);
            }
            const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, word, 8);
            const bool lowrow = (lane & 8) == 0;  // row % 16 < 8: the low halves' lane
            const uint32_t mw = lowrow ? ((word & 0xFFFFu) | (other << 16)) : ((other >> 16) | (word & 0xFFFF0000u));
            const int rr = row & (kMetaRows - 1);
            const int tl = (rr >> 4) * 16 + (lowrow ? 0 : 8) + (rr & 7);
            if (row < m_pad && col0 < a.N)
              *reinterpret_cast<uint32_t*>(a.hmeta + (static_cast<int64_t>(row / kMetaRows) * (a.N / kMetaBlockCols) +
                                                      col0 / kMetaBlockCols) * kMetaChunkBytes +
                                           tl * 16 + ((col0 % kMetaBlockCols) / 32) * 4) = mw;
          }
        }
        write_chunk(c);
      };
      if (!SPLIT || un.nseg == 1) {  // a whole tile (stream-K leaves some tiles whole)
#pragma unroll
        for (int c2 = 0; c2 < NC; c2 += 2) {
          const bool two = c2 + 1 < NC;
          uint32_t r0[32], r1[32];
          tc_ld_32x32b_x32(taddr_warp + ab * C::ACC_STRIDE + c2 * 32, r0);
          if (two) tc_ld_32x32b_x32(taddr_warp + ab * C::ACC_STRIDE + (c2 + 1) * 32, r1);
          tc_wait_ld();
          if (c2 + 2 >= NC) {
            tc_fence_before();
            __syncwarp();
            // the pair's accumulators may be overwritten: this warp's TMEM reads have completed (wait::ld)
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader0 + 8 * ab);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 v0 = __floats2bfloat162_rn(__uint_as_float(r0[2 * j]) * sc, __uint_as_float(r0[2 * j + 1]) * sc);
            pk[c2 * 16 + j] = *reinterpret_cast<uint32_t*>(&v0);
            if (two) {
              __nv_bfloat162 v1 = __floats2bfloat162_rn(__uint_as_float(r1[2 * j]) * sc, __uint_as_float(r1[2 * j + 1]) * sc);
              pk[(c2 + 1) * 16 + j] = *reinterpret_cast<uint32_t*>(&v1);
            }
          }
          if (c2 < EARLY) finish_chunk(c2);
          if (c2 + 1 < EARLY) finish_chunk(c2 + 1);
        }
        // Write-out of the rest, overlapping the next tile's main loop: one bulk group per chunk, the warp's
        // staging boxes used in turn over the whole tile sequence.
#pragma unroll
        for (int c = EARLY; c < NC; ++c) finish_chunk(c);
        ybox += NC;
        if constexpr (GELU) {
          if (a.hvals && live) a.hnorm[static_cast<int64_t>(row) * a.hnorm_slots + n0 / COLS] = make_float2(hn_all, hn_kept);
        }
      } else {
        if (un.nseg > S) {  // never: the host enables stream-K only where a tile has at most S parts
          if (lane == 0) {
            *abort_flag = 1;
            record_error(a.ctl, SITE_EPILOGUE);
          }
          break;
        }
        // Split K: this unit's fp32 partial (this CTA's rows of the tile) goes to global memory, laid out as
        // [tile][split][CTA of the pair][TN][ROWS]: column-major, so that one store of the 32 lanes (32 rows of a
        // column) fills 128 contiguous bytes.
        const int64_t tile_elems = static_cast<int64_t>(C::ROWS) * TN;
        const int64_t pcol = static_cast<int64_t>(col_off) * C::ROWS + h * BLOCK + q * 32 + lane;
        float* mine = a.partials + ((static_cast<int64_t>(tile) * S + ks) * 2 + rank) * tile_elems + pcol;
#pragma unroll
        for (int c2 = 0; c2 < NC; c2 += 2) {
          const bool two = c2 + 1 < NC;
          uint32_t r0[32], r1[32];
          tc_ld_32x32b_x32(taddr_warp + ab * C::ACC_STRIDE + c2 * 32, r0);
          if (two) tc_ld_32x32b_x32(taddr_warp + ab * C::ACC_STRIDE + (c2 + 1) * 32, r1);
          tc_wait_ld();
          if (c2 + 2 >= NC) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader0 + 8 * ab);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) __stcg(mine + (c2 * 32 + j) * C::ROWS, __uint_as_float(r0[j]));
          if (two) {
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(mine + ((c2 + 1) * 32 + j) * C::ROWS, __uint_as_float(r1[j]));
          }
        }
        // Publish: every epilogue warp's partial is written (fence, then one arrival per warp); one thread
        // takes the tile's arrival ticket.  The unit that draws the last ticket adds the tile's nseg partials in
        // k order -- the same order whichever unit finishes last, so the result does not depend on timing --
        // and writes Y.  No unit waits for another: the others go on to their next unit.
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_bar);
        ok = mbar_wait(epi_bar, nsplit & 1, a.ctl, SITE_EPILOGUE);
        if (ok && warp == 2 && lane == 0) {
          unsigned int ticket;
          asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                       : "=r"(ticket)
                       : "l"(a.counters + 2 * tile + static_cast<int>(rank))
                       : "memory");
          *last_flag = ticket == static_cast<unsigned int>(un.nseg - 1);
          mbar_arrive(epi_bar2);
        }
        ok = ok && mbar_wait(epi_bar2, nsplit & 1, a.ctl, SITE_EPILOGUE);
        ok = __all_sync(0xFFFFFFFFu, ok);
        ++nsplit;
        if (!ok) break;
        if (*last_flag) {
          __threadfence();
          const float* base = a.partials + (static_cast<int64_t>(tile) * S * 2 + rank) * tile_elems + pcol;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            float acc[32];
            // eight columns at a time: every split's loads are issued before the columns are added in split order
#pragma unroll
            for (int j0 = 0; j0 < 32; j0 += 8) {
              float t[kPairMaxSplit][8];
#pragma unroll
              for (int s2 = 0; s2 < kPairMaxSplit; ++s2)
                if (s2 < un.nseg)
#pragma unroll
                  for (int jj = 0; jj < 8; ++jj)
                    t[s2][jj] = __ldcg(base + s2 * 2 * tile_elems + (c * 32 + j0 + jj) * C::ROWS);
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                float sum = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < kPairMaxSplit; ++s2)
                  if (s2 < un.nseg) sum += t[s2][jj];
                acc[j0 + jj] = sum;
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              __nv_bfloat162 v0 = __floats2bfloat162_rn(acc[2 * j] * sc, acc[2 * j + 1] * sc);
              pk[c * 16 + j] = *reinterpret_cast<uint32_t*>(&v0);
            }
            write_chunk(c);
          }
          ybox += NC;
        }
      }
    }
    if (y_tma && lane == 0) bulk_wait_all();
  }
  __syncwarp();
  __syncthreads();

  if (*abort_flag && leader && warp == 0 && lane == 0) {
    // Let every copy of this stage sequence land (both CTAs signal the leader's barriers).
    const int issued = *issued_sh;
    const int consumed = NISS == 2 && consumed_sh[1] < consumed_sh[0] ? consumed_sh[1] : consumed_sh[0];
    for (int g = consumed; g < issued; ++g) {
      if (a.ctl.inject == 1 && g == 0) continue;
      if (!mbar_wait(&full[g % C::NST], (g / C::NST) & 1, a.ctl, SITE_DRAIN)) break;
    }
  }
  if (F1 && *abort_flag && warp == 0 && lane == 0) {
    // this CTA's X loads of the last stages issued land before it leaves
    const int issued = *issued_sh;
    for (int g = issued > C::NST ? issued - C::NST : 0; g < issued; ++g)
      if (!mbar_wait(&xfull[g % C::NST], (g / C::NST) & 1, a.ctl, SITE_DRAIN)) break;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still read its shared memory or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <bool SPARSE, bool LORA, int MB, int TN, bool TRANS = false, bool SPLIT = false, bool GELU = false,
          bool F1 = false>
cudaError_t launch(const PairArgs& a, cudaStream_t st) {
  using C = PairCfg<SPARSE, MB, TN, F1>;
  auto* k = gemm_pair_kernel<SPARSE, LORA, MB, TN, TRANS, SPLIT, GELU, F1>;
  constexpr int smem = C::SMEM + ((GELU || F1) ? 256 : 0) + (F1 ? 512 : 0);  // + the selection table, s
  static_assert(smem <= SMEM_LIMIT, "shared memory budget");
  static std::atomic<bool> attr_set[64] = {};  // per device; setting it twice from racing threads is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int ntiles = ((a.M + 2 * C::ROWS - 1) / (2 * C::ROWS)) * ((a.N + TN - 1) / TN);
  const int nk = (a.K + C::BK - 1) / C::BK;
  // stream-K: every pair takes a share of the k-steps (at least one each); otherwise one pair per unit at most
  const int64_t nunits = (SPLIT && a.stream_k) ? static_cast<int64_t>(ntiles) * nk
                                               : static_cast<int64_t>(ntiles) * (SPLIT ? a.splits : 1);
  int clusters = sm_count() / 2;
  if (clusters > nunits) clusters = static_cast<int>(nunits);
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the previous kernel ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(2 * clusters);  // the cluster shape (2, 1, 1) is the kernel's own attribute
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace

cudaError_t launch_gemm_pair(bool sparse, bool lora, PairShape shape, const PairArgs& a, cudaStream_t st,
                             bool gelu) {
  if (!pair_shape_valid(sparse, shape)) return cudaErrorInvalidValue;
  if (gelu) {  // the MLP up layer: sparse with LoRA, or dense
    if (!sparse && shape.tn == 448)
      return lora ? launch<false, true, 1, 448, false, false, true>(a, st)
                  : launch<false, false, 1, 448, false, false, true>(a, st);
    if (!sparse)
      return lora ? launch<false, true, 1, 256, false, false, true>(a, st)
                  : launch<false, false, 1, 256, false, false, true>(a, st);
    if (!lora) return cudaErrorInvalidValue;
    if (shape.rb == 2 && shape.tn == 224) return launch<true, true, 2, 224, false, false, true>(a, st);
    if (shape.rb == 2) return launch<true, true, 2, 192, false, false, true>(a, st);
    if (shape.tn == 192) return launch<true, true, 1, 192, false, false, true>(a, st);
    return launch<true, true, 1, 256, false, false, true>(a, st);
  }
  if (!sparse && shape.tn == 448) return lora ? launch<false, true, 1, 448>(a, st) : launch<false, false, 1, 448>(a, st);
  if (!sparse) return lora ? launch<false, true, 1, 256>(a, st) : launch<false, false, 1, 256>(a, st);
  if (shape.rb == 2 && shape.tn == 224)
    return lora ? launch<true, true, 2, 224>(a, st) : launch<true, false, 2, 224>(a, st);
  if (shape.rb == 2)
    return lora ? launch<true, true, 2, 192>(a, st) : launch<true, false, 2, 192>(a, st);
  // split K: the one-row-block tiles only (the shapes few-tile problems take)
  if (shape.tn == 192) {
    if (a.splits > 1)
      return lora ? launch<true, true, 1, 192, false, true>(a, st) : launch<true, false, 1, 192, false, true>(a, st);
    return lora ? launch<true, true, 1, 192>(a, st) : launch<true, false, 1, 192>(a, st);
  }
  if (a.splits > 1)
    return lora ? launch<true, true, 1, 256, false, true>(a, st) : launch<true, false, 1, 256, false, true>(a, st);
  return lora ? launch<true, true, 1, 256>(a, st) : launch<true, false, 1, 256>(a, st);
}

cudaError_t launch_gemm_pair_f1(const PairArgs& a, cudaStream_t st) {
  if (!a.lora_t || a.splits != 1) return cudaErrorInvalidValue;
  return launch<true, true, 1, 256, false, false, false, true>(a, st);
}

cudaError_t launch_gemm_pair_transposed(bool lora, PairShape shape, const PairArgs& a, cudaStream_t st) {
  if (!pair_shape_valid(true, shape)) return cudaErrorInvalidValue;
  if (shape.rb == 2 && shape.tn == 224)
    return lora ? launch<true, true, 2, 224, true>(a, st) : launch<true, false, 2, 224, true>(a, st);
  if (shape.rb == 2)
    return lora ? launch<true, true, 2, 192, true>(a, st) : launch<true, false, 2, 192, true>(a, st);
  if (shape.tn == 192) return lora ? launch<true, true, 1, 192, true>(a, st) : launch<true, false, 1, 192, true>(a, st);
  return lora ? launch<true, true, 1, 256, true>(a, st) : launch<true, false, 1, 256, true>(a, st);
}

}  // namespace lynx
