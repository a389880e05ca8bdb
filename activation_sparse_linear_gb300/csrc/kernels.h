// Internal launch interface between the C-ABI layer (lynx_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "../../include/lynx.h"

namespace lynx {

// Metadata tiling shared by the sparsify kernel, the sparse GEMMs and the host
// conversion to the canonical layout.  One tcgen05.mma.sp (M = 128 rows per
// CTA, 32 input channels) reads one 32-bit TMEM column: 8 groups x 4 bits per
// row.  Inside every 16-row block the hardware pairs rows r and r+8 by 16-bit
// halves: lane 16b+i (i < 8) holds bits 0-15 of row 16b+i in its low half and
// bits 0-15 of row 16b+8+i in its high half; lane 16b+8+i holds bits 16-31 of
// the same two rows.  A row's 32 bits carry group g (channels 4g..4g+3 of the
// chunk) in bits 4g..4g+3 as i0 | i1 << 2.  The MMA's metadata address must
// be an even column; bit 0 of the instruction descriptor (sparsity selector)
// selects that column or the next one.
//
// In global memory every (128-row block, 128-channel block) owns a 2 KiB chunk
// of 128 lanes x 16 bytes, row blocks outermost: word w of lane L is the TMEM
// word of lane L for channels 32w..32w+31 of the block, so one
// tcgen05.cp.128x128b lands four MMAs' metadata in four TMEM columns.
// Channels are padded to a multiple of 128 and rows to a multiple of 256 (a
// CTA pair) with the pattern of an all-zero group (0x4).
constexpr int kMetaRows = 128;
constexpr int kMetaRowPad = 256;
constexpr int kMetaChunkCols = 32;
constexpr int kMetaBlockCols = 128;
constexpr int kMetaChunkBytes = kMetaRows * 16;
__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
__host__ __device__ inline int64_t meta_blocks_k(int64_t K) { return round_up(K, kMetaBlockCols) / kMetaBlockCols; }
__host__ __device__ inline int64_t meta_bytes(int64_t M, int64_t K) {
  return round_up(M, kMetaRowPad) / kMetaRows * meta_blocks_k(K) * kMetaChunkBytes;
}
// Byte offset of the 16-bit half holding bits [16q, 16q+16) of row r's word for 32-channel chunk c.
__host__ __device__ inline int64_t meta_half_offset(int64_t r, int64_t c, int q, int64_t blocks_k) {
  const int64_t blk = r / kMetaRows, rr = r % kMetaRows;
  const int64_t lane = (rr / 16) * 16 + q * 8 + (rr % 8);
  const int64_t h = (rr % 16) / 8;
  return (blk * blocks_k + c / 4) * kMetaChunkBytes + lane * 16 + (c % 4) * 4 + h * 2;
}


// Fused sparsification + LoRA down-projection (prologue.cu).
constexpr int kRankLB = 64;            // LoRA rank handled by the tensor-core paths
constexpr int kMaxPrologueSplit = 16;  // CTAs (one cluster) per row block; 16 is a non-portable cluster size
struct ProArgs {
  CUtensorMap tmX;   // X (M x K bf16), box 64 x 128, 128-byte swizzle
  CUtensorMap tmLB;  // LB (64 x K bf16), box 64 x 64, 128-byte swizzle (LoRA branch only)
  uint16_t* vals;    // compressed values, M x K/2 bf16 (row-major)
  uint8_t* meta;     // metadata chunks (layout above)
  float* s;          // s = sqrt(sum x^2 / sum kept x^2) (1 for an all-zero row), M floats
  void* T;           // LoRA: T' = (X LB^T) / s, M x 64 bf16
  unsigned int* zero;  // words set to 0 before anything else (the next GEMM's split-K counters), or NULL
  int nzero;
  int M, K, M_pad, split, nkb;  // M_pad = round_up(M, 256); split = cluster size; nkb = 128-channel blocks
  DevCtl ctl;
};
int prologue_split(int M, int K);
cudaError_t launch_prologue(const ProArgs& a, bool lora, cudaStream_t st);

enum ScaleMode : int { SCALE_NONE = 0, SCALE_MUL = 1, SCALE_DIV = 2 };

struct GemmArgs {
  CUtensorMap tmA;    // A: X (M x K), box 64 x 128, 128-byte swizzle
  CUtensorMap tmB;    // B: LB (64 x K), box 64 x 64, 128-byte swizzle
  const float* rowscale;
  int scale_mode;     // SCALE_NONE or SCALE_DIV (T' = X LB^T / s)
  void* Y;
  int64_t ldy;
  int M, N, K;        // N = 64
  DevCtl ctl;
};

// The dense single-CTA tcgen05 GEMM on 128 x 64 tiles (gemm.cu).
cudaError_t launch_proj_gemm(const GemmArgs& a, cudaStream_t st);

// Pair-tile shapes: rb = 128-row blocks per CTA (the pair covers 256 * rb rows), tn = output columns per tile
// (W and LA are staged tn / 2 rows per CTA).  The sparse path uses 512 x 224, 512 x 192 or 256 x 256 tiles,
// whichever costs the fewest tile waves x shared-memory bytes for the shape; the dense path uses 256 x 256.
struct PairShape {
  int rb, tn;
};
PairShape pair_shape(bool sparse, int M, int N);
// The same choice for a GPU with `clusters` CTA pairs (host logic only; no device call).
PairShape pair_shape_for(bool sparse, int M, int N, int64_t clusters);
bool pair_shape_valid(bool sparse, PairShape shape);

struct PairArgs {
  CUtensorMap tmA;     // sparse: compressed values; dense: X (both box 64 x 128, 128-byte swizzle)
  CUtensorMap tmB;     // W, box 64 x TileN/2 (one CTA's half of a column tile), 128-byte swizzle
  CUtensorMap tmMeta;  // metadata as uint32 [2 * chunks][256]; box 256 x 2 = one 2 KiB chunk
  CUtensorMap tmT;     // T' (M x 64), box 64 x 128, 128-byte swizzle
  CUtensorMap tmLA;    // LA (N x 64), box 64 x TileN/2, 128-byte swizzle
  CUtensorMap tmY;     // Y (M x N bf16), box 32 x 32, 64-byte swizzle; used when y_tma != 0 (N % 8 == 0)
  int y_tma;
  const float* rowscale;
  int scale_mode;      // SCALE_NONE or SCALE_MUL
  void* Y;
  int64_t ldy;
  int M, N, K;
  int splits;              // k-splits per tile (1: none); > 1 needs partials and counters
  int stream_k;            // with splits = kPairMaxSplit: stream-K (contiguous k-step ranges per CTA pair)
  float* partials;         // fp32 partial tiles, [tile][split][CTA][rows][TN] (splits > 1)
  unsigned int* counters;  // one arrival counter per (tile, CTA), zero on entry (splits > 1)
  // GELU epilogue (the MLP up layer): Y = bf16(GELU(bf16(y))); with hvals non-NULL the epilogue also writes the
  // 2:4 sparsification of that output for the next layer: compressed values (M x N/2 bf16), metadata chunks
  // (lynx_meta_bytes(M, N), N % 128 == 0) and, per row and per 32 x (columns of one epilogue warp) slot, the
  // fp32 pair (sum h^2, sum kept h^2).
  uint16_t* hvals;
  uint8_t* hmeta;
  float2* hnorm;
  int hnorm_slots;         // slots per row
  unsigned int* zero;      // words set to 0 once the previous kernel is done (the next kernel's counters), or NULL
  int nzero;
  const uint16_t* lora_t;  // in-GEMM selection: T = X LB^T (M x 64 bf16, not divided by s)
  DevCtl ctl;
};

// The CTA-pair (cta_group::2) GEMM with the given tile shape (one of those pair_shape returns); gelu selects the
// GELU epilogue (sparse tiles with LoRA, and the dense tile).
cudaError_t launch_gemm_pair(bool sparse, bool lora, PairShape shape, const PairArgs& a, cudaStream_t st,
                             bool gelu = false);
// Norm-partial slots per row of the GELU epilogue for an output of N columns with this tile shape.
int gelu_norm_slots(bool sparse, PairShape shape, int N);
// The sparse pair GEMM that selects the 2:4 pattern itself (256 x 256 tiles): a.tmA maps the dense X (box 64 x
// 128, 128-byte swizzle), a.lora_t holds T = X LB^T; s comes from the GEMM's own row sums (a.rowscale unused).
cudaError_t launch_gemm_pair_f1(const PairArgs& a, cudaStream_t st);
// The sparse pair GEMM whose accumulator tile is the transpose of Y: a.M and a.N count the accumulator's rows
// and columns (Y's columns and rows), tmY and ldy describe Y itself (rows of ldy elements).
cudaError_t launch_gemm_pair_transposed(bool lora, PairShape shape, const PairArgs& a, cudaStream_t st);

// LoRA down-projection and row scale of a sparse layer whose input H was sparsified by the previous layer's
// GELU epilogue (lora_fin.cu): T' = bf16(H LB^T / s), s from the epilogue's norm partials.
struct FinArgs {
  CUtensorMap tmH;         // H (M x K bf16), box 64 x 128, 128-byte swizzle
  CUtensorMap tmLB;        // LB (64 x K bf16), box 64 x 64, 128-byte swizzle
  const float2* hnorm;     // (sum h^2, sum kept h^2) per row and slot, slots per row
  int slots;
  float* s;                // out: M fp32
  void* T;                 // out: M x 64 bf16
  float* partials;         // splits > 1: fp32 partials [tile][split][128][64]
  unsigned int* counters;  // splits > 1: one arrival counter per 128-row tile, zero on entry
  int M, K, splits;
  DevCtl ctl;
};
int lora_fin_splits(int M, int K);
size_t lora_fin_partial_bytes(int M, int splits);
int lora_fin_counters(int M);
cudaError_t launch_lora_fin(const FinArgs& a, cudaStream_t st);

int sm_count();

// Host argument checks of lynx_linear and lynx_linear_dense (lynx_api.cu): the status either call would return
// before launching anything, LYNX_OK when it would launch.
int linear_arg_status(const void* X, const void* W, const void* LA, const void* LB, const void* Y, int64_t M,
                      int64_t N, int64_t K, int64_t R, const void* workspace, size_t workspace_bytes);
int dense_arg_status(const void* X, const void* W, const void* LA, const void* LB, const void* Y, int64_t M,
                     int64_t N, int64_t K, int64_t R, const void* workspace, size_t workspace_bytes);
// Drops this thread's pending stage-timing request (lynx_profile_next), so that a graph capture records none.
void clear_stage_request();

// Layer sequences (lynx_api.cu, used by layers.cu): the status the sequence would return before launching (the
// failing index in *failed), its workspace bytes, and its launches.  A layer with the GELU flag followed by a
// sparse layer that reads its output runs as one fused pair when the workspace holds the pair's plan.
int seq_status(const lynx_layer* layers, int32_t n, const void* ws, size_t ws_bytes, int32_t* failed);
size_t seq_workspace_bytes(const lynx_layer* layers, int32_t n);
int seq_enqueue(const lynx_layer* layers, int32_t n, void* ws, size_t ws_bytes, cudaStream_t st);
// Byte offsets in the workspace of the fused pair (i, i + 1): the down layer's values, metadata, s, T', and the
// pair's total workspace bytes (out[0..4]); LYNX_ERR_UNSUPPORTED when the two layers do not fuse.
int seq_pair_offsets(const lynx_layer* layers, int32_t n, int32_t i, size_t* out);

}  // namespace lynx
