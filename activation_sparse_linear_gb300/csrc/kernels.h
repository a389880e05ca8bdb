// Internal launch interface between the C-ABI layer (lynx_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace lynx {

// Metadata tiling shared by the sparsify kernel, the sparse GEMM and the host
// conversion to the canonical layout.  One tcgen05.mma.sp (M = 128 rows, 32
// input channels) reads one 32-bit TMEM column: 8 groups x 4 bits per row.
// Inside every 16-row block the hardware pairs rows r and r+8 by 16-bit
// halves: lane 16b+i (i < 8) holds bits 0-15 of row 16b+i in its low half and
// bits 0-15 of row 16b+8+i in its high half; lane 16b+8+i holds bits 16-31 of
// the same two rows.  A row's 32 bits carry group g (channels 4g..4g+3 of the
// chunk) in bits 4g..4g+3 as i0 | i1 << 2.
//
// In global memory every (128-row block, 32-channel chunk) owns a 2 KiB chunk
// of 128 lanes x 16 bytes, row blocks outermost; word 0 of lane L is the TMEM
// word of lane L, words 1-3 are never written or read as metadata.  The 16-byte
// lane pitch lets tcgen05.cp.128x128b land each chunk on its own 32-column
// aligned TMEM slot.  Channels are padded to a multiple of 64 (one GEMM stage)
// and rows to a multiple of 128 with the pattern of an all-zero group (0x4).
constexpr int kMetaRows = 128;
constexpr int kMetaChunkCols = 32;
constexpr int kMetaChunkBytes = kMetaRows * 16;
constexpr int kMetaKPad = 64;
__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
__host__ __device__ inline int64_t meta_chunks_k(int64_t K) { return round_up(K, kMetaKPad) / kMetaChunkCols; }
__host__ __device__ inline int64_t meta_bytes(int64_t M, int64_t K) {
  return round_up(M, kMetaRows) / kMetaRows * meta_chunks_k(K) * kMetaChunkBytes;
}
// Byte offset of the 16-bit half holding bits [16q, 16q+16) of row r's word for chunk c.
__host__ __device__ inline int64_t meta_half_offset(int64_t r, int64_t c, int q, int64_t chunks_k) {
  const int64_t blk = r / kMetaRows, rr = r % kMetaRows;
  const int64_t lane = (rr / 16) * 16 + q * 8 + (rr % 8);
  const int64_t h = (rr % 16) / 8;
  return (blk * chunks_k + c) * kMetaChunkBytes + lane * 16 + h * 2;
}

cudaError_t launch_sparsify(const void* X, int M, int K, void* vals, void* meta, float* s, cudaStream_t st);

enum ScaleMode : int { SCALE_NONE = 0, SCALE_MUL = 1, SCALE_DIV = 2 };

struct GemmArgs {
  CUtensorMap tmA;    // A operand: X (dense) or compressed values (sparse)
  CUtensorMap tmB;    // B operand: W (N x K) or LB (R x K)
  CUtensorMap tmT;    // LoRA-up A: T' (M x R)
  CUtensorMap tmLA;   // LoRA-up B: LA (N x R)
  const uint8_t* meta;
  const float* rowscale;
  int scale_mode;
  void* Y;
  int64_t ldy;
  int M, N, K;
  DevCtl ctl;
};

// kind: 0 = dense, 256-wide tiles; 1 = dense + LoRA-up tail; 2 = sparse + LoRA-up tail;
// 3 = sparse, no LoRA; 4 = dense, 64-wide tiles (LoRA down-projection).
cudaError_t launch_gemm(int kind, const GemmArgs& a, cudaStream_t st);

}  // namespace lynx
