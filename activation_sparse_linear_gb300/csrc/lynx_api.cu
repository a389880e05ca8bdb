// C-ABI of the RT-Lynx activation-sparse linear layer: argument checks, tensor
// maps, workspace carving, kernel launches and the device error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/lynx.h"
#include "kernels.h"

namespace lynx {
namespace {

constexpr int64_t kMaxM = 65535LL * 128;  // keeps int row indices and TMA coordinates far inside 32 bits
constexpr int64_t kMaxN = 1LL << 24;
constexpr int64_t kMaxMN = 1LL << 40;     // keeps the GEMMs' int tile counts (<= M N / 2^15) inside 32 bits
constexpr int64_t kMaxK = 1LL << 20;
constexpr int kRank = 64;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

__device__ int g_error_word;

std::atomic<int> g_inject{0};
std::atomic<int> g_force_tile{0};  // 0: tile shape by problem shape; else a forced shape, rb << 16 | tn
std::atomic<int> g_force_split{0};  // 0: pre-pass cluster size by occupancy; else a forced size
thread_local void* const* t_prof_events = nullptr;
thread_local int t_prof_count = 0;

// Consumes the stage-timing request of this thread (see lynx_profile_next).
struct StageEvents {
  void* const* ev = nullptr;
  int n = 0;
  StageEvents(int expected) {
    if (t_prof_events && t_prof_count == expected) {
      ev = t_prof_events;
      n = expected;
    }
    t_prof_events = nullptr;
    t_prof_count = 0;
  }
  cudaError_t mark(int i, cudaStream_t st) const {
    if (!ev || i >= n) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
  }
};
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

int* error_word_ptr() {
  static int* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// 2-D tensor map over a row-major [rows x cols] array with row stride `ld` elements (bf16 by default).
bool make_map(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swz,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t esize = dtype == CU_TENSOR_MAP_DATA_TYPE_UINT32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, dtype, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output tensor map for the pair GEMM's TMA-store epilogue: rows of N bf16 need a 16-byte multiple stride,
// so other N keep the direct per-lane stores.
bool set_y_map(PairArgs* g, void* Y, int64_t M, int64_t N) {
  g->y_tma = 0;
  if (N % 8 != 0) return true;
  if (!make_map(&g->tmY, Y, N, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) return false;
  g->y_tma = 1;
  return true;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

int check_mk(int64_t M, int64_t K) {
  if (M < 1 || M > kMaxM || K < 16 || K > kMaxK || K % 16 != 0) return LYNX_ERR_SHAPE;
  return LYNX_OK;
}

int check_n(int64_t M, int64_t N) {
  if (N < 1 || N > kMaxN || M * N > kMaxMN) return LYNX_ERR_SHAPE;
  return LYNX_OK;
}

DevCtl make_ctl() {
  DevCtl c;
  c.err = error_word_ptr();
  c.wait_ns = g_wait_ns.load();
  c.inject = g_inject.load();
  return c;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LYNX_OK : LYNX_ERR_CUDA; }


struct Workspace {
  void* vals;
  void* meta;
  float* s;
  void* T;
  size_t bytes;
};

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

Workspace carve(void* base, int64_t M, int64_t K, int64_t R) {
  Workspace w{};
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  size_t off = 0;
  w.vals = reinterpret_cast<void*>(b + off);
  off += align256(static_cast<size_t>(M) * static_cast<size_t>(K));  // M x K/2 bf16
  w.meta = reinterpret_cast<void*>(b + off);
  off += align256(static_cast<size_t>(meta_bytes(M, K)));
  w.s = reinterpret_cast<float*>(b + off);
  off += align256(static_cast<size_t>(M) * 4);
  w.T = reinterpret_cast<void*>(b + off);
  off += align256(static_cast<size_t>(M) * static_cast<size_t>(R) * 2);
  w.bytes = off;
  (void)R;
  return w;
}

// T = X LB^T [/ s] on the 64-wide tcgen05 tile (standalone down-projection and the dense path).
int run_lora_down(const void* X, const void* LB, const float* s, void* T, int64_t M, int64_t K, cudaStream_t st) {
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  if (!make_map(&g.tmA, X, K, M, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LYNX_ERR_CUDA;
  if (!make_map(&g.tmB, LB, K, kRank, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return LYNX_ERR_CUDA;
  g.rowscale = s;
  g.scale_mode = s ? SCALE_DIV : SCALE_NONE;
  g.Y = T;
  g.ldy = kRank;
  g.M = static_cast<int>(M);
  g.N = kRank;
  g.K = static_cast<int>(K);
  g.ctl = make_ctl();
  return cuda_status(launch_proj_gemm(g, st));
}

// Prologue arguments: X (and LB for the LoRA branch) in, vals / meta / s (/ T') out, shares in the workspace.
int make_prologue(ProArgs* pa, const void* X, const void* LB, int64_t M, int64_t K, void* vals, void* meta, float* s,
                  void* T) {
  std::memset(pa, 0, sizeof(*pa));
  if (!make_map(&pa->tmX, X, K, M, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&pa->tmV, vals, K / 2, M, K / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      (LB && !make_map(&pa->tmLB, LB, K, kRank, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)))
    return LYNX_ERR_CUDA;
  pa->meta = static_cast<uint8_t*>(meta);
  pa->s = s;
  pa->T = T;
  pa->M = static_cast<int>(M);
  pa->K = static_cast<int>(K);
  pa->M_pad = static_cast<int>(round_up(M, kMetaRowPad));
  pa->nkb = static_cast<int>(meta_blocks_k(K));
  const int forced = g_force_split.load();
  pa->split = forced ? (forced < pa->nkb ? forced : pa->nkb) : prologue_split(pa->M, pa->K);
  pa->ctl = make_ctl();
  return LYNX_OK;
}

}  // namespace

int linear_arg_status(const void* X, const void* W, const void* LA, const void* LB, const void* Y, int64_t M,
                      int64_t N, int64_t K, int64_t R, const void* workspace, size_t workspace_bytes) {
  if (!X || !W || !LA || !LB || !Y || !workspace) return LYNX_ERR_NULL;
  if (int e = check_mk(M, K)) return e;
  if (int e = check_n(M, N)) return e;
  if (R != kRank) return R < 1 ? LYNX_ERR_SHAPE : LYNX_ERR_UNSUPPORTED;
  if (misaligned(X) || misaligned(W) || misaligned(LA) || misaligned(LB) || misaligned(Y) || misaligned(workspace))
    return LYNX_ERR_ALIGN;
  if (workspace_bytes < carve(nullptr, M, K, R).bytes) return LYNX_ERR_WORKSPACE;
  return LYNX_OK;
}

int dense_arg_status(const void* X, const void* W, const void* LA, const void* LB, const void* Y, int64_t M,
                     int64_t N, int64_t K, int64_t R, const void* workspace, size_t workspace_bytes) {
  if (!X || !W || !Y) return LYNX_ERR_NULL;
  const bool lora = LA || LB;
  if (lora && (!LA || !LB || !workspace)) return LYNX_ERR_NULL;
  if (int e = check_mk(M, K)) return e;
  if (int e = check_n(M, N)) return e;
  if (lora && R != kRank) return R < 1 ? LYNX_ERR_SHAPE : LYNX_ERR_UNSUPPORTED;
  if (misaligned(X) || misaligned(W) || misaligned(Y) ||
      (lora && (misaligned(LA) || misaligned(LB) || misaligned(workspace))))
    return LYNX_ERR_ALIGN;
  if (lora && workspace_bytes < align256(static_cast<size_t>(M) * static_cast<size_t>(R) * 2))
    return LYNX_ERR_WORKSPACE;
  return LYNX_OK;
}

void clear_stage_request() {
  t_prof_events = nullptr;
  t_prof_count = 0;
}

}  // namespace lynx

using namespace lynx;

extern "C" {

size_t lynx_meta_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 1) return 0;
  return static_cast<size_t>(meta_bytes(M, K));
}

size_t lynx_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R) {
  (void)N;
  if (M < 1 || K < 1 || R < 0) return 0;
  return carve(nullptr, M, K, R).bytes;
}

size_t lynx_dense_workspace_bytes(int64_t M, int64_t R) {
  if (M < 1 || R < 0) return 0;
  return align256(static_cast<size_t>(M) * static_cast<size_t>(R) * 2);
}

int lynx_sparsify(const void* X, int64_t M, int64_t K, void* vals, void* meta, float* s, void* stream) {
  return lynx_sparsify_lora(X, nullptr, M, K, kRank, vals, meta, s, nullptr, stream);
}

int lynx_lora_down(const void* X, const void* LB, const float* s, void* T, int64_t M, int64_t K, int64_t R,
                   void* stream) {
  if (!X || !LB || !T) return LYNX_ERR_NULL;
  if (int e = check_mk(M, K)) return e;
  if (R != kRank) return R < 1 ? LYNX_ERR_SHAPE : LYNX_ERR_UNSUPPORTED;
  if (misaligned(X) || misaligned(LB) || misaligned(T) || (s && (reinterpret_cast<uintptr_t>(s) & 3)))
    return LYNX_ERR_ALIGN;
  return run_lora_down(X, LB, s, T, M, K, static_cast<cudaStream_t>(stream));
}

int lynx_linear(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M, int64_t N,
                int64_t K, int64_t R, void* workspace, size_t workspace_bytes, void* stream) {
  if (int e = linear_arg_status(X, W, LA, LB, Y, M, N, K, R, workspace, workspace_bytes)) return e;
  Workspace ws = carve(workspace, M, K, R);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  PairArgs g;
  std::memset(&g, 0, sizeof(g));
  const int forced = g_force_tile.load();
  const PairShape shape = forced ? PairShape{forced >> 16, forced & 0xFFFF}
                                 : pair_shape(true, static_cast<int>(M), static_cast<int>(N));
  const uint64_t meta_rows = 2 * static_cast<uint64_t>(meta_bytes(M, K) / kMetaChunkBytes);  // 1 KiB rows
  if (!make_map(&g.tmA, ws.vals, K / 2, M, K / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmB, W, K, N, K, 64, shape.tn / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmMeta, ws.meta, 256, meta_rows, 256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_DATA_TYPE_UINT32) ||
      !make_map(&g.tmT, ws.T, R, M, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmLA, LA, R, N, R, 64, shape.tn / 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return LYNX_ERR_CUDA;
  if (!set_y_map(&g, Y, M, N)) return LYNX_ERR_CUDA;
  g.rowscale = ws.s;
  g.scale_mode = SCALE_MUL;
  g.Y = Y;
  g.ldy = N;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.ctl = make_ctl();

  ProArgs pa;
  if (int e = make_prologue(&pa, X, LB, M, K, ws.vals, ws.meta, ws.s, ws.T)) return e;

  StageEvents prof(3);
  if (cudaError_t e = prof.mark(0, st)) return cuda_status(e);
  if (cudaError_t e = launch_prologue(pa, true, st)) return cuda_status(e);
  if (cudaError_t e = prof.mark(1, st)) return cuda_status(e);
  if (cudaError_t e = launch_gemm_pair(true, true, shape, g, st)) return cuda_status(e);
  return cuda_status(prof.mark(2, st));
}

int lynx_sparsify_lora(const void* X, const void* LB, int64_t M, int64_t K, int64_t R, void* vals, void* meta,
                       float* s, void* T, void* stream) {
  if (!X || !vals || !meta || !s) return LYNX_ERR_NULL;
  if ((LB == nullptr) != (T == nullptr)) return LYNX_ERR_NULL;
  if (int e = check_mk(M, K)) return e;
  if (LB && R != kRank) return R < 1 ? LYNX_ERR_SHAPE : LYNX_ERR_UNSUPPORTED;
  if (misaligned(X) || misaligned(vals) || misaligned(meta) || misaligned(s) ||
      (LB && (misaligned(LB) || misaligned(T))))
    return LYNX_ERR_ALIGN;
  ProArgs pa;
  if (int e = make_prologue(&pa, X, LB, M, K, vals, meta, s, T)) return e;
  return cuda_status(launch_prologue(pa, LB != nullptr, static_cast<cudaStream_t>(stream)));
}

int lynx_linear_dense(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M,
                      int64_t N, int64_t K, int64_t R, void* workspace, size_t workspace_bytes, void* stream) {
  if (int e = dense_arg_status(X, W, LA, LB, Y, M, N, K, R, workspace, workspace_bytes)) return e;
  const bool lora = LA || LB;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  PairArgs g;
  std::memset(&g, 0, sizeof(g));
  if (!make_map(&g.tmA, X, K, M, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmB, W, K, N, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return LYNX_ERR_CUDA;
  if (lora) {
    if (!make_map(&g.tmT, workspace, R, M, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&g.tmLA, LA, R, N, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
      return LYNX_ERR_CUDA;
  }
  if (!set_y_map(&g, Y, M, N)) return LYNX_ERR_CUDA;
  g.rowscale = nullptr;
  g.scale_mode = SCALE_NONE;
  g.Y = Y;
  g.ldy = N;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.ctl = make_ctl();
  StageEvents prof(lora ? 3 : 2);
  if (cudaError_t e = prof.mark(0, st)) return cuda_status(e);
  if (lora) {
    if (int e = run_lora_down(X, LB, nullptr, workspace, M, K, st)) return e;
    if (cudaError_t e = prof.mark(1, st)) return cuda_status(e);
    if (cudaError_t e = launch_gemm_pair(false, true, PairShape{1, 256}, g, st)) return cuda_status(e);
    return cuda_status(prof.mark(2, st));
  }
  if (cudaError_t e = launch_gemm_pair(false, false, PairShape{1, 256}, g, st)) return cuda_status(e);
  return cuda_status(prof.mark(1, st));
}

int lynx_linear_wsparse(const void* X, const void* Wvals, const void* Wmeta, const void* LA, const void* LB, void* Y,
                        int64_t M, int64_t N, int64_t K, int64_t R, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (!X || !Wvals || !Wmeta || !Y) return LYNX_ERR_NULL;
  const bool lora = LA || LB;
  if (lora && (!LA || !LB || !workspace)) return LYNX_ERR_NULL;
  if (int e = check_mk(M, K)) return e;
  if (int e = check_n(M, N)) return e;
  if (N > kMaxM) return LYNX_ERR_SHAPE;  // W's rows are the GEMM's row blocks
  if (lora && R != kRank) return R < 1 ? LYNX_ERR_SHAPE : LYNX_ERR_UNSUPPORTED;
  if (misaligned(X) || misaligned(Wvals) || misaligned(Wmeta) || misaligned(Y) ||
      (lora && (misaligned(LA) || misaligned(LB) || misaligned(workspace))))
    return LYNX_ERR_ALIGN;
  if (lora && workspace_bytes < lynx_dense_workspace_bytes(M, R)) return LYNX_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // The sparse operand is W~ (N rows), the dense one X (M rows): the accumulator tile is Y^T.  The LoRA stage
  // swaps likewise: LA (N x 64) on the sparse operand's side, T = X LB^T (M x 64) on the other.
  PairArgs g;
  std::memset(&g, 0, sizeof(g));
  const int forced = g_force_tile.load();
  const PairShape shape = forced ? PairShape{forced >> 16, forced & 0xFFFF}
                                 : pair_shape(true, static_cast<int>(N), static_cast<int>(M));
  const uint64_t meta_rows = 2 * static_cast<uint64_t>(meta_bytes(N, K) / kMetaChunkBytes);
  if (!make_map(&g.tmA, Wvals, K / 2, N, K / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmB, X, K, M, K, 64, shape.tn / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmMeta, Wmeta, 256, meta_rows, 256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_DATA_TYPE_UINT32))
    return LYNX_ERR_CUDA;
  if (lora && (!make_map(&g.tmT, LA, R, N, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
               !make_map(&g.tmLA, workspace, R, M, R, 64, shape.tn / 2, CU_TENSOR_MAP_SWIZZLE_128B)))
    return LYNX_ERR_CUDA;
  if (!set_y_map(&g, Y, M, N)) return LYNX_ERR_CUDA;
  g.rowscale = nullptr;
  g.scale_mode = SCALE_NONE;
  g.Y = Y;
  g.ldy = N;
  g.M = static_cast<int>(N);
  g.N = static_cast<int>(M);
  g.K = static_cast<int>(K);
  g.ctl = make_ctl();
  StageEvents prof(lora ? 3 : 2);
  if (cudaError_t e = prof.mark(0, st)) return cuda_status(e);
  if (lora) {
    if (int e = run_lora_down(X, LB, nullptr, workspace, M, K, st)) return e;
    if (cudaError_t e = prof.mark(1, st)) return cuda_status(e);
    if (cudaError_t e = launch_gemm_pair_transposed(true, shape, g, st)) return cuda_status(e);
    return cuda_status(prof.mark(2, st));
  }
  if (cudaError_t e = launch_gemm_pair_transposed(false, shape, g, st)) return cuda_status(e);
  return cuda_status(prof.mark(1, st));
}

int lynx_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return LYNX_ERR_CUDA;
  int* p = error_word_ptr();
  if (!p) return LYNX_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LYNX_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return LYNX_ERR_CUDA;
    return LYNX_ERR_TIMEOUT;
  }
  return LYNX_OK;
}

const char* lynx_status_string(int status) {
  switch (status) {
    case LYNX_OK: return "ok";
    case LYNX_ERR_NULL: return "null pointer argument";
    case LYNX_ERR_SHAPE: return "shape out of range (M,N >= 1; K >= 16, K % 16 == 0)";
    case LYNX_ERR_ALIGN: return "pointer not 16-byte aligned";
    case LYNX_ERR_WORKSPACE: return "workspace too small";
    case LYNX_ERR_CUDA: return "CUDA call failed";
    case LYNX_ERR_TIMEOUT: return "device-side wait timed out";
    case LYNX_ERR_UNSUPPORTED: return "unsupported configuration (LoRA rank must be 64)";
    case LYNX_ERR_TOO_LARGE: return "problem needs more scratch than lynx_linear_noalloc's fixed array";
    default: return "unknown status";
  }
}

int lynx_meta_to_canonical(const void* meta, uint8_t* canonical, int64_t M, int64_t K) {
  if (!meta || !canonical) return LYNX_ERR_NULL;
  if (M < 1 || K < 8 || K % 8 != 0) return LYNX_ERR_SHAPE;
  const uint8_t* base = static_cast<const uint8_t*>(meta);
  const int64_t blocks_k = meta_blocks_k(K);
  for (int64_t m = 0; m < M; ++m) {
    uint8_t* out = canonical + m * (K / 8);
    for (int64_t c = 0; c * kMetaChunkCols < K; ++c) {
      uint16_t lo, hi;
      std::memcpy(&lo, base + meta_half_offset(m, c, 0, blocks_k), 2);
      std::memcpy(&hi, base + meta_half_offset(m, c, 1, blocks_k), 2);
      const uint32_t word = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      for (int j = 0; j < 4 && c * kMetaChunkCols + 8 * j < K; ++j)  // byte j of the word = channels 8j..8j+7
        out[c * 4 + j] = static_cast<uint8_t>(word >> (8 * j));
    }
  }
  return LYNX_OK;
}

int lynx_linear_kernel_count(int64_t M, int64_t N, int64_t K, int64_t R) {
  (void)N;
  (void)R;
  if (M < 1 || K < 1) return 0;
  return 2;
}

void lynx_profile_next(void* const* events, int count) {
  t_prof_events = events;
  t_prof_count = count;
}

void lynx_debug_set_fault(int inject, uint64_t wait_ns) {
  g_inject.store(inject);
  g_wait_ns.store(wait_ns ? wait_ns : kDefaultWaitNs);
}

int lynx_debug_force_split(int split) {
  if (split < 0 || split > kMaxPrologueSplit) return LYNX_ERR_UNSUPPORTED;
  g_force_split.store(split);
  return LYNX_OK;
}

int lynx_debug_prologue_split(int64_t M, int64_t K) {
  if (check_mk(M, K) != LYNX_OK) return 0;
  return prologue_split(static_cast<int>(M), static_cast<int>(K));
}

int lynx_debug_force_tile(int tile_rows, int tile_cols) {
  if (tile_rows == 0 && tile_cols == 0) {
    g_force_tile.store(0);
    return LYNX_OK;
  }
  const PairShape shape{tile_rows / 256, tile_cols};
  if (tile_rows % 256 != 0 || !pair_shape_valid(true, shape)) return LYNX_ERR_UNSUPPORTED;
  g_force_tile.store(shape.rb << 16 | shape.tn);
  return LYNX_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- lynx_linear_noalloc
// Scratch for callers that cannot allocate: a file-scope device array, so the
// CUDA module loader reserves it with the library's device image.  Host code
// must not hand the symbol itself to a kernel (on the host it only names a
// host-side shadow); its device address comes from cudaGetSymbolAddress, looked
// up once per device with that device current.
namespace lynx {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[LYNX_NOALLOC_SCRATCH_BYTES];

void* noalloc_scratch() {
  static void* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace lynx

extern "C" int lynx_linear_noalloc(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M,
                                   int64_t N, int64_t K, int64_t R, void* stream) {
  // The arguments are checked as lynx_linear checks them (with a stand-in workspace that passes every workspace
  // check, never dereferenced), so that a bad pointer or shape reports its own status; only a valid problem is
  // then measured against the fixed array.
  static const uint8_t stand_in[16] __attribute__((aligned(16))) = {};
  if (int e = lynx::linear_arg_status(X, W, LA, LB, Y, M, N, K, R, stand_in, SIZE_MAX)) return e;
  if (lynx_workspace_bytes(M, N, K, R) > LYNX_NOALLOC_SCRATCH_BYTES) return LYNX_ERR_TOO_LARGE;
  void* ws = lynx::noalloc_scratch();
  if (!ws) return LYNX_ERR_CUDA;
  return lynx_linear(X, W, LA, LB, Y, M, N, K, R, ws, LYNX_NOALLOC_SCRATCH_BYTES, stream);
}
