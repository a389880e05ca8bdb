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
std::atomic<int> g_force_ksplit{0};  // 0: GEMM k-splits by tile count; else a forced count (one-row-block tiles)
std::atomic<int> g_force_dense_tile{0};  // 0: dense tile columns by problem shape; else 256 or 448
constexpr int kMaxKSplit = 4;
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

constexpr int kStreamK = LYNX_KSPLIT_STREAM;  // schedule code of stream-K; its partials use kMaxKSplit slots

// Partial slots per tile of a k-split schedule (1: none).
int split_stride(int sched) { return sched == kStreamK ? kMaxKSplit : sched; }

// Stream-K cuts a tile into at most kMaxKSplit parts where there are at least half as many tiles as CTA pairs and
// each tile has at least 8 k-steps: every pair's range then spans at least half a tile.
bool stream_k_fits(PairShape shape, int64_t M, int64_t N, int64_t K, int64_t clusters) {
  const int64_t nk = (K + 127) / 128;
  const int64_t tiles = ((M + 255) / 256) * ((N + shape.tn - 1) / shape.tn);
  return shape.rb == 1 && clusters >= 1 && 2 * tiles >= clusters && nk >= 8;
}

// k-split schedule of the sparse GEMM: only the one-row-block tiles (the ones few-tile problems take) split, and
// only when their tiles leave more than half of the CTA pairs idle; the split count (2-4, at least 8 k-steps per
// unit) that fills the waves best wins.  Stream-K is never chosen here: it was slower than the unsplit schedule at
// every few-tile shape measured (a tile's last part ends with its pair's range, so every pair finishes with a
// partial sum); the test hook selects it.  A forced count (test hook) is clamped to the k-steps.
int ksplit_auto(PairShape shape, int64_t M, int64_t N, int64_t K, int64_t clusters) {
  if (shape.rb != 1) return 1;
  const int64_t nk = (K + 127) / 128;
  if (clusters < 4) return 1;
  const int64_t tiles = ((M + 255) / 256) * ((N + shape.tn - 1) / shape.tn);
  if (2 * tiles > clusters) return 1;
  int best = 1;
  double best_eff = static_cast<double>(tiles) / static_cast<double>(clusters);
  for (int sp = 2; sp <= kMaxKSplit && nk >= 8 * sp; ++sp) {
    const int64_t units = tiles * sp, waves = (units + clusters - 1) / clusters;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * clusters);
    if (eff > best_eff + 0.05) {
      best = sp;
      best_eff = eff;
    }
  }
  return best;
}

int ksplit_for(PairShape shape, int64_t M, int64_t N, int64_t K) {
  if (shape.rb != 1) return 1;
  const int64_t nk = (K + 127) / 128;
  const int forced = g_force_ksplit.load();
  if (forced == kStreamK) return stream_k_fits(shape, M, N, K, sm_count() / 2) ? kStreamK : 1;
  if (forced) return static_cast<int>(forced < nk ? forced : nk);
  return ksplit_auto(shape, M, N, K, sm_count() / 2);
}

// Bytes of the split-K region for `splits` (0 for 1): fp32 partial tiles [tile][split][CTA][128 rb][tn], then one
// arrival counter per (tile, CTA), each part 256-byte aligned.
size_t split_bytes(PairShape shape, int64_t M, int64_t N, int splits, size_t* counters_off = nullptr) {
  if (splits <= 1) return 0;
  const int64_t tiles = ((M + 256 * shape.rb - 1) / (256 * shape.rb)) * ((N + shape.tn - 1) / shape.tn);
  const size_t partials = align256(static_cast<size_t>(tiles) * splits * 2 * 128 * shape.rb * shape.tn * 4);
  if (counters_off) *counters_off = partials;
  return partials + align256(static_cast<size_t>(tiles) * 2 * 4);
}

PairShape sparse_shape(int64_t M, int64_t N) {
  const int forced = g_force_tile.load();
  return forced ? PairShape{forced >> 16, forced & 0xFFFF} : pair_shape(true, static_cast<int>(M), static_cast<int>(N));
}

PairShape dense_shape(int64_t M, int64_t N) {
  const int forced = g_force_dense_tile.load();
  return forced ? PairShape{1, forced} : pair_shape(false, static_cast<int>(M), static_cast<int>(N));
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
      (LB && !make_map(&pa->tmLB, LB, K, kRank, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)))
    return LYNX_ERR_CUDA;
  pa->vals = static_cast<uint16_t*>(vals);
  pa->meta = static_cast<uint8_t*>(meta);
  pa->s = s;
  pa->T = T;
  pa->M = static_cast<int>(M);
  pa->K = static_cast<int>(K);
  pa->M_pad = static_cast<int>(round_up(M, kMetaRowPad));
  pa->nkb = static_cast<int>(meta_blocks_k(K));
  const int forced = g_force_split.load();
  pa->split = forced ? (forced < pa->nkb ? forced : pa->nkb) : prologue_split(pa->M, pa->K);
  pa->zero = nullptr;
  pa->nzero = 0;
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

namespace {

// The GELU epilogue's sparsified output for the next layer (hvals NULL: none) and the words it zeroes.
struct FuseOut {
  uint16_t* hvals = nullptr;
  uint8_t* hmeta = nullptr;
  float2* hnorm = nullptr;
  int slots = 0;
  unsigned int* zero = nullptr;
  int nzero = 0;
};

void set_fuse(PairArgs* g, const FuseOut* fo) {
  if (!fo) return;
  g->hvals = fo->hvals;
  g->hmeta = fo->hmeta;
  g->hnorm = fo->hnorm;
  g->hnorm_slots = fo->slots;
  g->zero = fo->zero;
  g->nzero = fo->nzero;
}

// Arguments of the sparse pair GEMM over compressed values / metadata / s / T' of an M x K activation.
int sparse_gemm_args(PairArgs* g, const void* vals, const void* meta, const float* s, const void* T, const void* W,
                     const void* LA, void* Y, int64_t M, int64_t N, int64_t K, int64_t R, PairShape shape) {
  std::memset(g, 0, sizeof(*g));
  const uint64_t meta_rows = 2 * static_cast<uint64_t>(meta_bytes(M, K) / kMetaChunkBytes);  // 1 KiB rows
  if (!make_map(&g->tmA, vals, K / 2, M, K / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g->tmB, W, K, N, K, 64, shape.tn / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g->tmMeta, meta, 256, meta_rows, 256, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_DATA_TYPE_UINT32) ||
      !make_map(&g->tmT, T, R, M, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g->tmLA, LA, R, N, R, 64, shape.tn / 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return LYNX_ERR_CUDA;
  if (!set_y_map(g, Y, M, N)) return LYNX_ERR_CUDA;
  g->rowscale = s;
  g->scale_mode = SCALE_MUL;
  g->Y = Y;
  g->ldy = N;
  g->M = static_cast<int>(M);
  g->N = static_cast<int>(N);
  g->K = static_cast<int>(K);
  g->splits = 1;
  g->ctl = make_ctl();
  return LYNX_OK;
}

// lynx_linear after its argument checks; gelu: the GELU epilogue, with fo its sparsified output (no split K).
int linear_impl(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M, int64_t N, int64_t K,
                int64_t R, void* workspace, size_t workspace_bytes, cudaStream_t st, bool gelu, const FuseOut* fo,
                const StageEvents& prof) {
  Workspace ws = carve(workspace, M, K, R);
  const PairShape shape = sparse_shape(M, N);
  PairArgs g;
  if (int e = sparse_gemm_args(&g, ws.vals, ws.meta, ws.s, ws.T, W, LA, Y, M, N, K, R, shape)) return e;
  // split K when the workspace holds the partials (else the unsplit schedule, which needs only the base part)
  const int sched = gelu ? 1 : ksplit_for(shape, M, N, K);
  int splits = split_stride(sched);
  size_t counters_off = 0;
  if (splits > 1 && workspace_bytes < ws.bytes + split_bytes(shape, M, N, splits, &counters_off)) splits = 1;
  g.splits = splits;
  g.stream_k = splits > 1 && sched == kStreamK;
  if (splits > 1) {
    g.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws.bytes);
    g.counters = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + ws.bytes + counters_off);
  }
  set_fuse(&g, fo);

  ProArgs pa;
  if (int e = make_prologue(&pa, X, LB, M, K, ws.vals, ws.meta, ws.s, ws.T)) return e;
  if (splits > 1) {  // the pre-pass zeroes the GEMM's arrival counters: the whole counter block split_bytes sized
    pa.zero = g.counters;
    pa.nzero = static_cast<int>((split_bytes(shape, M, N, splits) - counters_off) / 4);
  }
  if (cudaError_t e = prof.mark(0, st)) return cuda_status(e);
  if (cudaError_t e = launch_prologue(pa, true, st)) return cuda_status(e);
  if (cudaError_t e = prof.mark(1, st)) return cuda_status(e);
  if (cudaError_t e = launch_gemm_pair(true, true, shape, g, st, gelu)) return cuda_status(e);
  return cuda_status(prof.mark(2, st));
}

// lynx_linear_dense after its argument checks (gelu, fo as for linear_impl).
int dense_impl(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M, int64_t N, int64_t K,
               int64_t R, void* workspace, cudaStream_t st, bool gelu, const FuseOut* fo, const StageEvents& prof) {
  const bool lora = LA || LB;
  PairArgs g;
  std::memset(&g, 0, sizeof(g));
  // W and LA rows per load: this CTA's half of a 256-column tile, or of one 224-column half of a 448-column tile
  const PairShape shape = dense_shape(M, N);
  const uint32_t w_rows = shape.tn > 256 ? shape.tn / 4 : shape.tn / 2;
  if (!make_map(&g.tmA, X, K, M, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmB, W, K, N, K, 64, w_rows, CU_TENSOR_MAP_SWIZZLE_128B))
    return LYNX_ERR_CUDA;
  if (lora) {
    if (!make_map(&g.tmT, workspace, R, M, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&g.tmLA, LA, R, N, R, 64, w_rows, CU_TENSOR_MAP_SWIZZLE_128B))
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
  g.splits = 1;
  g.ctl = make_ctl();
  set_fuse(&g, fo);
  if (cudaError_t e = prof.mark(0, st)) return cuda_status(e);
  if (lora) {
    if (int e = run_lora_down(X, LB, nullptr, workspace, M, K, st)) return e;
    if (cudaError_t e = prof.mark(1, st)) return cuda_status(e);
    if (cudaError_t e = launch_gemm_pair(false, true, shape, g, st, gelu)) return cuda_status(e);
    return cuda_status(prof.mark(2, st));
  }
  if (cudaError_t e = launch_gemm_pair(false, false, shape, g, st, gelu)) return cuda_status(e);
  return cuda_status(prof.mark(1, st));
}

// ---------------------------------------------------------------- layer sequences and the fused MLP pair
constexpr int32_t kKnownFlags = LYNX_LAYER_SPARSE | LYNX_LAYER_GELU | LYNX_LAYER_FUSE_SPARSIFY;

bool is_sparse(const lynx_layer& l) { return (l.flags & LYNX_LAYER_SPARSE) != 0; }
bool is_gelu(const lynx_layer& l) { return (l.flags & LYNX_LAYER_GELU) != 0; }

size_t single_workspace_bytes(const lynx_layer& l) {
  if (is_sparse(l)) return is_gelu(l) ? carve(nullptr, l.M, l.K, l.R).bytes : lynx_workspace_bytes(l.M, l.N, l.K, l.R);
  return (l.LA || l.LB) ? lynx_dense_workspace_bytes(l.M, l.R) : 0;
}

int single_status(const lynx_layer& l, const void* ws, size_t ws_bytes) {
  if (l.flags & ~kKnownFlags) return LYNX_ERR_UNSUPPORTED;
  return is_sparse(l) ? linear_arg_status(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes)
                      : dense_arg_status(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes);
}

// Workspace plan of a fused pair (up = the GELU layer, dn = the sparse layer reading its output): the up layer's
// own part first, then the down layer's values, metadata, s and T', the norm partials, the LoRA pass's partials,
// one block of counters (the LoRA pass's, then the down GEMM's) that the up GEMM zeroes, and the down GEMM's
// split-K partials.
struct PairPlan {
  PairShape up_shape{1, 256}, dn_shape{1, 256};
  int slots = 0, fin_splits = 1, dn_splits = 1, fin_counters = 0, dn_counters = 0;
  bool dn_stream = false;  // the down GEMM runs the stream-K schedule (dn_splits = its partial slots)
  size_t up_bytes = 0, dn_off = 0, hnorm_off = 0, fin_off = 0, cnt_off = 0, dsplit_off = 0, total = 0;
};

bool fusable(const lynx_layer& up, const lynx_layer& dn) {
  return is_gelu(up) && (up.flags & LYNX_LAYER_FUSE_SPARSIFY) && is_sparse(dn) && !is_gelu(dn) && dn.X == up.Y &&
         dn.M == up.M && dn.K == up.N &&
         up.N % kMetaBlockCols == 0 && !(up.flags & ~kKnownFlags) && !(dn.flags & ~kKnownFlags);
}

PairPlan plan_pair(const lynx_layer& up, const lynx_layer& dn) {
  PairPlan p;
  const int64_t M = up.M;
  p.up_shape = is_sparse(up) ? sparse_shape(M, up.N) : dense_shape(M, up.N);
  p.up_bytes = is_sparse(up) ? carve(nullptr, M, up.K, up.R).bytes
                             : ((up.LA || up.LB) ? lynx_dense_workspace_bytes(M, up.R) : 0);
  p.slots = gelu_norm_slots(is_sparse(up), p.up_shape, static_cast<int>(up.N));
  p.fin_splits = lora_fin_splits(static_cast<int>(M), static_cast<int>(dn.K));
  p.dn_shape = sparse_shape(M, dn.N);
  const int dn_sched = ksplit_for(p.dn_shape, M, dn.N, dn.K);
  p.dn_splits = split_stride(dn_sched);
  p.dn_stream = dn_sched == kStreamK;
  p.fin_counters = p.fin_splits > 1 ? lora_fin_counters(static_cast<int>(M)) : 0;
  size_t dn_cnt_off = 0;
  const size_t dsplit = split_bytes(p.dn_shape, M, dn.N, p.dn_splits, &dn_cnt_off);
  p.dn_counters = p.dn_splits > 1 ? static_cast<int>((dsplit - dn_cnt_off) / 4) : 0;
  size_t off = align256(p.up_bytes);
  p.dn_off = off;
  off += carve(nullptr, M, dn.K, dn.R).bytes;
  p.hnorm_off = off;
  off += align256(static_cast<size_t>(M) * p.slots * sizeof(float2));
  p.fin_off = off;
  off += align256(lora_fin_partial_bytes(static_cast<int>(M), p.fin_splits));
  p.cnt_off = off;
  off += align256(static_cast<size_t>(p.fin_counters + p.dn_counters) * 4);
  p.dsplit_off = off;
  off += p.dn_splits > 1 ? dn_cnt_off : 0;  // the down GEMM's partials (its counters live in the block above)
  p.total = off;
  return p;
}

int run_pair(const lynx_layer& up, const lynx_layer& dn, const PairPlan& p, void* workspace, cudaStream_t st) {
  uint8_t* base = static_cast<uint8_t*>(workspace);
  const int64_t M = up.M;
  Workspace dws = carve(base + p.dn_off, M, dn.K, dn.R);
  unsigned int* counters = reinterpret_cast<unsigned int*>(base + p.cnt_off);
  FuseOut fo;
  fo.hvals = static_cast<uint16_t*>(dws.vals);
  fo.hmeta = static_cast<uint8_t*>(dws.meta);
  fo.hnorm = reinterpret_cast<float2*>(base + p.hnorm_off);
  fo.slots = p.slots;
  if (p.fin_counters + p.dn_counters > 0) {
    fo.zero = counters;
    fo.nzero = p.fin_counters + p.dn_counters;
  }
  const StageEvents none(-1);
  const int e = is_sparse(up) ? linear_impl(up.X, up.W, up.LA, up.LB, up.Y, M, up.N, up.K, up.R, base, p.up_bytes, st,
                                            true, &fo, none)
                              : dense_impl(up.X, up.W, up.LA, up.LB, up.Y, M, up.N, up.K, up.R, base, st, true, &fo,
                                           none);
  if (e) return e;
  // the down layer's LoRA down-projection over H = up.Y and its row scale, from the epilogue's norm partials
  FinArgs f;
  std::memset(&f, 0, sizeof(f));
  if (!make_map(&f.tmH, dn.X, dn.K, M, dn.K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&f.tmLB, dn.LB, dn.K, kRank, dn.K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return LYNX_ERR_CUDA;
  f.hnorm = fo.hnorm;
  f.slots = p.slots;
  f.s = dws.s;
  f.T = dws.T;
  f.partials = reinterpret_cast<float*>(base + p.fin_off);
  f.counters = counters;
  f.M = static_cast<int>(M);
  f.K = static_cast<int>(dn.K);
  f.splits = p.fin_splits;
  f.ctl = make_ctl();
  if (cudaError_t ce = launch_lora_fin(f, st)) return cuda_status(ce);
  // the down layer's sparse GEMM on the values and metadata the up layer's epilogue wrote
  PairArgs g;
  if (int ge = sparse_gemm_args(&g, dws.vals, dws.meta, dws.s, dws.T, dn.W, dn.LA, dn.Y, M, dn.N, dn.K, dn.R,
                                p.dn_shape))
    return ge;
  g.splits = p.dn_splits;
  g.stream_k = p.dn_splits > 1 && p.dn_stream;
  if (p.dn_splits > 1) {
    g.partials = reinterpret_cast<float*>(base + p.dsplit_off);
    g.counters = counters + p.fin_counters;
  }
  return cuda_status(launch_gemm_pair(true, true, p.dn_shape, g, st));
}

int run_single(const lynx_layer& l, void* ws, size_t ws_bytes, cudaStream_t st) {
  const StageEvents none(-1);
  if (is_sparse(l))
    return linear_impl(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, ws_bytes, st, is_gelu(l), nullptr, none);
  return dense_impl(l.X, l.W, l.LA, l.LB, l.Y, l.M, l.N, l.K, l.R, ws, st, is_gelu(l), nullptr, none);
}

}  // namespace

int seq_status(const lynx_layer* layers, int32_t n, const void* ws, size_t ws_bytes, int32_t* failed) {
  if (failed) *failed = -1;
  if (n > 0 && !layers) return LYNX_ERR_NULL;
  if (n < 0) return LYNX_ERR_SHAPE;
  for (int32_t i = 0; i < n; ++i) {
    if (int e = single_status(layers[i], ws, ws_bytes)) {
      if (failed) *failed = i;
      return e;
    }
  }
  return LYNX_OK;
}

size_t seq_workspace_bytes(const lynx_layer* layers, int32_t n) {
  if (!layers || n < 1) return 0;
  size_t b = 0;
  for (int32_t i = 0; i < n; ++i) {
    size_t w = single_workspace_bytes(layers[i]);
    if (i + 1 < n && fusable(layers[i], layers[i + 1])) {
      const size_t f = plan_pair(layers[i], layers[i + 1]).total;
      if (f > w) w = f;
    }
    if (w > b) b = w;
  }
  return b;
}

int seq_pair_offsets(const lynx_layer* layers, int32_t n, int32_t i, size_t* out) {
  if (!layers || !out) return LYNX_ERR_NULL;
  if (i < 0 || i + 1 >= n || !fusable(layers[i], layers[i + 1])) return LYNX_ERR_UNSUPPORTED;
  const PairPlan p = plan_pair(layers[i], layers[i + 1]);
  const Workspace d = carve(nullptr, layers[i].M, layers[i + 1].K, layers[i + 1].R);
  out[0] = p.dn_off + reinterpret_cast<uintptr_t>(d.vals);
  out[1] = p.dn_off + reinterpret_cast<uintptr_t>(d.meta);
  out[2] = p.dn_off + reinterpret_cast<uintptr_t>(d.s);
  out[3] = p.dn_off + reinterpret_cast<uintptr_t>(d.T);
  out[4] = p.total;
  return LYNX_OK;
}

int seq_enqueue(const lynx_layer* layers, int32_t n, void* ws, size_t ws_bytes, cudaStream_t st) {
  for (int32_t i = 0; i < n; ++i) {
    if (i + 1 < n && fusable(layers[i], layers[i + 1])) {
      const PairPlan p = plan_pair(layers[i], layers[i + 1]);
      if (p.total <= ws_bytes) {
        if (int e = run_pair(layers[i], layers[i + 1], p, ws, st)) return e;
        ++i;
        continue;
      }
    }
    if (int e = run_single(layers[i], ws, ws_bytes, st)) return e;
  }
  return LYNX_OK;
}

}  // namespace lynx

using namespace lynx;

extern "C" {

size_t lynx_meta_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 1) return 0;
  return static_cast<size_t>(meta_bytes(M, K));
}

size_t lynx_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R) {
  if (M < 1 || K < 1 || R < 0) return 0;
  size_t b = carve(nullptr, M, K, R).bytes;
  if (N >= 1 && N <= (int64_t(1) << 24) && M <= 65535LL * 128) {
    const PairShape shape = sparse_shape(M, N);
    b += split_bytes(shape, M, N, split_stride(ksplit_for(shape, M, N, K)));
  }
  return b;
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
  StageEvents prof(3);
  return linear_impl(X, W, LA, LB, Y, M, N, K, R, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false,
                     nullptr, prof);
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
  StageEvents prof((LA || LB) ? 3 : 2);
  return dense_impl(X, W, LA, LB, Y, M, N, K, R, workspace, static_cast<cudaStream_t>(stream), false, nullptr, prof);
}

int lynx_linear_fused(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M, int64_t N,
                      int64_t K, int64_t R, void* workspace, size_t workspace_bytes, void* stream) {
  if (!LA || !LB || !workspace) return LYNX_ERR_NULL;
  if (int e = dense_arg_status(X, W, LA, LB, Y, M, N, K, R, workspace, workspace_bytes)) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StageEvents prof(3);
  PairArgs g;
  std::memset(&g, 0, sizeof(g));
  if (!make_map(&g.tmA, X, K, M, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmB, W, K, N, K, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&g.tmLA, LA, R, N, R, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return LYNX_ERR_CUDA;
  if (!set_y_map(&g, Y, M, N)) return LYNX_ERR_CUDA;
  g.scale_mode = SCALE_NONE;  // s comes from the GEMM's own row sums
  g.Y = Y;
  g.ldy = N;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.splits = 1;
  g.lora_t = static_cast<const uint16_t*>(workspace);
  g.ctl = make_ctl();
  if (cudaError_t e = prof.mark(0, st)) return cuda_status(e);
  if (int e = run_lora_down(X, LB, nullptr, workspace, M, K, st)) return e;  // T = X LB^T, not divided by s
  if (cudaError_t e = prof.mark(1, st)) return cuda_status(e);
  if (cudaError_t e = launch_gemm_pair_f1(g, st)) return cuda_status(e);
  return cuda_status(prof.mark(2, st));
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

int lynx_debug_force_ksplit(int splits) {
  if ((splits < 0 || splits > kMaxKSplit) && splits != kStreamK) return LYNX_ERR_UNSUPPORTED;
  g_force_ksplit.store(splits);
  return LYNX_OK;
}

int lynx_debug_linear_ksplit(int64_t M, int64_t N, int64_t K) {
  if (check_mk(M, K) != LYNX_OK || check_n(M, N) != LYNX_OK) return 0;
  return ksplit_for(sparse_shape(M, N), M, N, K);
}

int lynx_debug_auto_plan(int sparse, int64_t M, int64_t N, int64_t K, int sms, int32_t* plan) {
  if (!plan) return LYNX_ERR_NULL;
  if (check_mk(M, K) != LYNX_OK || check_n(M, N) != LYNX_OK || sms < 2) return LYNX_ERR_SHAPE;
  const int64_t clusters = sms / 2;
  const PairShape shape = pair_shape_for(sparse != 0, static_cast<int>(M), static_cast<int>(N), clusters);
  plan[0] = 256 * shape.rb;
  plan[1] = shape.tn;
  plan[2] = sparse ? ksplit_auto(shape, M, N, K, clusters) : 1;
  return LYNX_OK;
}

int lynx_debug_dense_tile(int64_t M, int64_t N) {
  if (M < 1 || M > kMaxM || check_n(M, N) != LYNX_OK) return 0;
  return dense_shape(M, N).tn;
}

int lynx_debug_force_dense_tile(int tile_cols) {
  if (tile_cols != 0 && !pair_shape_valid(false, PairShape{1, tile_cols})) return LYNX_ERR_UNSUPPORTED;
  g_force_dense_tile.store(tile_cols);
  return LYNX_OK;
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
