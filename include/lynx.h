/*
 * lynx.h -- C ABI of the RT-Lynx 2:4 activation-sparse linear layer (sm_103a).
 *
 * The layer (RT-Lynx page, aitrends.kr article 60737, Method / Code examples):
 *
 *     Y = S(X) W^T + X (LA LB)^T,     S(X) = s * X~,
 *     X~ = the two largest-|x| entries of every 4 consecutive input channels of
 *          each token row (ties to the lower channel index),
 *     s  = ||X||_2 / ||X~||_2 per row (s = 1 when X~ is all zero),
 *
 * with a rank-R (R = 64) LoRA branch on the dense X.
 *
 * Conventions shared by every entry point:
 *   - Matrices are row-major device arrays of bf16 (stored as 16-bit words)
 *     unless stated: X is M x K, W is N x K (nn.Linear layout), LA is N x R,
 *     LB is R x K, Y is M x N.  Every pointer must be 16-byte aligned.
 *   - K must be a positive multiple of 16; M and N are any value >= 1;
 *     R must be 64 wherever a LoRA branch is computed.
 *   - All memory is owned by the caller.  The library allocates nothing;
 *     scratch space is passed in as `workspace`.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work and returns; results are ready when the stream
 *     is.
 *   - Return value: LYNX_OK or a negative lynx_status.  Argument errors are
 *     detected on the host and returned before anything is enqueued.
 *     Device-side failures (a bounded wait that ran out) are recorded in a
 *     device error word and returned by lynx_sync_status.
 *   - No entry point aborts the process or traps on the device.
 */
#ifndef LYNX_H_
#define LYNX_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LYNX_API __attribute__((visibility("default")))
#else
#define LYNX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LYNX_OK = 0,
  LYNX_ERR_NULL = -1,        /* a required pointer is NULL */
  LYNX_ERR_SHAPE = -2,       /* M, N, K or R out of range, or K % 16 != 0.  Ranges:
                                1 <= M <= 8388480 (65535 * 128), 1 <= N <= 2^24,
                                16 <= K <= 2^20, M * N <= 2^40, R >= 1 */
  LYNX_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
  LYNX_ERR_WORKSPACE = -4,   /* workspace smaller than lynx_*workspace_bytes() */
  LYNX_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed */
  LYNX_ERR_TIMEOUT = -6,     /* a device-side bounded wait ran out */
  LYNX_ERR_UNSUPPORTED = -7, /* valid but not implemented (R != 64) */
  LYNX_ERR_TOO_LARGE = -8    /* needs more scratch than lynx_linear_noalloc owns */
} lynx_status;

/* Bytes of 2:4 metadata for an M x K activation:
 *     (ceil(M/256) * 2) * ceil(K/128) * 2048.
 * Layout (the one the sparse GEMM copies into tensor memory): one 2 KiB chunk
 * per (128-row block, 128-channel block), row blocks outermost.  A chunk holds
 * 128 lanes of 16 bytes: little-endian 32-bit word w of a lane is the tensor
 * memory word of that lane for channels 32w..32w+31 of the block.  A row's
 * word for 32 channels carries group g (channels 4g..4g+3 of them) in bits
 * 4g..4g+3 as i0 | (i1 << 2), i0 < i1 the kept positions.  Inside each
 * 16-row block the words of rows r and r+8 are stored by 16-bit halves: lane
 * 16b+i (i < 8) holds the low halves of rows 16b+i (bits 0-15) and 16b+8+i
 * (bits 16-31), lane 16b+8+i their high halves -- the order in which
 * tcgen05.mma.sp reads metadata from tensor memory.  Padding rows and
 * channels (up to multiples of 256 and 128) hold the pattern of an all-zero
 * group (0x4). */
LYNX_API size_t lynx_meta_bytes(int64_t M, int64_t K);

/* Workspace bytes needed by lynx_linear on the current device: compressed
 * values (M x K/2 bf16), metadata (lynx_meta_bytes), s (M fp32) and the M x R
 * LoRA intermediate T' (bf16), each 256-byte aligned -- the base part --
 * and, for problems whose output tiles would leave a large share of the GPU
 * idle, the split-K region of the sparse GEMM: fp32 partial tiles and one
 * arrival counter per tile and CTA (this part depends on N).  lynx_linear
 * accepts any workspace that holds the base part; it runs the split-K
 * schedule only when the whole amount is there. */
LYNX_API size_t lynx_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R);

/* Workspace bytes needed by lynx_linear_dense when a LoRA branch is given
 * (the M x R intermediate X LB^T); 0 suffices without LoRA. */
LYNX_API size_t lynx_dense_workspace_bytes(int64_t M, int64_t R);

/* Online 2:4 sparsification: S(X) in the form the sparse tensor core consumes.
 * (RT-Lynx page, Method: Top-K based 2:4 activation selection, done online,
 * handed to the kernel in the sparse-tensor-core format; Code examples,
 * first formula for s.)
 *   X    [in]  M x K bf16.
 *   vals [out] M x K/2 bf16: the two kept entries of each group, lower index first.
 *   meta [out] lynx_meta_bytes(M, K) bytes, layout above.
 *   s    [out] M fp32: ||X_m|| / ||X~_m|| (1 for a row whose kept entries are zero).
 * The values are copies of the inputs; s is applied later, by the GEMM epilogue. */
LYNX_API int lynx_sparsify(const void* X, int64_t M, int64_t K, void* vals, void* meta, float* s, void* stream);

/* LoRA down-projection of the dense activation:
 *   T[m, r] = bf16( sum_k X[m,k] LB[r,k] / s[m] )      (s == NULL: no division)
 *   X [in] M x K, LB [in] R x K, s [in] M fp32 or NULL, T [out] M x R bf16; R = 64.
 * (RT-Lynx page, Method: Yr = X (LA LB)^T; the division by s lets the fused
 * epilogue scale the whole accumulator by s.) */
LYNX_API int lynx_lora_down(const void* X, const void* LB, const float* s, void* T, int64_t M, int64_t K, int64_t R,
                   void* stream);

/* Fused first half of lynx_linear: one pass over X gives S(X) (exactly as
 * lynx_sparsify) and, with LB, the LoRA down-projection divided by s:
 *   T[m, r] = bf16( sum_k X[m,k] LB[r,k] / s[m] ),  R = 64.
 * (RT-Lynx page, Method: top-2-of-4 selection and the row scale s; CUDA
 * kernel optimisation: the low-rank branch reuses the activation tile.)
 *   X [in] M x K bf16; LB [in] R x K bf16 or NULL (then T must be NULL);
 *   vals, meta, s [out] as for lynx_sparsify; T [out] M x R bf16 or NULL.
 * One kernel: a row block's channels may be shared by a cluster of CTAs, whose
 * partial sums are added in a fixed order through distributed shared memory. */
LYNX_API int lynx_sparsify_lora(const void* X, const void* LB, int64_t M, int64_t K, int64_t R, void* vals,
                                void* meta, float* s, void* T, void* stream);

/* The full RT-Lynx sparse linear: Y = bf16( s * (X~ W^T) + (X LB^T) LA^T ).
 *   X [in] M x K, W [in] N x K, LA [in] N x R, LB [in] R x K, Y [out] M x N bf16.
 *   workspace: >= lynx_workspace_bytes(M, N, K, R) bytes of device memory,
 *   16-byte aligned, not shared with a concurrent call.
 * Enqueues two kernels: the fused sparsify + LoRA down-projection pass
 * (lynx_sparsify_lora) and the tcgen05 2:4-sparse GEMM whose extra K-steps
 * accumulate T' LA^T into the same tensor-memory accumulator, with s applied
 * in the epilogue.
 * (RT-Lynx page, Method and CUDA kernel optimisation.) */
LYNX_API int lynx_linear(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M, int64_t N,
                int64_t K, int64_t R, void* workspace, size_t workspace_bytes, void* stream);

/* The same Y = S(X) W^T + X (LA LB)^T with the 2:4 selection inside the GEMM (the page's own design, "RT-Lynx"
 * page, CUDA kernel optimisation: 2:4 activations built directly in registers): no compressed copy of X goes
 * through global memory.  Enqueues the LoRA down-projection T = X LB^T (into workspace) and one GEMM on
 * 256 x 256 tiles whose epilogue warps, while a tile's k-steps stream in, select the top two of every four
 * channels of the dense X tile, write the compressed values and metadata into shared memory for the sparse
 * MMAs, and sum x^2 and kept x^2 over the row; at the tile's last step they form s and T' = bf16(T / s).
 *   Arguments as for lynx_linear (LA, LB, workspace required; R = 64); workspace: >= lynx_dense_workspace_bytes(M,
 *   R) bytes (T).  Results agree with lynx_linear within the stated tolerance: s is summed in another order and
 *   T is rounded to bf16 before the division by s.  Every column tile repeats its rows' selection, so this
 *   path trades the sparsify pass's global-memory round trip for N / 256 selections per row. */
LYNX_API int lynx_linear_fused(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M,
                               int64_t N, int64_t K, int64_t R, void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed scratch array behind lynx_linear_noalloc, per GPU. */
#define LYNX_NOALLOC_SCRATCH_BYTES (64u << 20)

/* lynx_linear for callers that must not allocate device memory.  (No
 * counterpart on the RT-Lynx page: this is a deployment convenience.)
 *
 * Some callers cannot call cudaMalloc or any allocator on the path that runs
 * the layer: a request loop in a serving process that must never stall on
 * an allocation (cudaMalloc can synchronise the device), or a plug-in inside
 * another runtime that owns every byte of device memory and gives its
 * plug-ins none.  This entry point takes the same arguments as lynx_linear
 * minus the workspace: its scratch is one array of LYNX_NOALLOC_SCRATCH_BYTES
 * in the library's own device image, which every GPU that loads the library
 * holds until the process exits.  It allocates nothing itself and calls no
 * allocating routine.
 *
 * Limits and rules:
 *   - arguments are checked as lynx_linear checks them (NULL, shape, rank,
 *     alignment statuses first); a valid problem whose
 *     lynx_workspace_bytes(M, N, K, R) exceeds LYNX_NOALLOC_SCRATCH_BYTES is
 *     then rejected with LYNX_ERR_TOO_LARGE, before anything is enqueued;
 *   - the first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture;
 *   - the CUDA runtime loads the library's device code on a device lazily, at
 *     the first lynx_* call that launches or looks up a symbol there, and the
 *     array is reserved at that moment: that first call can allocate and
 *     synchronise.  A caller that must never stall makes one warm-up call per
 *     device (any lynx_* call that enqueues work, or this entry point on a
 *     small problem) outside its request loop and before any capture;
 *   - every call on a device shares the one array and leaves its contents
 *     behind (nothing in it has to start at zero), so calls whose kernels
 *     overlap on the GPU -- on different streams, or from different threads --
 *     race and corrupt each other's results: order them on one stream. */
LYNX_API int lynx_linear_noalloc(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M,
                                 int64_t N, int64_t K, int64_t R, void* stream);

/* A selectively skipped (dense) layer: Y = bf16( X W^T [+ (X LB^T) LA^T] ).
 * LA and LB are both NULL (no LoRA) or both given (then R = 64 and the
 * workspace must hold lynx_dense_workspace_bytes(M, R) bytes).
 * (RT-Lynx page, Method: Selective Layer Skipping.) */
LYNX_API int lynx_linear_dense(const void* X, const void* W, const void* LA, const void* LB, void* Y, int64_t M,
                      int64_t N, int64_t K, int64_t R, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- layer sequences
 * A DiT block stack with selective layer skipping (RT-Lynx page, Method:
 * Selective Layer Skipping) is a fixed sequence of sparse and dense linears.
 * These calls run such a sequence in order on one stream, or capture it once
 * into a CUDA graph that replays every kernel of it with one host call.
 * (The graph is a deployment convenience, not part of the page's method.) */

/* One layer.  flags & LYNX_LAYER_SPARSE: Y = lynx_linear(X, W, LA, LB) (LA
 * and LB required, R = 64); otherwise Y = lynx_linear_dense(X, W, LA, LB) (LA
 * and LB both NULL, or both given with R = 64).  flags & LYNX_LAYER_GELU: the
 * layer's bf16 result y is passed through the exact-erf GELU, Y = bf16(GELU(y))
 * (the activation between a DiT MLP's up and down projections).  Device
 * pointers and layouts as for those calls.  A layer may read the Y of an
 * earlier layer of the same sequence.
 *
 * The fused MLP pair: a GELU layer with LYNX_LAYER_FUSE_SPARSIFY, followed by
 * a sparse layer whose X is that Y (same pointer and M, its K equal to the
 * GELU layer's N, N % 128 == 0), runs as one pair ("RT-Lynx" page, CUDA
 * kernel optimisation: one execution path for the online sparsification):
 * the GELU layer's epilogue also writes the 2:4 values, metadata and partial
 * row norms of its output, and the sparse layer's sparsify pass is replaced
 * by a LoRA down-projection that finishes s and T'.  Y of the GELU layer is
 * still written; the results equal those of the two layers run one by one, up
 * to the fp32 summation order of the row norms.  The fused pair needs more
 * workspace (lynx_layers_workspace_bytes counts it); with less, or without the
 * flag, the pair runs as two layers (the GELU epilogue, then the sparse
 * layer's own sparsify pass), which measures faster on GB300. */
#define LYNX_LAYER_SPARSE 1
#define LYNX_LAYER_GELU 2
#define LYNX_LAYER_FUSE_SPARSIFY 4
typedef struct {
  int32_t flags;
  const void* X;
  const void* W;
  const void* LA;
  const void* LB;
  void* Y;
  int64_t M, N, K, R;
} lynx_layer;

/* Workspace for a sequence: the largest any one layer, or fused MLP pair,
 * needs (they run one after another and reuse it).  0 if layers is NULL or
 * n < 1. */
LYNX_API size_t lynx_layers_workspace_bytes(const lynx_layer* layers, int32_t n);

/* Enqueues the n layers in order on `stream` (asynchronous).  Every layer is
 * checked on the host first: if one fails, nothing is enqueued, its status is
 * returned and its index is stored in *failed_layer (when failed_layer is not
 * NULL; -1 otherwise).  Flags other than the three above give
 * LYNX_ERR_UNSUPPORTED.  n = 0 enqueues nothing and returns LYNX_OK. */
LYNX_API int lynx_run_layers(const lynx_layer* layers, int32_t n, void* workspace, size_t workspace_bytes,
                             void* stream, int32_t* failed_layer);

/* An instantiated CUDA graph of a layer sequence. */
typedef struct lynx_graph_s* lynx_graph;

/* Captures lynx_run_layers(layers, n, workspace, workspace_bytes) on a
 * private stream and instantiates the graph into *graph_out.  Pointers,
 * shapes and the workspace are baked in: the caller keeps every buffer alive
 * and at the same address while the graph exists (their contents may change
 * between launches).  Returns the first failing layer's status (nothing
 * captured) as lynx_run_layers does, LYNX_ERR_SHAPE for n < 1, LYNX_ERR_NULL
 * for a NULL layers or graph_out, LYNX_ERR_CUDA if capture or instantiation
 * fails.  Call it once before any other capture is open on this thread. */
LYNX_API int lynx_graph_create(const lynx_layer* layers, int32_t n, void* workspace, size_t workspace_bytes,
                               lynx_graph* graph_out, int32_t* failed_layer);

/* Enqueues one replay of the whole sequence on `stream` (asynchronous).
 * Replays on one stream run in order; concurrent replays of one graph, or of
 * graphs sharing a workspace, race. */
LYNX_API int lynx_graph_launch(lynx_graph graph, void* stream);

/* Frees the graph (NULL is a no-op).  Call it after the replays it enqueued
 * have completed (e.g. after lynx_sync_status on their stream). */
LYNX_API int lynx_graph_destroy(lynx_graph graph);

/* The weight-2:4 comparator: Y = bf16( X W~^T [+ (X LB^T) LA^T] ), W~ keeping
 * the two largest |w| of every 4 consecutive input channels of each row of W
 * (ties to the lower index), with no rescaling.  (RT-Lynx page, Main results:
 * the "Sparse Weight" baseline; Key idea: weight against activation
 * sparsity.  Provided as a speed comparator of the same tensor-core path.)
 *   X [in] M x K bf16; Y [out] M x N bf16.
 *   Wvals, Wmeta [in]: W~ compressed as lynx_sparsify(W, N, K, ...) writes it
 *     (its s output is not used); prune once, reuse for every call.
 *   LA, LB: both NULL (no LoRA) or both given (R = 64; the workspace then holds
 *     lynx_dense_workspace_bytes(M, R) bytes).
 * Enqueues the LoRA down-projection (with LoRA) and one 2:4-sparse GEMM whose
 * sparse operand is W~: its accumulator tile is Y^T, written out transposed. */
LYNX_API int lynx_linear_wsparse(const void* X, const void* Wvals, const void* Wmeta, const void* LA, const void* LB,
                                 void* Y, int64_t M, int64_t N, int64_t K, int64_t R, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Waits for `stream`, then reads and clears the device error word of the
 * current device.  Returns LYNX_OK, LYNX_ERR_TIMEOUT or LYNX_ERR_CUDA. */
LYNX_API int lynx_sync_status(void* stream);

/* Static, human-readable text of a status code. */
LYNX_API const char* lynx_status_string(int status);

/* Host-side helper: converts metadata in the layout above (a host copy of
 * lynx_meta_bytes(M, K) bytes) to the canonical row-major M x K/8 bytes,
 * byte j = nibble(group 2j) | nibble(group 2j+1) << 4.  K % 8 == 0. */
LYNX_API int lynx_meta_to_canonical(const void* meta, uint8_t* canonical, int64_t M, int64_t K);

/* Number of kernels lynx_linear enqueues for these sizes on the current
 * device: 2 (the fused sparsify + LoRA down-projection pass and the sparse
 * GEMM). */
LYNX_API int lynx_linear_kernel_count(int64_t M, int64_t N, int64_t K, int64_t R);

/* Stage-timing hook.  The next lynx_linear or lynx_linear_dense call made
 * from this host thread records events[0] on its stream before its first
 * stage and events[i] right after its i-th stage; count must be the number
 * of stages + 1 (3 for lynx_linear: the fused sparsify + LoRA down-projection
 * pass, the sparse GEMM; 3 for lynx_linear_dense with LoRA, 2 without).  The events are
 * cudaEvent_t handles owned by the caller.  The setting is used by that one
 * call and then cleared; a count that does not match is ignored. */
LYNX_API void lynx_profile_next(void* const* events, int count);

/* Tensor-core rate microbenchmark: every SM issues `iters` back-to-back
 * instructions of shape 128 x 256 with operands resident in shared memory:
 * mode 0 tcgen05.mma (dense), mode 1 tcgen05.mma.sp (2:4 sparse A, metadata
 * resident in tensor memory), mode 2 tcgen05.mma.sp each preceded by the
 * tcgen05.cp of its 2 KiB metadata chunk, mode 3 tcgen05.mma.sp with a
 * tcgen05.commit after every two MMAs, mode 4 with two commits after every
 * four MMAs, mode 5 tcgen05.mma.sp with A in 64-byte rows (64-byte swizzle);
 * modes 6-8 run on CTA pairs (tcgen05 cta_group::2, M = 256 over two SMs):
 * 6 sparse with 128-byte-swizzled A, 7 sparse with 64-byte-swizzled A,
 * 8 dense.  Writes the dense-equivalent rate (2*M*N*K per instruction,
 * K = 16 dense or 32 logical sparse) in TFLOP/s and in MACs per SM clock.
 * Other modes return LYNX_ERR_UNSUPPORTED.  Synchronises `stream`. */
LYNX_API int lynx_mma_rate(int mode, int iters, double* tflops, double* macs_per_clock, void* stream);

/* Test hook.  For layers i and i + 1 of a sequence that run as a fused MLP pair, writes the byte offsets in the
 * sequence's workspace of the sparse layer's compressed values, metadata, s and T' (written by the pair's first
 * two kernels) to offsets[0..3] and the pair's workspace bytes to offsets[4].  LYNX_ERR_UNSUPPORTED when the two
 * layers do not fuse, LYNX_ERR_NULL for NULL arguments. */
LYNX_API int lynx_debug_pair_offsets(const lynx_layer* layers, int32_t n, int32_t i, size_t* offsets);

/* Test hook.  inject = 1 makes the next GEMM launches never deliver their
 * first pipeline stage, so their bounded waits run out after wait_ns
 * nanoseconds and lynx_sync_status reports LYNX_ERR_TIMEOUT.  inject = 0
 * restores normal operation; wait_ns = 0 restores the default bound (2 s). */
LYNX_API void lynx_debug_set_fault(int inject, uint64_t wait_ns);

/* Test hook.  split = 1 .. 16 makes the sparsify pass of every later call run each 128-row block on a
 * cluster of that many CTAs (at most one per 128-channel block; a size the GPU cannot hold makes the launch
 * fail with LYNX_ERR_CUDA); 0 restores the automatic choice.  Returns LYNX_OK, or LYNX_ERR_UNSUPPORTED
 * (setting unchanged) for other values. */
LYNX_API int lynx_debug_force_split(int split);

/* The cluster size the sparsify pass picks on the current device for an M x K activation (1 = no cluster:
 * each CTA owns whole rows); 0 for sizes out of range. */
LYNX_API int lynx_debug_prologue_split(int64_t M, int64_t K);

/* Schedule code of the sparse GEMM's stream-K schedule ("RT-Lynx" page, Method, CUDA kernel optimisation: the
 * page splits its sparse GEMM's work stream-K fashion): CTA pair c of P takes the contiguous range
 * [c T / P, (c + 1) T / P) of all T = tiles x k-steps, so a tile is cut wherever a range ends; the pairs that
 * share a tile leave fp32 partials and the last to finish adds them in k order.  Only the test hook selects it:
 * it was slower than the unsplit schedule at every few-tile shape measured. */
#define LYNX_KSPLIT_STREAM 8

/* Test hook.  splits = 1 .. 4 makes the sparse GEMM of every later lynx_linear call whose tile shape has one row
 * block per CTA (256 x 256 or 256 x 192) split each tile's k-steps over that many work units (clamped to the tile's
 * 128-channel steps; 1 = never split); LYNX_KSPLIT_STREAM selects the stream-K schedule for those tiles wherever
 * it applies (at least half as many tiles as CTA pairs and 8 k-steps per tile; elsewhere no split); 0 restores
 * the automatic choice.  lynx_workspace_bytes follows the setting.  Returns LYNX_OK, or LYNX_ERR_UNSUPPORTED
 * (setting unchanged) for other values. */
LYNX_API int lynx_debug_force_ksplit(int splits);

/* The k-split schedule lynx_linear picks on the current device for these sizes (1 = no split, 2 .. 4 = that many
 * equal k-ranges per tile, LYNX_KSPLIT_STREAM = stream-K); 0 for sizes out of range. */
LYNX_API int lynx_debug_linear_ksplit(int64_t M, int64_t N, int64_t K);

/* Test hook.  Makes lynx_linear (and lynx_linear_wsparse, whose tile rows are output columns) use sparse
 * pair tiles of tile_rows x tile_cols for every shape: 512 x 224,
 * 512 x 192, 256 x 256 or 256 x 192 (all must give the same result); 0 x 0 restores the automatic choice by
 * shape.
 * Returns LYNX_OK, or LYNX_ERR_UNSUPPORTED (setting unchanged) for any other shape. */
LYNX_API int lynx_debug_force_tile(int tile_rows, int tile_cols);

/* Test hook.  Makes the dense GEMM (lynx_linear_dense and the dense layers of lynx_run_layers and the graphs
 * built after the call) use 256 x tile_cols pair tiles for every shape: 256 (one 256-column MMA per K step) or 448
 * (two 224-column MMAs sharing one read of X); both give the same result.  0 restores the automatic choice by
 * shape.  Returns LYNX_OK, or LYNX_ERR_UNSUPPORTED (setting unchanged) for any other value. */
LYNX_API int lynx_debug_force_dense_tile(int tile_cols);

/* The columns of the dense GEMM's pair tile (256 or 448) lynx_linear_dense picks on the current device for
 * these sizes (the forced value while lynx_debug_force_dense_tile holds one); 0 for sizes out of range. */
LYNX_API int lynx_debug_dense_tile(int64_t M, int64_t N);

/* Host logic only (no device call, no test hook applies): the pair tile and k-split count that lynx_linear
 * (sparse != 0) or lynx_linear_dense (sparse == 0) would choose for these sizes on a GPU with `sms` SMs.
 * plan[0] = tile rows, plan[1] = tile columns, plan[2] = the k-split schedule as lynx_debug_linear_ksplit reports it
 * (1 for the dense layer).  Returns LYNX_OK,
 * LYNX_ERR_NULL for a NULL plan, LYNX_ERR_SHAPE for sizes out of range or sms < 2. */
LYNX_API int lynx_debug_auto_plan(int sparse, int64_t M, int64_t N, int64_t K, int sms, int32_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* LYNX_H_ */
