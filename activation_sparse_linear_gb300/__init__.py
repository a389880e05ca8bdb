"""Python binding of liblynx.so, the RT-Lynx 2:4 activation-sparse linear layer.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
CPU path; importing this package on a machine where the library cannot be
loaded raises.

Names and arguments follow ``include/lynx.h``.  Tensors are bf16 CUDA tensors
(``torch.bfloat16``) laid out row-major; ``s`` is float32.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB, build, up_to_date

__all__ = [
    "LynxError", "lib", "LYNX_OK", "LYNX_ERR_TIMEOUT",
    "lynx_meta_bytes", "lynx_workspace_bytes", "lynx_dense_workspace_bytes",
    "lynx_sparsify", "lynx_sparsify_lora", "lynx_lora_down", "lynx_linear",
    "lynx_linear_dense", "lynx_linear_fused", "lynx_prune_weight", "lynx_linear_wsparse",
    "lynx_sync_status", "lynx_status_string", "lynx_meta_to_canonical", "lynx_debug_set_fault",
    "lynx_debug_force_tile", "lynx_debug_force_split", "lynx_debug_prologue_split",
    "lynx_debug_force_ksplit", "lynx_debug_linear_ksplit", "lynx_debug_force_dense_tile",
    "lynx_debug_dense_tile", "lynx_debug_auto_plan",
    "lynx_profile_next", "lynx_linear_kernel_count", "lynx_mma_rate",
    "LynxLayer", "lynx_layer", "lynx_layers_workspace_bytes", "lynx_run_layers", "LynxGraph",
    "LYNX_LAYER_SPARSE", "LYNX_LAYER_GELU", "LYNX_LAYER_FUSE_SPARSIFY", "lynx_debug_pair_offsets",
]

LYNX_OK = 0
LYNX_ERR_TIMEOUT = -6
LYNX_LAYER_SPARSE = 1
LYNX_LAYER_GELU = 2
LYNX_LAYER_FUSE_SPARSIFY = 4
LYNX_KSPLIT_STREAM = 8  # lynx_debug_force_ksplit / lynx_debug_linear_ksplit: the stream-K schedule

_c_i64, _c_sz, _c_p = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p


class LynxLayer(ctypes.Structure):
    """``lynx_layer`` of include/lynx.h: one sparse (lynx_linear) or dense (lynx_linear_dense) layer; ``flags``
    bit 0 = sparse, bit 1 = GELU of the output."""
    _fields_ = [("flags", ctypes.c_int32), ("X", _c_p), ("W", _c_p), ("LA", _c_p), ("LB", _c_p), ("Y", _c_p),
                ("M", _c_i64), ("N", _c_i64), ("K", _c_i64), ("R", _c_i64)]


_c_layers = ctypes.POINTER(LynxLayer)
_c_i32p = ctypes.POINTER(ctypes.c_int32)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB) or (os.environ.get("LYNX_AUTOBUILD", "1") == "1" and not up_to_date()):
        build()
    L = ctypes.CDLL(LIB)
    sig = {
        "lynx_meta_bytes": (_c_sz, [_c_i64, _c_i64]),
        "lynx_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i64, _c_i64]),
        "lynx_dense_workspace_bytes": (_c_sz, [_c_i64, _c_i64]),
        "lynx_sparsify": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p]),
        "lynx_lora_down": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p]),
        "lynx_sparsify_lora": (ctypes.c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p]),
        "lynx_linear": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_p, _c_sz, _c_p]),
        "lynx_linear_dense": (ctypes.c_int,
                              [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_p, _c_sz, _c_p]),
        "lynx_linear_fused": (ctypes.c_int,
                              [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_p, _c_sz, _c_p]),
        "lynx_linear_wsparse": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64,
                                                _c_p, _c_sz, _c_p]),
        "lynx_sync_status": (ctypes.c_int, [_c_p]),
        "lynx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "lynx_meta_to_canonical": (ctypes.c_int, [_c_p, _c_p, _c_i64, _c_i64]),
        "lynx_debug_set_fault": (None, [ctypes.c_int, ctypes.c_uint64]),
        "lynx_debug_force_tile": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
        "lynx_debug_force_split": (ctypes.c_int, [ctypes.c_int]),
        "lynx_debug_prologue_split": (ctypes.c_int, [_c_i64, _c_i64]),
        "lynx_debug_force_ksplit": (ctypes.c_int, [ctypes.c_int]),
        "lynx_debug_force_dense_tile": (ctypes.c_int, [ctypes.c_int]),
        "lynx_debug_dense_tile": (ctypes.c_int, [_c_i64, _c_i64]),
        "lynx_debug_auto_plan": (ctypes.c_int, [ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_int32)]),
        "lynx_debug_linear_ksplit": (ctypes.c_int, [_c_i64, _c_i64, _c_i64]),
        "lynx_profile_next": (None, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
        "lynx_linear_kernel_count": (ctypes.c_int, [_c_i64, _c_i64, _c_i64, _c_i64]),
        "lynx_mma_rate": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_double), _c_p]),
        "lynx_layers_workspace_bytes": (_c_sz, [_c_layers, ctypes.c_int32]),
        "lynx_run_layers": (ctypes.c_int, [_c_layers, ctypes.c_int32, _c_p, _c_sz, _c_p, _c_i32p]),
        "lynx_graph_create": (ctypes.c_int, [_c_layers, ctypes.c_int32, _c_p, _c_sz, ctypes.POINTER(_c_p), _c_i32p]),
        "lynx_graph_launch": (ctypes.c_int, [_c_p, _c_p]),
        "lynx_graph_destroy": (ctypes.c_int, [_c_p]),
        "lynx_debug_pair_offsets": (ctypes.c_int, [_c_layers, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.POINTER(ctypes.c_size_t)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    return L


lib = _load()


class LynxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.lynx_status_string(status).decode()} (status {status})")


def _check(status: int, where: str) -> None:
    if status != LYNX_OK:
        raise LynxError(status, where)


def _torch():
    import torch
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int | None:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t, name, dtype=None, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def lynx_meta_bytes(M: int, K: int) -> int:
    return lib.lynx_meta_bytes(M, K)


def lynx_workspace_bytes(M: int, N: int, K: int, R: int = 64) -> int:
    return lib.lynx_workspace_bytes(M, N, K, R)


def lynx_dense_workspace_bytes(M: int, R: int = 64) -> int:
    return lib.lynx_dense_workspace_bytes(M, R)


def lynx_sparsify(X, vals=None, meta=None, s=None, stream=None):
    """Compressed 2:4 values (M x K/2 bf16), metadata (uint8, lynx_meta_bytes) and s (M fp32)."""
    torch = _torch()
    _need(X, "X", torch.bfloat16)
    M, K = X.shape
    vals = torch.empty((M, K // 2), dtype=torch.bfloat16, device=X.device) if vals is None else vals
    meta = torch.empty(lynx_meta_bytes(M, K), dtype=torch.uint8, device=X.device) if meta is None else meta
    s = torch.empty(M, dtype=torch.float32, device=X.device) if s is None else s
    _check(lib.lynx_sparsify(_ptr(X), M, K, _ptr(vals), _ptr(meta), _ptr(s), _stream(stream)), "lynx_sparsify")
    return vals, meta, s


def lynx_sparsify_lora(X, LB=None, vals=None, meta=None, s=None, T=None, stream=None):
    """One pass over X: (vals, meta, s) as lynx_sparsify and, with LB, T = bf16(X LB^T / s) (else None)."""
    torch = _torch()
    _need(X, "X", torch.bfloat16)
    M, K = X.shape
    R = 64
    if LB is not None:
        _need(LB, "LB", torch.bfloat16)
        R = LB.shape[0]
        T = torch.empty((M, R), dtype=torch.bfloat16, device=X.device) if T is None else T
    vals = torch.empty((M, K // 2), dtype=torch.bfloat16, device=X.device) if vals is None else vals
    meta = torch.empty(lynx_meta_bytes(M, K), dtype=torch.uint8, device=X.device) if meta is None else meta
    s = torch.empty(M, dtype=torch.float32, device=X.device) if s is None else s
    _check(lib.lynx_sparsify_lora(_ptr(X), _ptr(LB), M, K, R, _ptr(vals), _ptr(meta), _ptr(s), _ptr(T),
                                  _stream(stream)), "lynx_sparsify_lora")
    return vals, meta, s, T


def lynx_lora_down(X, LB, s=None, T=None, stream=None):
    """T = bf16(X LB^T / s) (s=None: no division); M x R bf16."""
    torch = _torch()
    _need(X, "X", torch.bfloat16)
    _need(LB, "LB", torch.bfloat16)
    M, K = X.shape
    R = LB.shape[0]
    T = torch.empty((M, R), dtype=torch.bfloat16, device=X.device) if T is None else T
    _check(lib.lynx_lora_down(_ptr(X), _ptr(LB), _ptr(s), _ptr(T), M, K, R, _stream(stream)), "lynx_lora_down")
    return T


def lynx_linear(X, W, LA, LB, Y=None, workspace=None, stream=None):
    """Y = bf16(s * (X~ W^T) + (X LB^T) LA^T), the RT-Lynx sparse linear."""
    torch = _torch()
    for t, n in ((X, "X"), (W, "W"), (LA, "LA"), (LB, "LB")):
        _need(t, n, torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    R = LB.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    need = lynx_workspace_bytes(M, N, K, R)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    _check(lib.lynx_linear(_ptr(X), _ptr(W), _ptr(LA), _ptr(LB), _ptr(Y), M, N, K, R, _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream)), "lynx_linear")
    return Y


def lynx_linear_dense(X, W, LA=None, LB=None, Y=None, workspace=None, stream=None):
    """Y = bf16(X W^T [+ (X LB^T) LA^T]): a selectively skipped layer."""
    torch = _torch()
    _need(X, "X", torch.bfloat16)
    _need(W, "W", torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    R = 0 if LB is None else LB.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    if LA is not None and workspace is None:
        workspace = torch.empty(lynx_dense_workspace_bytes(M, R), dtype=torch.uint8, device=X.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.lynx_linear_dense(_ptr(X), _ptr(W), _ptr(LA), _ptr(LB), _ptr(Y), M, N, K, R, _ptr(workspace), wbytes,
                                 _stream(stream)), "lynx_linear_dense")
    return Y


def lynx_linear_fused(X, W, LA, LB, Y=None, workspace=None, stream=None):
    """Y = S(X) W^T + X (LA LB)^T with the 2:4 selection inside the GEMM (no sparsify pass; see include/lynx.h)."""
    torch = _torch()
    for t, n in ((X, "X"), (W, "W"), (LA, "LA"), (LB, "LB")):
        _need(t, n, torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    R = LB.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    if workspace is None:
        workspace = torch.empty(lynx_dense_workspace_bytes(M, R), dtype=torch.uint8, device=X.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check(lib.lynx_linear_fused(_ptr(X), _ptr(W), _ptr(LA), _ptr(LB), _ptr(Y), M, N, K, R, _ptr(workspace), wbytes,
                                 _stream(stream)), "lynx_linear_fused")
    return Y


def lynx_prune_weight(W, stream=None):
    """W~ of the weight-2:4 comparator, compressed: (values N x K/2 bf16, metadata) via lynx_sparsify."""
    vals, meta, _ = lynx_sparsify(W, stream=stream)
    return vals, meta


def lynx_linear_wsparse(X, Wvals, Wmeta, LA=None, LB=None, Y=None, workspace=None, stream=None):
    """Y = bf16(X W~^T [+ (X LB^T) LA^T]): the weight-2:4 comparator on pruned, compressed W (lynx_prune_weight)."""
    torch = _torch()
    _need(X, "X", torch.bfloat16)
    _need(Wvals, "Wvals", torch.bfloat16)
    M, K = X.shape
    N = Wvals.shape[0]
    R = 0 if LB is None else LB.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    if LA is not None and workspace is None:
        workspace = torch.empty(lynx_dense_workspace_bytes(M, R), dtype=torch.uint8, device=X.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.lynx_linear_wsparse(_ptr(X), _ptr(Wvals), _ptr(Wmeta), _ptr(LA), _ptr(LB), _ptr(Y), M, N, K, R,
                                   _ptr(workspace), wbytes, _stream(stream)), "lynx_linear_wsparse")
    return Y


def lynx_sync_status(stream=None) -> int:
    return lib.lynx_sync_status(_stream(stream))


def lynx_status_string(status: int) -> str:
    return lib.lynx_status_string(status).decode()


def lynx_meta_to_canonical(meta_host, M: int, K: int):
    """Host conversion of the tensor-core metadata layout to canonical M x K/8 bytes (numpy uint8)."""
    import numpy as np
    src = np.ascontiguousarray(meta_host, dtype=np.uint8)
    out = np.empty((M, K // 8), dtype=np.uint8)
    _check(lib.lynx_meta_to_canonical(src.ctypes.data, out.ctypes.data, M, K), "lynx_meta_to_canonical")
    return out


def lynx_linear_kernel_count(M: int, N: int, K: int, R: int = 64) -> int:
    return lib.lynx_linear_kernel_count(M, N, K, R)


def lynx_mma_rate(mode: int, iters: int = 20000, stream=None) -> tuple[float, float]:
    """(dense-equivalent TFLOP/s, MACs per SM clock) of back-to-back smem-resident MMAs.

    mode 0 dense, 1 2:4 sparse, 2 2:4 sparse with a metadata tcgen05.cp per MMA,
    3 sparse with a commit per two MMAs, 4 sparse with two commits per four MMAs, 5 sparse with
    64-byte-swizzled A; 6-8 on CTA pairs: 6 sparse (A 128-byte swizzle), 7 sparse (A 64-byte swizzle),
    8 dense."""
    tf, mpc = ctypes.c_double(), ctypes.c_double()
    _check(lib.lynx_mma_rate(int(mode), iters, ctypes.byref(tf), ctypes.byref(mpc), _stream(stream)), "lynx_mma_rate")
    return tf.value, mpc.value


def lynx_profile_next(events) -> None:
    """Have the next lynx_linear / lynx_linear_dense call on this thread record ``events``
    (torch.cuda.Event objects, already created) around its kernels."""
    handles = [e.cuda_event for e in events]
    if any(h == 0 for h in handles):
        raise ValueError("record each event once before passing it (torch creates events lazily)")
    arr = (ctypes.c_void_p * len(handles))(*handles)
    _profile_keepalive[:] = [arr]
    lib.lynx_profile_next(arr, len(handles))


_profile_keepalive: list = []


def lynx_debug_set_fault(inject: int, wait_ns: int = 0) -> None:
    lib.lynx_debug_set_fault(inject, wait_ns)


def lynx_debug_force_tile(tile_rows: int, tile_cols: int) -> None:
    """Test hook: forces the 512x224, 512x192, 256x256 or 256x192 sparse tile shape; (0, 0) restores the automatic
    choice."""
    _check(lib.lynx_debug_force_tile(tile_rows, tile_cols), "lynx_debug_force_tile")


def lynx_debug_force_split(split: int) -> None:
    """Test hook: the sparsify pass runs each 128-row block on a cluster of ``split`` CTAs; 0 = automatic."""
    _check(lib.lynx_debug_force_split(split), "lynx_debug_force_split")


def lynx_debug_force_dense_tile(tile_cols: int) -> None:
    """Test hook: the dense GEMM uses 256 x ``tile_cols`` pair tiles (256 or 448) for every shape; 0 = automatic."""
    _check(lib.lynx_debug_force_dense_tile(tile_cols), "lynx_debug_force_dense_tile")


def lynx_debug_auto_plan(sparse: bool, M: int, N: int, K: int, sms: int) -> tuple:
    """Host logic only: (tile rows, tile columns, k-splits) the sparse (or dense) layer would choose on a GPU
    with ``sms`` SMs."""
    plan = (ctypes.c_int32 * 3)()
    _check(lib.lynx_debug_auto_plan(1 if sparse else 0, M, N, K, sms, plan), "lynx_debug_auto_plan")
    return tuple(plan)


def lynx_debug_dense_tile(M: int, N: int) -> int:
    """The dense GEMM's tile columns (256 or 448) for these sizes on the current device; 0 out of range."""
    return lib.lynx_debug_dense_tile(M, N)


def lynx_debug_force_ksplit(splits: int) -> None:
    """Test hook: the sparse GEMM splits the k-steps of each one-row-block tile (256 x 256, 256 x 192) over
    ``splits`` units, or runs the stream-K schedule (``LYNX_KSPLIT_STREAM``) where it applies; 0 = automatic."""
    _check(lib.lynx_debug_force_ksplit(splits), "lynx_debug_force_ksplit")


def lynx_debug_linear_ksplit(M: int, N: int, K: int) -> int:
    """The k-split schedule lynx_linear picks on this device for M x K -> N (1 = none, 2-4 = equal splits,
    ``LYNX_KSPLIT_STREAM`` = stream-K)."""
    return lib.lynx_debug_linear_ksplit(M, N, K)


def lynx_debug_prologue_split(M: int, K: int) -> int:
    """Cluster size the sparsify pass picks on this device for an M x K activation."""
    return lib.lynx_debug_prologue_split(M, K)


# ------------------------------------------------------------------ layer sequences and their CUDA graphs
def lynx_layer(X, W, LA=None, LB=None, Y=None, sparse: bool = True, gelu: bool = False, fuse: bool = False) -> dict:
    """One layer of a sequence: Y = lynx_linear(X, W, LA, LB) (sparse) or lynx_linear_dense(X, W, LA, LB), passed
    through GELU when ``gelu`` (the MLP up layer).  ``fuse`` (with ``gelu``): a following sparse layer that reads
    this Y runs fused with it (include/lynx.h, LYNX_LAYER_FUSE_SPARSIFY).  Allocates Y (M x N bf16) when not given.
    The dict keeps the tensors alive."""
    torch = _torch()
    _need(X, "X", torch.bfloat16)
    _need(W, "W", torch.bfloat16)
    M, K = X.shape
    N = W.shape[0]
    R = 64 if LB is None else LB.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    return {"sparse": bool(sparse), "gelu": bool(gelu), "fuse": bool(fuse), "X": X, "W": W, "LA": LA, "LB": LB, "Y": Y,
            "M": M, "N": N, "K": K, "R": R}


def _c_layer_array(layers):
    arr = (LynxLayer * max(len(layers), 1))()
    for i, l in enumerate(layers):
        flags = ((LYNX_LAYER_SPARSE if l["sparse"] else 0) | (LYNX_LAYER_GELU if l.get("gelu") else 0) |
                 (LYNX_LAYER_FUSE_SPARSIFY if l.get("fuse") else 0))
        arr[i] = LynxLayer(flags, _ptr(l["X"]), _ptr(l["W"]), _ptr(l["LA"]), _ptr(l["LB"]), _ptr(l["Y"]),
                           l["M"], l["N"], l["K"], l["R"])
    return arr


def lynx_layers_workspace_bytes(layers) -> int:
    return lib.lynx_layers_workspace_bytes(_c_layer_array(layers), len(layers))


def _layer_error(status: int, failed: ctypes.c_int32, where: str) -> None:
    if status != LYNX_OK:
        raise LynxError(status, f"{where} (layer {failed.value})" if failed.value >= 0 else where)


def lynx_run_layers(layers, workspace=None, stream=None):
    """Runs the layers in order on one stream; returns the list of their Y tensors."""
    torch = _torch()
    if workspace is None and layers:
        workspace = torch.empty(max(lynx_layers_workspace_bytes(layers), 1), dtype=torch.uint8,
                                device=layers[0]["X"].device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    failed = ctypes.c_int32(-1)
    _layer_error(lib.lynx_run_layers(_c_layer_array(layers), len(layers), _ptr(workspace), wbytes, _stream(stream),
                                     ctypes.byref(failed)), failed, "lynx_run_layers")
    return [l["Y"] for l in layers]


def lynx_debug_pair_offsets(layers, i: int) -> dict:
    """Workspace byte offsets of the fused MLP pair (i, i + 1): the sparse layer's vals, meta, s, T' and the
    pair's total bytes."""
    out = (ctypes.c_size_t * 5)()
    _check(lib.lynx_debug_pair_offsets(_c_layer_array(layers), len(layers), i, out), "lynx_debug_pair_offsets")
    return {"vals": out[0], "meta": out[1], "s": out[2], "T": out[3], "total": out[4]}


class LynxGraph:
    """A layer sequence captured once into a CUDA graph; ``launch()`` replays all of its kernels.
    Holds references to every tensor of the layers and to the workspace, whose addresses the graph uses."""

    def __init__(self, layers, workspace=None):
        torch = _torch()
        self.layers = list(layers)
        if workspace is None:
            workspace = torch.empty(max(lynx_layers_workspace_bytes(self.layers), 1), dtype=torch.uint8,
                                    device=self.layers[0]["X"].device)
        self.workspace = workspace
        self._streams = {}  # every stream a replay was enqueued on (by handle), for __exit__
        handle, failed = _c_p(), ctypes.c_int32(-1)
        _layer_error(lib.lynx_graph_create(_c_layer_array(self.layers), len(self.layers), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), ctypes.byref(handle),
                                           ctypes.byref(failed)), failed, "lynx_graph_create")
        self._handle = handle

    def launch(self, stream=None) -> None:
        if not self._handle:
            raise LynxError(-1, "LynxGraph.launch after close")
        torch = _torch()
        s = torch.cuda.current_stream() if stream is None else stream
        self._streams[s.cuda_stream] = s
        _check(lib.lynx_graph_launch(self._handle, s.cuda_stream), "lynx_graph_launch")

    def close(self) -> None:
        """Frees the graph; call after the replays have completed."""
        if self._handle:
            _check(lib.lynx_graph_destroy(self._handle), "lynx_graph_destroy")
            self._handle = _c_p()

    def __enter__(self) -> "LynxGraph":
        return self

    def __exit__(self, exc_type, exc, tb) -> None:
        """Waits for every stream a replay was launched on, then frees the graph (always, even when a wait
        fails).  A failure here is raised only when no exception is already leaving the with-block.  The
        device error word is left for the caller's lynx_sync_status."""
        if not self._handle:
            return
        try:
            for s in self._streams.values():
                s.synchronize()
        except Exception:
            if exc_type is None:
                raise
        finally:
            self._streams.clear()
            try:
                self.close()
            except Exception:
                if exc_type is None:
                    raise
