"""C-ABI checks that need no GPU: the library loads, exports every symbol that
include/lynx.h declares, and rejects bad arguments on the host before it
touches the device.  The metadata layout helper is checked against the layout
the header documents, re-derived here in Python."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lynx.h")


@pytest.fixture(scope="module")
def asl():
    import activation_sparse_linear_gb300 as asl
    return asl


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"LYNX_API\s+[\w\s\*]+?\b(lynx_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("lynx_sparsify", "lynx_sparsify_lora", "lynx_linear", "lynx_linear_dense", "lynx_sync_status",
                 "lynx_meta_bytes",
                 "lynx_workspace_bytes"):
        assert name in syms


def test_library_exports_every_declared_symbol(asl):
    for name in declared_symbols():
        assert hasattr(asl.lib, name), name
        assert ctypes.cast(getattr(asl.lib, name), ctypes.c_void_p).value


def test_no_cpu_fallback_in_package():
    pkg = os.path.join(ROOT, "activation_sparse_linear_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("the oracle", ""), f


def test_sizes(asl):
    # one 2 KiB chunk per (128-row block, 128-channel block); rows padded to 256, channels to 128
    assert asl.lynx_meta_bytes(4608, 3072) == 36 * 24 * 2048
    assert asl.lynx_meta_bytes(1, 16) == 2 * 1 * 2048
    assert asl.lynx_meta_bytes(129, 130) == 2 * 2 * 2048
    assert asl.lynx_meta_bytes(257, 3072) == 4 * 24 * 2048
    ws = asl.lynx_workspace_bytes(4608, 9216, 3072, 64)
    assert ws >= 4608 * 3072 + 36 * 24 * 2048 + 4608 * 4 + 4608 * 64 * 2
    assert asl.lynx_dense_workspace_bytes(100, 64) >= 100 * 64 * 2


A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced by the host checks below


@pytest.mark.parametrize("args,status", [
    ((0, A, A, A, A, 16, 16, 16, 64, A, 1 << 30), -1),            # null X
    ((A, A, A, A, A, 16, 16, 24, 64, A, 1 << 30), -2),            # K % 16
    ((A, A, A, A, A, 0, 16, 16, 64, A, 1 << 30), -2),             # M = 0
    ((A, A, A, A, A, 16, 0, 16, 64, A, 1 << 30), -2),             # N = 0
    ((A, A, A, A, A, 16, (1 << 24) + 1, 16, 64, A, 1 << 62), -2), # N above 2^24
    ((A, A, A, A, A, 65535 * 128 + 1, 16, 16, 64, A, 1 << 62), -2),  # M above 65535 * 128
    ((A, A, A, A, A, 16, 16, (1 << 20) + 16, 64, A, 1 << 62), -2),   # K above 2^20
    ((A, A, A, A, A, 65535 * 128, 1 << 24, 16, 64, A, 1 << 62), -2),  # M N above 2^40
    ((A, A, A, A, A, 16, 16, 16, 32, A, 1 << 30), -7),            # R != 64
    ((A + 8, A, A, A, A, 16, 16, 16, 64, A, 1 << 30), -3),        # misaligned X
    ((A, A, A, A, A + 2, 16, 16, 16, 64, A, 1 << 30), -3),        # misaligned Y
    ((A, A, A, A, A, 16, 16, 16, 64, A, 100), -4),                # workspace too small
])
def test_linear_rejects_bad_arguments_on_host(asl, args, status):
    X, W, LA, LB, Y, M, N, K, R, ws, wsb = args
    assert asl.lib.lynx_linear(X or None, W, LA, LB, Y, M, N, K, R, ws, wsb, None) == status


def test_other_entry_points_reject_bad_arguments(asl):
    L = asl.lib
    assert L.lynx_sparsify(None, 4, 16, A, A, A, None) == -1
    assert L.lynx_sparsify(A, 4, 20, A, A, A, None) == -2
    assert L.lynx_sparsify(A, 4, 16, A + 4, A, A, None) == -3
    assert L.lynx_sparsify_lora(A, None, 4, 16, 64, A, A, A, A, None) == -1      # T without LB
    assert L.lynx_sparsify_lora(A, A, 4, 16, 64, A, A, A, None, None) == -1      # LB without T
    assert L.lynx_sparsify_lora(A, A, 4, 16, 32, A, A, A, A, None) == -7         # rank other than 64
    assert L.lynx_sparsify_lora(A, A, 4, 16, 64, A, A, A, A + 8, None) == -3     # misaligned T
    assert L.lynx_sparsify_lora(A, A, 0, 16, 64, A, A, A, A, None) == -2         # M = 0
    assert L.lynx_lora_down(A, A, None, A, 4, 16, 16, None) == -7
    assert L.lynx_linear_dense(A, A, A, None, A, 4, 16, 16, 64, A, 1 << 20, None) == -1   # one LoRA factor
    assert L.lynx_linear_dense(A, A, A, A, A, 4, 16, 16, 64, A, 10, None) == -4
    assert L.lynx_linear_dense(A, A, None, None, A, 4, 16, 17, 64, None, 0, None) == -2
    assert L.lynx_linear_dense(A, A, None, None, A, 1 << 22, 1 << 19, 16, 64, None, 0, None) == -2   # M N > 2^40
    assert L.lynx_linear_wsparse(A, None, A, None, None, A, 4, 16, 16, 64, None, 0, None) == -1       # no W values
    assert L.lynx_linear_wsparse(A, A, A, A, None, A, 4, 16, 16, 64, A, 1 << 20, None) == -1          # one LoRA factor
    assert L.lynx_linear_wsparse(A, A, A, None, None, A, 4, 16, 24, 64, None, 0, None) == -2          # K % 16
    assert L.lynx_linear_wsparse(A, A + 8, A, None, None, A, 4, 16, 16, 64, None, 0, None) == -3      # misaligned
    assert L.lynx_linear_wsparse(A, A, A, A, A, A, 4, 16, 16, 64, A, 10, None) == -4                  # workspace
    assert L.lynx_linear_wsparse(A, A, A, A, A, A, 4, 16, 16, 32, A, 1 << 20, None) == -7             # rank
    for code in range(-7, 1):
        assert L.lynx_status_string(code)


def test_noalloc_checks_arguments_before_the_scratch_size(asl):
    """Bad pointers, ranks and shapes report their own status, not LYNX_ERR_TOO_LARGE (host checks only)."""
    fn = asl.lib.lynx_linear_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 4 + [ctypes.c_void_p]
    assert fn(None, A, A, A, A, 16, 16, 16, 64, None) == -1                  # NULL X
    assert fn(A, A, A, A, A, 16, 16, 16, 4096, None) == -7                   # rank other than 64
    assert fn(A, A, A, A, A, 4608, 9216, 3072, 4096, None) == -7             # ... even when its bytes are large
    assert fn(A, A, A, A, A, 16, 16, 24, 64, None) == -2                     # K % 16
    assert fn(A + 8, A, A, A, A, 16, 16, 16, 64, None) == -3                 # misaligned X
    assert fn(A, A, A, A, A, 16384, 3072, 12288, 64, None) == -8             # valid, beyond the scratch


def test_force_split_range(asl):
    L = asl.lib
    try:
        for bad in (-1, 17, 100):
            assert L.lynx_debug_force_split(bad) == -7
        for ok in (1, 2, 3, 12, 16):
            assert L.lynx_debug_force_split(ok) == 0
    finally:
        assert L.lynx_debug_force_split(0) == 0
    assert L.lynx_debug_prologue_split(0, 3072) == 0 and L.lynx_debug_prologue_split(64, 24) == 0  # host checks


def test_force_ksplit_range(asl):
    L = asl.lib
    try:
        for bad in (-1, 5, 7, 9, 64):
            assert L.lynx_debug_force_ksplit(bad) == -7
        for ok in (1, 2, 3, 4, asl.LYNX_KSPLIT_STREAM):
            assert L.lynx_debug_force_ksplit(ok) == 0
    finally:
        assert L.lynx_debug_force_ksplit(0) == 0
    assert L.lynx_debug_linear_ksplit(0, 16, 16) == 0 and L.lynx_debug_linear_ksplit(16, 16, 24) == 0
    # the binding's schedule code is the header's
    assert re.search(r"#define LYNX_KSPLIT_STREAM (\d+)", open(HEADER).read()).group(1) == str(asl.LYNX_KSPLIT_STREAM)


def test_force_tile_accepts_only_built_shapes(asl):
    L = asl.lib
    try:
        for rows, cols in [(512, 256), (256, 224), (384, 224), (1, 1), (0, 224)]:
            assert L.lynx_debug_force_tile(rows, cols) == -7
        for rows, cols in [(512, 224), (512, 192), (256, 256), (256, 192)]:
            assert L.lynx_debug_force_tile(rows, cols) == 0
    finally:
        assert L.lynx_debug_force_tile(0, 0) == 0


def test_force_dense_tile_accepts_only_built_shapes(asl):
    L = asl.lib
    try:
        for cols in [224, 192, 512, -1, 1]:
            assert L.lynx_debug_force_dense_tile(cols) == -7
        for cols in [256, 448]:
            assert L.lynx_debug_force_dense_tile(cols) == 0
    finally:
        assert L.lynx_debug_force_dense_tile(0) == 0


def test_auto_plan_on_152_sms(asl):
    """The tile and split choice for the DiT shapes on a 152-SM GPU (76 CTA pairs), host logic only.  Waves =
    ceil(tiles / 76); the cost compares waves x tile work x shared-memory bytes per MAC."""
    plan = asl.lynx_debug_auto_plan
    # sparse: QKV 9 x 42 = 378 tiles of 512 x 224 = 4.97 waves (432 tiles of 512 x 192 would take 6)
    assert plan(True, 4608, 9216, 3072, 152) == (512, 224, 1)
    assert plan(True, 4608, 12288, 3072, 152) == (512, 224, 1)
    assert plan(True, 16384, 9216, 3072, 152) == (512, 224, 1)
    # N = 3072: 224-wide columns (14 x 9 = 126 tiles) and 192-wide (16 x 9 = 144) both take 2 waves; 192 is cheaper
    assert plan(True, 4608, 3072, 12288, 152) == (512, 192, 1)
    # few row tiles: 4 x 36 = 144 tiles of 256 x 256 fill 2 waves; 4 x 16 = 64 of 256 x 192 fit in one (stream-K,
    # measured slower there, is never chosen)
    assert plan(True, 1024, 9216, 3072, 152) == (256, 256, 1)
    assert plan(True, 1024, 3072, 12288, 152) == (256, 192, 1)
    assert plan(True, 1024, 3072, 3072, 152) == (256, 192, 1)
    # 16 tiles leave 60 pairs idle: split K four ways (64 units, one wave)
    assert plan(True, 256, 3072, 12288, 152) == (256, 192, 4)
    # dense: 378 tiles of 256 x 448 (4.97 waves) beat 648 of 256 x 256 (8.53); N = 3072 at 4608 keeps 256
    assert plan(False, 4608, 9216, 3072, 152) == (256, 448, 1)
    assert plan(False, 4608, 12288, 3072, 152) == (256, 448, 1)
    assert plan(False, 16384, 3072, 3072, 152) == (256, 448, 1)
    assert plan(False, 4608, 3072, 3072, 152) == (256, 256, 1)
    assert plan(False, 1024, 3072, 3072, 152) == (256, 256, 1)
    # a GPU with 8 SMs (4 pairs) never splits (too few pairs to gain) and keeps the big sparse tile
    assert plan(True, 256, 3072, 12288, 8)[2] == 1
    import ctypes
    p = (ctypes.c_int32 * 3)()
    assert asl.lib.lynx_debug_auto_plan(1, 0, 8, 16, 152, p) == -2
    assert asl.lib.lynx_debug_auto_plan(1, 8, 8, 16, 1, p) == -2
    assert asl.lib.lynx_debug_auto_plan(1, 8, 8, 16, 152, None) == -1


@pytest.mark.parametrize("M,K", [(1, 16), (5, 136), (130, 256), (17, 96), (300, 512)])
def test_meta_to_canonical_matches_documented_layout(asl, M, K):
    from helpers import pack_meta_reference
    rng = np.random.default_rng(M * 1000 + K)
    nibs = np.array([0x4, 0x8, 0xC, 0x9, 0xD, 0xE], dtype=np.uint8)
    g = nibs[rng.integers(0, 6, size=(M, K // 4))]
    canon = (g[:, 0::2] | (g[:, 1::2] << 4)).astype(np.uint8)
    packed = pack_meta_reference(canon, M, K)
    assert packed.size == asl.lynx_meta_bytes(M, K)
    assert np.array_equal(asl.lynx_meta_to_canonical(packed, M, K), canon)


def test_meta_layout_pairs_rows_r_and_r_plus_8():
    """Spot check of the documented 16-bit pairing on two hand-made rows (0 and 8 of a block)."""
    from helpers import pack_meta_reference
    M, K = 16, 128
    canon = np.full((M, K // 8), 0x44, dtype=np.uint8)
    canon[0, :4] = [0x98, 0xDC, 0x49, 0xEC]   # row 0, channels 0..31
    canon[8, 4:8] = [0x8E, 0x9D, 0xC4, 0x48]  # row 8, channels 32..63
    words = pack_meta_reference(canon, M, K).view(np.uint32).reshape(2, 1, 128, 4)[0, 0]
    row0 = 0x98 | 0xDC << 8 | 0x49 << 16 | 0xEC << 24
    row8 = 0x8E | 0x9D << 8 | 0xC4 << 16 | 0x48 << 24
    assert words[0, 0] == (row0 & 0xFFFF) | (0x4444 << 16)          # lane 0, chunk 0: low halves of rows 0, 8
    assert words[8, 0] == (row0 >> 16) | (0x4444 << 16)             # lane 8, chunk 0: high halves
    assert words[0, 1] == 0x4444 | ((row8 & 0xFFFF) << 16)          # lane 0, chunk 1
    assert words[8, 1] == 0x4444 | ((row8 >> 16) << 16)             # lane 8, chunk 1
    assert words[1, 0] == 0x44444444 and words[9, 3] == 0x44444444


def _layers(asl, specs):
    arr = (asl.LynxLayer * len(specs))()
    for i, sp in enumerate(specs):
        arr[i] = asl.LynxLayer(*sp)
    return arr


def test_layer_sequences_check_every_layer_before_launching(asl):
    import ctypes
    L = asl.lib
    sparse = (1, A, A, A, A, A, 300, 384, 512, 64)
    dense = (0, A, A, None, None, A, 300, 256, 384, 64)
    dense_lora = (0, A, A, A, A, A, 300, 528, 256, 64)
    ok = _layers(asl, [sparse, dense, dense_lora])
    need = max(asl.lynx_workspace_bytes(300, 384, 512, 64), asl.lynx_dense_workspace_bytes(300, 64))
    assert L.lynx_layers_workspace_bytes(ok, 3) == need
    assert L.lynx_layers_workspace_bytes(ok, 0) == 0
    failed = ctypes.c_int32(7)
    # a bad layer anywhere: its status and index, nothing launched (no GPU here)
    for bad, status in [((0, A, A, None, None, A, 300, 256, 250, 64), -2),   # K % 16
                        ((1, A, A, None, A, A, 300, 256, 512, 64), -1),      # sparse without LA
                        ((0, A, A, A, None, A, 300, 256, 512, 64), -1),      # one LoRA factor
                        ((1, A, A, A, A, A + 8, 300, 256, 512, 64), -3),     # misaligned Y
                        ((1, A, A, A, A, A, 300, 256, 512, 32), -7)]:        # rank other than 64
        seq = _layers(asl, [sparse, dense, bad])
        assert L.lynx_run_layers(seq, 3, A, need, None, ctypes.byref(failed)) == status
        assert failed.value == 2
    assert L.lynx_run_layers(ok, 3, A, 100, None, ctypes.byref(failed)) == -4     # workspace too small
    assert failed.value == 0
    assert L.lynx_run_layers(ok, 0, None, 0, None, ctypes.byref(failed)) == 0     # nothing to do
    assert failed.value == -1
    assert L.lynx_run_layers(None, 2, A, need, None, None) == -1
    handle = ctypes.c_void_p(123)
    bad = _layers(asl, [sparse, (0, A, A, None, None, A, 0, 256, 384, 64)])  # M = 0
    assert L.lynx_graph_create(bad, 2, A, need, ctypes.byref(handle), ctypes.byref(failed)) == -2
    assert failed.value == 1 and not handle.value
    assert L.lynx_graph_create(ok, 0, A, need, ctypes.byref(handle), None) == -2
    assert L.lynx_graph_create(ok, 3, A, need, None, None) == -1
    assert L.lynx_graph_launch(None, None) == -1
    assert L.lynx_graph_destroy(None) == 0
