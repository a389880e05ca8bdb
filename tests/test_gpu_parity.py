"""Parity of the CUDA path (through the C-ABI) with the CPU oracle, element by
element, on sizes that span several tiles and a ragged tail, plus the edge and
degenerate cases of the method."""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import REL_FRO, S_RTOL, assert_y_close, pack_meta_reference, to_bits, to_dev, widen

pytestmark = pytest.mark.gpu


def _x(kind, M, K, seed=1):
    if kind == "act":
        return synth.act_bf16((M, K, seed), M, K, 0.05, 8.0)
    if kind == "gelu":  # GELU of the up projection's Gaussian pre-activations (variance 3.97)
        return synth.gelu_bf16((M, K, seed), M, K, 3.97, 0.0, 1.0)
    return synth.structured_x(kind, M, K, seed)


SPARSIFY_CASES = [
    (256, 512, "act"), (1, 16, "act"), (3, 48, "act"), (129, 528, "act"), (300, 3072, "act"),
    (77, 1040, "mixed"), (64, 256, "equal"), (64, 256, "two4"), (40, 128, "zero"), (64, 256, "ties"),
    (130, 12288, "gelu"),
]


@pytest.mark.parametrize("M,K,kind", SPARSIFY_CASES)
def test_sparsify_bit_exact(lynx, M, K, kind):
    import torch
    X = _x(kind, M, K)
    vals, meta, s = lynx.lynx_sparsify(to_dev(X))
    assert lynx.lynx_sync_status() == 0
    ref = O.sparsify(X)
    assert np.array_equal(to_bits(vals), ref["vals"])
    meta_h = meta.cpu().numpy()
    assert np.array_equal(lynx.lynx_meta_to_canonical(meta_h, M, K), ref["meta"])
    assert np.array_equal(meta_h, pack_meta_reference(ref["meta"], M, K))  # every byte, padding included
    np.testing.assert_allclose(s.cpu().numpy(), ref["s"], rtol=S_RTOL, atol=0)
    torch.cuda.synchronize()


def test_sparsify_exhaustive_tuples(lynx):
    """Every 4-tuple over {-2,-1,-0,+0,1,2,3} (ties and signed zeros everywhere), bit-exact."""
    import itertools
    tuples = np.array(list(itertools.product([-2.0, -1.0, -0.0, 0.0, 1.0, 2.0, 3.0], repeat=4)), dtype=np.float32)
    G = 16  # groups per row (K = 64)
    rows = -(-len(tuples) // G)
    pad = np.zeros((rows * G - len(tuples), 4), dtype=np.float32)
    X = synth.bf16_bits(np.concatenate([tuples, pad]).reshape(rows, 4 * G))
    vals, meta, s = lynx.lynx_sparsify(to_dev(X))
    assert lynx.lynx_sync_status() == 0
    ref = O.sparsify(X)
    assert np.array_equal(to_bits(vals), ref["vals"])
    assert np.array_equal(lynx.lynx_meta_to_canonical(meta.cpu().numpy(), rows, 4 * G), ref["meta"])
    np.testing.assert_allclose(s.cpu().numpy(), ref["s"], rtol=S_RTOL, atol=0)


def test_sparsify_special_values(lynx):
    s = lynx.lynx_sparsify(to_dev(_x("equal", 32, 256)))[2].cpu().numpy()
    np.testing.assert_allclose(s, np.sqrt(2.0), rtol=1e-6)
    s = lynx.lynx_sparsify(to_dev(_x("two4", 32, 256)))[2].cpu().numpy()
    assert np.all(s == 1.0)
    s = lynx.lynx_sparsify(to_dev(_x("zero", 32, 256)))[2].cpu().numpy()
    assert np.all(s == 1.0)


# the fused pass over X (lynx_sparsify_lora), as lynx_linear runs it: the sparsify outputs bit-exact, T' against
# the oracle; (10000, 256) makes each CTA own whole rows (no split), the others split a row's channels
FUSED_CASES = SPARSIFY_CASES + [(10000, 256, "act"), (4608, 3072, "act")]


@pytest.mark.parametrize("M,K,kind", FUSED_CASES)
@pytest.mark.parametrize("with_lb", [True, False])
def test_sparsify_lora_fused(lynx, M, K, kind, with_lb):
    X = _x(kind, M, K)
    LB = synth.gaussian_bf16((M, K, 5), (64, K), 0.02) if with_lb else None
    vals, meta, s, T = lynx.lynx_sparsify_lora(to_dev(X), to_dev(LB) if with_lb else None)
    assert lynx.lynx_sync_status() == 0
    ref = O.sparsify(X)
    assert np.array_equal(to_bits(vals), ref["vals"])
    meta_h = meta.cpu().numpy()
    assert np.array_equal(meta_h, pack_meta_reference(ref["meta"], M, K))  # every byte, padding included
    np.testing.assert_allclose(s.cpu().numpy(), ref["s"], rtol=S_RTOL, atol=0)
    if with_lb:
        assert_y_close(to_bits(T), O.lora_down(X, LB, ref["s"]), "T")
    else:
        assert T is None


@pytest.mark.parametrize("M,K,scaled", [(256, 512, True), (300, 528, True), (5, 3072, False), (129, 12288, True)])
def test_lora_down(lynx, M, K, scaled):
    X = _x("act", M, K, 3)
    LB = synth.gaussian_bf16((M, K, 4), (64, K), 0.02)
    s = O.sparsify(X)["s"] if scaled else None
    import torch
    s_dev = torch.from_numpy(s.astype(np.float32)).cuda() if scaled else None
    T = lynx.lynx_lora_down(to_dev(X), to_dev(LB), s_dev)
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(T), O.lora_down(X, LB, s), "T")


# N % 8 != 0 (1003, 130) takes the per-lane store epilogue; the others the TMA-store epilogue
LINEAR_CASES = [(256, 512, 512), (300, 520, 528), (1, 8, 16), (129, 136, 144), (200, 1000, 1024),
                (128, 256, 64), (384, 768, 3072), (200, 1003, 256), (600, 1160, 384)]


def _layer(M, N, K, seed=7, xkind="act"):
    X = _x(xkind, M, K, seed)
    W = synth.gaussian_bf16((seed, 1), (N, K), 1.0 / np.sqrt(K))
    LA = synth.gaussian_bf16((seed, 2), (N, 64), 0.02)
    LB = synth.gaussian_bf16((seed, 3), (64, K), 0.02)
    return X, W, LA, LB


@pytest.mark.parametrize("tile", [(512, 224), (512, 192), (256, 256), (256, 192)])  # sparse pair tile shapes
@pytest.mark.parametrize("M,N,K", LINEAR_CASES)
def test_linear_full_comparison(lynx, M, N, K, tile):
    X, W, LA, LB = _layer(M, N, K)
    lynx.lynx_debug_force_tile(*tile)
    try:
        Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_tile(0, 0)
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


@pytest.mark.parametrize("split", [1, 2, 3, 5, 7, 12])
def test_sparsify_lora_any_cluster_size(lynx, split):
    """The pre-pass gives the same bits for vals and metadata, and s and T' within tolerance, whatever number
    of CTAs (cluster size, not only powers of two) shares a row block's channels; Y follows."""
    M, N, K = 300, 520, 3072
    X, W, LA, LB = _layer(M, N, K, seed=5)
    lynx.lynx_debug_force_split(split)
    try:
        vals, meta, s, T = lynx.lynx_sparsify_lora(to_dev(X), to_dev(LB))
        Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_split(0)
    ref = O.sparsify(X)
    assert np.array_equal(to_bits(vals), ref["vals"])
    assert np.array_equal(meta.cpu().numpy(), pack_meta_reference(ref["meta"], M, K))  # every byte
    np.testing.assert_allclose(s.cpu().numpy(), ref["s"], rtol=S_RTOL, atol=0)
    assert_y_close(to_bits(T), O.lora_down(X, LB, ref["s"]), "T")
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


def test_prologue_split_choice(lynx):
    """The automatic cluster size never exceeds the channel blocks or the SM budget and is 1 for large M."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, K in [(1024, 3072), (1024, 12288), (4608, 3072), (9216, 3072), (16384, 3072), (100, 256)]:
        sp = lynx.lynx_debug_prologue_split(M, K)
        rb = -(-M // 256) * 2
        assert 1 <= sp <= min(16, -(-K // 128)), (M, K, sp)
        assert sp == 1 or rb * sp <= sms, (M, K, sp)
    assert lynx.lynx_debug_prologue_split(16384, 3072) == 1


@pytest.mark.parametrize("kind", ["mixed", "equal", "two4", "ties", "gelu"])
def test_linear_structured_inputs(lynx, kind):
    X, W, LA, LB = _layer(160, 384, 256, 11, kind)
    Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


def test_linear_zero_rows_give_lora_only(lynx):
    X, W, LA, LB = _layer(64, 256, 128, 12)
    X[5] = 0
    X[17] = 0
    Y = to_bits(lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB)))
    assert np.all(Y[5] == 0) and np.all(Y[17] == 0)  # X = 0 gives Ys = 0 and Yr = 0
    assert_y_close(Y, O.linear(X, W, LA, LB))


def test_linear_zero_lora_and_24_input_is_cublas_gemm(lynx):
    """Already-2:4 X with LA = 0 reduces to Y = X W^T: compare with cuBLAS and the oracle."""
    import torch
    M, N, K = 256, 512, 768
    X = _x("two4", M, K, 13)
    W = synth.gaussian_bf16((13, 1), (N, K), 1.0 / np.sqrt(K))
    LA = np.zeros((N, 64), dtype=np.uint16)
    LB = synth.gaussian_bf16((13, 3), (64, K), 0.02)
    Xd, Wd = to_dev(X), to_dev(W)
    Y = lynx.lynx_linear(Xd, Wd, to_dev(LA), to_dev(LB))
    assert lynx.lynx_sync_status() == 0
    ref = O.linear_dense(X, W)
    assert_y_close(to_bits(Y), ref)
    cub = to_bits(torch.matmul(Xd, Wd.t()))
    assert_y_close(cub, ref, "cuBLAS")
    # both are bf16 roundings of nearly the same fp32 sum
    assert np.mean(to_bits(Y) == cub) > 0.9


@pytest.mark.parametrize("tile", [256, 448])
@pytest.mark.parametrize("M,N,K,lora", [(256, 512, 512, False), (300, 520, 528, True), (129, 136, 144, False),
                                        (384, 768, 3072, True), (129, 130, 144, True), (520, 1000, 1040, True)])
def test_linear_dense(lynx, M, N, K, lora, tile):
    X, W, LA, LB = _layer(M, N, K, 17)
    lynx.lynx_debug_force_dense_tile(tile)
    try:
        if lora:
            Y = lynx.lynx_linear_dense(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
            ref = O.linear_dense(X, W, LA, LB)
        else:
            Y = lynx.lynx_linear_dense(to_dev(X), to_dev(W))
            ref = O.linear_dense(X, W)
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_dense_tile(0)
    assert_y_close(to_bits(Y), ref)


def test_dense_tile_choice(lynx):
    """On this GPU the dense layer takes 448-column tiles where their waves are about as full as the 256-column
    tiles' (the QKV shapes, N = 3072 at 16384 tokens) and 256-column tiles where a 448-column wave would stay
    partly idle (N = 3072 at 4608 tokens, 1024 tokens)."""
    for M, N in [(4608, 9216), (9216, 9216), (16384, 3072)]:
        assert lynx.lynx_debug_dense_tile(M, N) == 448, (M, N)
    for M, N in [(4608, 3072), (1024, 9216), (1024, 3072), (1024, 12288)]:
        assert lynx.lynx_debug_dense_tile(M, N) == 256, (M, N)
    lynx.lynx_debug_force_dense_tile(448)
    try:
        assert lynx.lynx_debug_dense_tile(1024, 3072) == 448
    finally:
        lynx.lynx_debug_force_dense_tile(0)
    assert lynx.lynx_debug_dense_tile(0, 8) == 0


@pytest.mark.parametrize("M,N,K", [(256, 896, 512), (300, 1000, 1040), (777, 448, 3072), (1, 8, 16)])
@pytest.mark.parametrize("lora", [False, True])
def test_dense_wide_tile_equals_narrow_tile(lynx, M, N, K, lora):
    """The dense 256 x 448 tile (two 224-column MMAs sharing one read of X) adds every output's products in the
    same k order as the 256 x 256 tile, LoRA stage last: the results agree bit for bit."""
    X, W, LA, LB = _layer(M, N, K, seed=23)
    args = [to_dev(a) for a in ((X, W, LA, LB) if lora else (X, W))]
    out = {}
    for tile in (448, 256):
        lynx.lynx_debug_force_dense_tile(tile)
        try:
            out[tile] = to_bits(lynx.lynx_linear_dense(*args))
            assert lynx.lynx_sync_status() == 0
        finally:
            lynx.lynx_debug_force_dense_tile(0)
    assert np.array_equal(out[448], out[256])
    assert_y_close(out[448], O.linear_dense(X, W, LA, LB) if lora else O.linear_dense(X, W))


def test_linear_is_deterministic(lynx):
    X, W, LA, LB = _layer(256, 512, 1024, 21)
    args = [to_dev(a) for a in (X, W, LA, LB)]
    y1 = to_bits(lynx.lynx_linear(*args))
    y2 = to_bits(lynx.lynx_linear(*args))
    assert np.array_equal(y1, y2)


def test_output_guard_band_untouched(lynx):
    """Y inside a larger buffer: the kernels write exactly M x N elements."""
    import torch
    M, N, K = 130, 264, 256
    X, W, LA, LB = _layer(M, N, K, 23)
    buf = torch.full((M * N + 4096,), -7.0, dtype=torch.bfloat16, device="cuda")
    Y = buf[2048:2048 + M * N].view(M, N)
    lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB), Y=Y)
    assert lynx.lynx_sync_status() == 0
    b = buf.float().cpu().numpy()
    assert np.all(b[:2048] == -7.0) and np.all(b[2048 + M * N:] == -7.0)
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


def test_mma_rate_microbenchmark_runs(lynx):
    for mode in (0, 1, 2):
        tf, mpc = lynx.lynx_mma_rate(mode, 2000)
        assert tf > 100 and mpc > 0


# ------------------------------------------------------------------ the weight-2:4 comparator
WSPARSE_CASES = [(256, 512, 512), (300, 520, 528), (1, 8, 16), (200, 1003, 256), (600, 1160, 384), (129, 136, 3072)]


@pytest.mark.parametrize("tile", [(512, 224), (512, 192), (256, 256), (256, 192)])
@pytest.mark.parametrize("M,N,K", WSPARSE_CASES)
def test_weight_sparse_linear(lynx, M, N, K, tile):
    """Y = X W~^T + X (LA LB)^T with W pruned and compressed by the sparsify pass: the GEMM runs W~ as the
    sparse operand and writes its transposed tile (N % 8 != 0 takes the per-lane stores)."""
    X, W, LA, LB = _layer(M, N, K, seed=9)
    Wv, Wm = lynx.lynx_prune_weight(to_dev(W))
    lynx.lynx_debug_force_tile(*tile)
    try:
        Y = lynx.lynx_linear_wsparse(to_dev(X), Wv, Wm, to_dev(LA), to_dev(LB))
        Y0 = lynx.lynx_linear_wsparse(to_dev(X), Wv, Wm)
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_tile(0, 0)
    assert_y_close(to_bits(Y), O.linear_wsparse(X, W, LA, LB))
    assert_y_close(to_bits(Y0), O.linear_wsparse(X, W), "Y without LoRA")


def test_weight_sparse_on_24_weights_matches_dense_layer(lynx):
    """Weights that are already 2:4 lose nothing: the result equals the dense layer's."""
    import torch
    M, N, K = 300, 264, 512
    X = _x("act", M, K, 4)
    W = synth.structured_x("two4", N, K, seed=4)
    Wv, Wm = lynx.lynx_prune_weight(to_dev(W))
    Y = lynx.lynx_linear_wsparse(to_dev(X), Wv, Wm)
    Yd = lynx.lynx_linear_dense(to_dev(X), to_dev(W))
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y), O.linear_dense(X, W))
    assert float((Y.float() - Yd.float()).abs().max()) <= float(Yd.float().abs().max()) * 2 ** -7
    torch.cuda.synchronize()


# ------------------------------------------------------------------ split K (few output tiles)
@pytest.mark.parametrize("tile", [(256, 256), (256, 192)])
@pytest.mark.parametrize("splits", [2, 3])
@pytest.mark.parametrize("M,N,K", LINEAR_CASES)
def test_linear_split_k(lynx, M, N, K, splits, tile):
    """The one-row-block sparse tiles with each tile's k-steps split over work units: every unit writes an fp32
    partial, the last one to finish adds them in split order; the LoRA stage runs in the last split."""
    X, W, LA, LB = _layer(M, N, K, seed=27)
    lynx.lynx_debug_force_tile(*tile)
    lynx.lynx_debug_force_ksplit(splits)
    try:
        Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_ksplit(0)
        lynx.lynx_debug_force_tile(0, 0)
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


def test_split_k_is_deterministic_and_reuses_its_workspace(lynx):
    """Arrival order varies between runs, the split order of the sum does not: repeated calls on one workspace
    (whose counters the pre-pass zeroes every call) give the same bits."""
    import torch
    M, N, K = 1024, 768, 3072
    X, W, LA, LB = (to_dev(a) for a in _layer(M, N, K, seed=29))
    lynx.lynx_debug_force_tile(256, 256)
    lynx.lynx_debug_force_ksplit(3)
    try:
        assert lynx.lynx_debug_linear_ksplit(M, N, K) == 3
        ws = torch.empty(lynx.lynx_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        outs = [to_bits(lynx.lynx_linear(X, W, LA, LB, workspace=ws)) for _ in range(3)]
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_ksplit(0)
        lynx.lynx_debug_force_tile(0, 0)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert_y_close(outs[0], O.linear(to_bits(X), to_bits(W), to_bits(LA), to_bits(LB)))


# ------------------------------------------------------------------ stream-K
@pytest.mark.parametrize("tile", [(256, 256), (256, 192)])
@pytest.mark.parametrize("M,N,K", [(1100, 2000, 1104), (520, 4000, 2048)])
def test_linear_stream_k(lynx, M, N, K, tile):
    """Stream-K: each CTA pair takes a contiguous share of all tiles' k-steps, so tiles are cut at arbitrary steps
    (ragged M, N and K included); the pairs that share a tile leave fp32 partials, the last to finish adds them in
    k order and the LoRA stage runs in the part holding the tile's last k-step; a tile one pair covers whole is
    written directly."""
    X, W, LA, LB = _layer(M, N, K, seed=33)
    lynx.lynx_debug_force_tile(*tile)
    lynx.lynx_debug_force_ksplit(lynx.LYNX_KSPLIT_STREAM)
    try:
        assert lynx.lynx_debug_linear_ksplit(M, N, K) == lynx.LYNX_KSPLIT_STREAM
        Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_ksplit(0)
        lynx.lynx_debug_force_tile(0, 0)
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


def test_stream_k_is_deterministic_and_falls_back(lynx):
    """Repeated stream-K calls on one workspace give the same bits (the parts of a tile are added in k order
    whichever pair finishes last); where stream-K cannot cut the tiles into at most four parts (fewer tiles than
    half the CTA pairs) the forced setting runs the unsplit schedule."""
    import torch
    M, N, K = 1024, 3072, 2048
    X, W, LA, LB = (to_dev(a) for a in _layer(M, N, K, seed=35))
    lynx.lynx_debug_force_tile(256, 192)
    lynx.lynx_debug_force_ksplit(lynx.LYNX_KSPLIT_STREAM)
    try:
        assert lynx.lynx_debug_linear_ksplit(M, N, K) == lynx.LYNX_KSPLIT_STREAM
        assert lynx.lynx_debug_linear_ksplit(256, 1536, 2048) == 1  # 8 tiles
        ws = torch.empty(lynx.lynx_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        outs = [to_bits(lynx.lynx_linear(X, W, LA, LB, workspace=ws)) for _ in range(3)]
        assert lynx.lynx_sync_status() == 0
    finally:
        lynx.lynx_debug_force_ksplit(0)
        lynx.lynx_debug_force_tile(0, 0)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    rows = np.arange(0, M, 37)
    Xh, Wh, LAh, LBh = (to_bits(a) for a in (X, W, LA, LB))
    assert_y_close(outs[0][rows], O.linear(Xh[rows], Wh, LAh, LBh))


def test_split_k_choice_and_workspace_fallback(lynx):
    """On this GPU a short, wide-K problem (256 tokens through the MLP down shape: 16 tiles of 256 x 192) splits;
    the DiT shapes do not (the MLP down shape at 1024 tokens fills one wave with 64 tiles of 256 x 192).  A
    workspace holding only the base part runs the unsplit schedule and gives the oracle's answer too."""
    import torch
    assert lynx.lynx_debug_linear_ksplit(256, 3072, 12288) > 1
    for M, N, K in [(4608, 9216, 3072), (4608, 3072, 12288), (16384, 9216, 3072), (1024, 9216, 3072),
                    (1024, 3072, 12288)]:
        assert lynx.lynx_debug_linear_ksplit(M, N, K) == 1, (M, N, K)
    M, N, K = 256, 1536, 3072
    X, W, LA, LB = _layer(M, N, K, seed=31)
    lynx.lynx_debug_force_ksplit(0)
    full = lynx.lynx_workspace_bytes(M, N, K)
    lynx.lynx_debug_force_ksplit(1)
    base = lynx.lynx_workspace_bytes(M, N, K)
    lynx.lynx_debug_force_ksplit(0)
    assert lynx.lynx_debug_linear_ksplit(M, N, K) > 1 and full > base
    ws = torch.empty(base, dtype=torch.uint8, device="cuda")
    Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB), workspace=ws)
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))
