"""The MLP pair run as one fused path: the up layer's epilogue applies GELU and writes the 2:4 sparsification of
its output for the down layer (values, metadata, row-norm partials), and the down layer's sparsify pass is
replaced by a LoRA down-projection that finishes s and T' ("RT-Lynx" page, CUDA kernel optimisation: one
execution path for the online sparsification).

The down layer's input is H = bf16(GELU(bf16(Y_up))): GELU applied to the up layer's bf16 output, as an
unfused bf16 pipeline computes it.  Where floating point decides the selection, both sides decide it on the
same bf16 values: the compressed values and the metadata are compared bit for bit with the oracle's
sparsification of the H the GPU produced.  H itself is compared with the oracle's H element by element within
the up layer's Y tolerance carried through GELU and the two bf16 roundings (see assert_h_close), and within the
Y tolerance in relative Frobenius error; the down layer's Y is held to the Y tolerance against the oracle on both
H's.
"""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import REL_FRO, S_RTOL, assert_y_close, pack_meta_reference, to_bits, to_dev, widen

pytestmark = pytest.mark.gpu


def up_reference(X, W, LA, LB, sparse, rows=None):
    """The oracle's up-layer output y (float64) and H = bf16(GELU(bf16(y))) for the given rows."""
    y = O.linear(X, W, LA, LB, rows) if sparse else O.linear_dense(X, W, LA, LB, rows)
    return y, O.gelu_bf16(O.round_bf16(y))


def assert_h_close(h_bits: np.ndarray, y_ref: np.ndarray, h_ref_bits: np.ndarray, what="H"):
    """H = bf16(GELU(bf16(y))) against the oracle's, element by element, and rel-Frobenius <= 5e-3.

    Bound per element: 1.13 (2e-2 rms(y) + ulp(y)) + ulp(h).  The up layer's y may differ from the oracle's by the
    Y tolerance (2e-2 rms(y)); its bf16 rounding adds up to one ulp of y, GELU's slope is at most 1.13 in
    magnitude, and the rounding of h to bf16 adds up to one ulp of h (half on each side)."""
    h, r = widen(h_bits), widen(h_ref_bits)

    def ulp(v):
        return np.exp2(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126))) - 7)

    rms_y = float(np.sqrt(np.mean(y_ref * y_ref)))
    bound = 1.13 * (2e-2 * rms_y + ulp(y_ref)) + ulp(r)
    err = np.abs(h - r)
    worst = float(np.max(err / bound)) if err.size else 0.0
    fro = float(np.linalg.norm(h - r) / max(np.linalg.norm(r), 1e-300))
    assert worst <= 1.0 and fro <= REL_FRO, (what, worst, fro, float(np.mean(err > 0)))


def _mlp_tensors(M, K, Nup, Nd, seed, up_sparse=True):
    X = synth.act_bf16((seed, M, K), M, K, 0.03, 10.0)
    Wu = synth.gaussian_bf16((seed, 1), (Nup, K), 1.0 / np.sqrt(K))
    LAu = synth.gaussian_bf16((seed, 2), (Nup, 64), 0.02) if up_sparse else None
    LBu = synth.gaussian_bf16((seed, 3), (64, K), 0.02) if up_sparse else None
    Wd = synth.gaussian_bf16((seed, 4), (Nd, Nup), 1.0 / np.sqrt(Nup))
    LAd = synth.gaussian_bf16((seed, 5), (Nd, 64), 0.02)
    LBd = synth.gaussian_bf16((seed, 6), (64, Nup), 0.02)
    return X, Wu, LAu, LBu, Wd, LAd, LBd


def _run_pair(lynx, X, Wu, LAu, LBu, Wd, LAd, LBd, up_sparse, workspace_bytes=None, fuse=True):
    import torch
    Xd = to_dev(X)
    up = lynx.lynx_layer(Xd, to_dev(Wu), None if LAu is None else to_dev(LAu), None if LBu is None else to_dev(LBu),
                         sparse=up_sparse, gelu=True, fuse=fuse)
    dn = lynx.lynx_layer(up["Y"], to_dev(Wd), to_dev(LAd), to_dev(LBd), sparse=True)
    layers = [up, dn]
    need = lynx.lynx_layers_workspace_bytes(layers)
    ws = torch.empty(need if workspace_bytes is None else workspace_bytes, dtype=torch.uint8, device="cuda")
    lynx.lynx_run_layers(layers, ws)
    assert lynx.lynx_sync_status() == 0
    return layers, ws


def _check_pair(lynx, layers, ws, X, Wu, LAu, LBu, Wd, LAd, LBd, up_sparse, rows=None):
    """H against the oracle's H; the fused sparsification (every row) bit for bit against the oracle's on the
    GPU's H; s and T'; Y of the down layer against the oracle on the GPU's H and on the oracle's own H."""
    import torch
    up, dn = layers
    M, K = up["M"], dn["K"]
    H = to_bits(up["Y"])
    rsel = slice(None) if rows is None else rows
    y_ref, H_ref = up_reference(X, Wu, LAu, LBu, up_sparse, rows)
    assert_h_close(H[rsel], y_ref, H_ref)
    off = lynx.lynx_debug_pair_offsets(layers, 0)
    sp = O.sparsify(H)
    vals = ws[off["vals"]:off["vals"] + M * K].view(torch.bfloat16).view(M, K // 2)
    meta = ws[off["meta"]:off["meta"] + lynx.lynx_meta_bytes(M, K)].cpu().numpy()
    s = ws[off["s"]:off["s"] + 4 * M].view(torch.float32).cpu().numpy()
    T = ws[off["T"]:off["T"] + 2 * 64 * M].view(torch.bfloat16).view(M, 64)
    assert np.array_equal(to_bits(vals), sp["vals"])
    assert np.array_equal(meta, pack_meta_reference(sp["meta"], M, K))  # every byte, padding included
    np.testing.assert_allclose(s, sp["s"], rtol=S_RTOL, atol=0)
    assert_y_close(to_bits(T)[rsel], O.lora_down(H[rsel], LBd, sp["s"][rsel]), "T'")
    Y = to_bits(dn["Y"])[rsel]
    st = assert_y_close(Y, O.linear(H[rsel], Wd, LAd, LBd), "Y on the GPU's H")
    # The chain against the oracle's own H: the selection is discontinuous, so a one-ulp difference of H near a
    # tie keeps another channel of the group and multiplies another column of W; only the relative Frobenius
    # error stays small (within 2 x 5e-3).
    y_chain = O.linear(H_ref, Wd, LAd, LBd)
    fro = float(np.linalg.norm(widen(Y) - y_chain) / np.linalg.norm(y_chain))
    assert fro <= 2 * REL_FRO, ("Y on the oracle's H", fro, st)


@pytest.mark.parametrize("tile", [(512, 224), (512, 192), (256, 256), (256, 192)])
@pytest.mark.parametrize("M,K,Nup,Nd", [(300, 256, 512, 200), (129, 512, 384, 264), (600, 384, 1024, 512)])
def test_fused_pair_sparse_up(lynx, M, K, Nup, Nd, tile):
    t = _mlp_tensors(M, K, Nup, Nd, seed=M + Nup)
    lynx.lynx_debug_force_tile(*tile)
    try:
        layers, ws = _run_pair(lynx, *t, up_sparse=True)
        _check_pair(lynx, layers, ws, *t, up_sparse=True)
    finally:
        lynx.lynx_debug_force_tile(0, 0)


def test_fused_pair_down_stream_k(lynx):
    """The fused pair with the down layer's GEMM on the stream-K schedule (forced; 256 x 192 tiles: 3 x 16 = 48
    tiles of 8 k-steps on the CTA pairs): its partials and arrival counters in the pair's workspace plan."""
    M, K, Nup, Nd = 600, 384, 1024, 3072
    t = _mlp_tensors(M, K, Nup, Nd, seed=43)
    lynx.lynx_debug_force_tile(256, 192)
    lynx.lynx_debug_force_ksplit(lynx.LYNX_KSPLIT_STREAM)
    try:
        assert lynx.lynx_debug_linear_ksplit(M, Nd, Nup) == lynx.LYNX_KSPLIT_STREAM
        layers, ws = _run_pair(lynx, *t, up_sparse=True)
        _check_pair(lynx, layers, ws, *t, up_sparse=True)
    finally:
        lynx.lynx_debug_force_ksplit(0)
        lynx.lynx_debug_force_tile(0, 0)


@pytest.mark.parametrize("tile", [256, 448])
@pytest.mark.parametrize("M,K,Nup,Nd", [(300, 256, 512, 200), (1, 128, 256, 64), (640, 512, 1024, 3072)])
def test_fused_pair_dense_up(lynx, M, K, Nup, Nd, tile):
    t = _mlp_tensors(M, K, Nup, Nd, seed=7 * M + Nup, up_sparse=False)
    lynx.lynx_debug_force_dense_tile(tile)
    try:
        layers, ws = _run_pair(lynx, *t, up_sparse=False)
    finally:
        lynx.lynx_debug_force_dense_tile(0)
    # the down layer run on its own (its own sparsify pass) on the same H: the same selection; only the fp32
    # order of the row-norm sums and of the LoRA down-projection differs
    up, dn = layers
    Y_alone = lynx.lynx_linear(up["Y"], dn["W"], dn["LA"], dn["LB"])
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y_alone), O.linear(to_bits(up["Y"]), t[4], t[5], t[6]), "down layer alone on the GPU's H")
    _check_pair(lynx, layers, ws, *t, up_sparse=False)


@pytest.mark.parametrize("how", ["small workspace", "no fuse flag"])
def test_fused_pair_equals_unfused_selection_and_y(lynx, how):
    """Without the fuse flag, or with a workspace too small for the fused plan, the pair runs unfused (the GELU
    epilogue, then the down layer's own sparsify pass): the same H, the same Y within tolerance (only the fp32
    summation order of the row norms differs)."""
    M, K, Nup, Nd = 384, 512, 1024, 256
    t = _mlp_tensors(M, K, Nup, Nd, seed=41)
    fused, ws = _run_pair(lynx, *t, up_sparse=True)
    small = max(lynx.lynx_workspace_bytes(M, Nup, K), lynx.lynx_workspace_bytes(M, Nd, Nup))
    assert small < lynx.lynx_debug_pair_offsets(fused, 0)["total"]
    if how == "small workspace":
        unfused, _ = _run_pair(lynx, *t, up_sparse=True, workspace_bytes=small)
    else:
        unfused, _ = _run_pair(lynx, *t, up_sparse=True, fuse=False)
        with pytest.raises(lynx.LynxError):
            lynx.lynx_debug_pair_offsets(unfused, 0)
        assert lynx.lynx_layers_workspace_bytes(unfused) == small
    assert np.array_equal(to_bits(fused[0]["Y"]), to_bits(unfused[0]["Y"]))
    yf, yu = to_bits(fused[1]["Y"]), to_bits(unfused[1]["Y"])
    assert_y_close(yf, widen(yu), "fused vs unfused")
    assert np.mean(yf == yu) > 0.98
    rows = np.arange(0, M, 7)
    assert_y_close(yu[rows], O.linear(to_bits(unfused[0]["Y"])[rows], t[4], t[5], t[6]), "unfused Y on the GPU's H")


def test_gelu_layer_alone(lynx):
    """A GELU layer followed by a dense layer does not fuse: Y = bf16(GELU(bf16(y)))."""
    import torch
    M, K, N = 300, 512, 640
    X, W, LA, LB, W2, _, _ = _mlp_tensors(M, K, N, 128, seed=5)
    l1 = lynx.lynx_layer(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB), sparse=True, gelu=True)
    l2 = lynx.lynx_layer(l1["Y"], to_dev(W2), sparse=False, gelu=True)
    with pytest.raises(lynx.LynxError):
        lynx.lynx_debug_pair_offsets([l1, l2], 0)
    lynx.lynx_run_layers([l1, l2])
    assert lynx.lynx_sync_status() == 0
    H1 = to_bits(l1["Y"])
    assert_h_close(H1, *up_reference(X, W, LA, LB, True))
    assert_h_close(to_bits(l2["Y"]), *up_reference(H1, W2, None, None, False), "dense GELU layer")
    torch.cuda.synchronize()


def test_mlp_pair_full_size(lynx):
    """The MLP pair of the DiT workload at 4608 tokens (up 3072 -> 12288 sparse with LoRA, GELU, down 12288 ->
    3072 sparse with LoRA), chained through lynx_run_layers: every row of the fused sparsification bit for bit,
    sampled rows of H and Y against the oracle (rows are independent)."""
    t = synth.layer_tensors("mlp", "up")
    d = synth.layer_tensors("mlp", "down", with_x=False)
    args = (t["X"], t["W"], t["LA"], t["LB"], d["W"], d["LA"], d["LB"])
    layers, ws = _run_pair(lynx, *args, up_sparse=True)
    rows = synth.sample_rows((3, 4608, 0, 9), 4608, n=256)
    _check_pair(lynx, layers, ws, *args, up_sparse=True, rows=rows)


@pytest.mark.parametrize("M", [1024, 4608])
def test_stack_mlp_pair_dense_up(lynx, M):
    """The block stack's MLP: dense up (selectively skipped, no LoRA) with GELU, then the sparse down layer."""
    t = synth.layer_tensors("stack", "up", M=M)
    d = synth.layer_tensors("stack", "down", M=M, with_x=False)
    args = (t["X"], t["W"], None, None, d["W"], d["LA"], d["LB"])
    layers, ws = _run_pair(lynx, *args, up_sparse=False)
    rows = synth.sample_rows((5, M, 0, 9), M, n=256)
    _check_pair(lynx, layers, ws, *args, up_sparse=False, rows=rows)


def test_fused_pair_in_a_graph(lynx):
    """A captured sequence with a fused pair replays the same bits as the eager run."""
    import torch
    M, K, Nup, Nd = 300, 256, 512, 200
    t = _mlp_tensors(M, K, Nup, Nd, seed=77)
    layers, ws = _run_pair(lynx, *t, up_sparse=True)
    ref = [to_bits(l["Y"]) for l in layers]
    g = lynx.LynxGraph(layers, ws)
    try:
        for l in layers:
            l["Y"].zero_()
        g.launch()
        assert lynx.lynx_sync_status() == 0
        for i, l in enumerate(layers):
            assert np.array_equal(to_bits(l["Y"]), ref[i]), i
    finally:
        torch.cuda.synchronize()
        g.close()
