"""The five DiT workloads at full size, run exactly as the bench launches them
(one lynx_linear / lynx_linear_dense call per layer on the current stream).

Rows are independent, so Y is compared with the oracle on seeded sampled rows
(512 random rows plus the first and last 64); the sparsification outputs are
compared bit-exactly on every row for the workloads whose oracle pass fits in
host memory, and on the sampled rows otherwise."""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import S_RTOL, assert_y_close, to_bits, to_dev

pytestmark = pytest.mark.gpu


def _run_layer(lynx, wl, layer, M=None, block=0, full_sparsify=True):
    t = synth.layer_tensors(wl, layer, M=M, block=block)
    X, W, LA, LB = t["X"], t["W"], t["LA"], t["LB"]
    M, N, K = t["M"], t["N"], t["K"]
    Xd = to_dev(X)
    if t["sparse"]:
        Y = lynx.lynx_linear(Xd, to_dev(W), to_dev(LA), to_dev(LB))
    else:
        Y = lynx.lynx_linear_dense(Xd, to_dev(W))
    assert lynx.lynx_sync_status() == 0
    rows = synth.sample_rows((WL_SEED[wl], M, block, len(layer)), M)
    Yb = to_bits(Y)[rows]
    if t["sparse"]:
        ref = O.linear(X, W, LA, LB, rows=rows)
    else:
        ref = O.linear_dense(X, W, rows=rows)
    st = assert_y_close(Yb, ref, f"{wl}/{layer}/M={M}/block={block}")
    if t["sparse"]:
        vals, meta, s = lynx.lynx_sparsify(Xd)
        assert lynx.lynx_sync_status() == 0
        sel = slice(None) if full_sparsify else rows
        ref_sp = O.sparsify(X[sel])
        canon = lynx.lynx_meta_to_canonical(meta.cpu().numpy(), M, K)
        assert np.array_equal(to_bits(vals)[sel], ref_sp["vals"])
        assert np.array_equal(canon[sel], ref_sp["meta"])
        np.testing.assert_allclose(s.cpu().numpy()[sel], ref_sp["s"], rtol=S_RTOL, atol=0)
    return st


WL_SEED = {k: v.seed for k, v in synth.WORKLOADS.items()}


def test_tiny_full(lynx):
    t = synth.layer_tensors("tiny", "linear")
    Y = lynx.lynx_linear(*(to_dev(t[k]) for k in ("X", "W", "LA", "LB")))
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y), O.linear(t["X"], t["W"], t["LA"], t["LB"]))


def test_qkv(lynx):
    _run_layer(lynx, "qkv", "qkv")


@pytest.mark.parametrize("layer", ["up", "down"])
def test_mlp_pair(lynx, layer):
    _run_layer(lynx, "mlp", layer)


@pytest.mark.parametrize("layer", ["qkv", "out", "up", "down"])
def test_cfg_batch2(lynx, layer):
    _run_layer(lynx, "cfg2", layer, full_sparsify=(layer != "down"))


@pytest.mark.parametrize("M", synth.STACK_M)
@pytest.mark.parametrize("layer", ["qkv", "out", "up", "down"])
def test_block_stack(lynx, M, layer):
    _run_layer(lynx, "stack", layer, M=M, block=0, full_sparsify=(M * 12288 <= 4608 * 12288))


@pytest.mark.parametrize("layer", ["qkv", "down"])
def test_block_stack_last_block(lynx, layer):
    _run_layer(lynx, "stack", layer, M=4608, block=7)
