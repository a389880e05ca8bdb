"""Layer sequences (a block stack with a selectively skipped dense layer) through lynx_run_layers and through
a captured CUDA graph: each layer reads the previous layer's output, the results equal the per-call results
bit for bit, and the oracle accepts every layer given the same inputs."""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import assert_y_close, to_bits, to_dev

pytestmark = pytest.mark.gpu

M = 300  # ragged: one full 256-row tile pair and a partial one


def _weights(seed):
    """sparse 512 -> 384, dense 384 -> 256, dense + LoRA 256 -> 528, sparse 528 -> 200."""
    shapes = [(True, 384, 512, True), (False, 256, 384, False), (False, 528, 256, True), (True, 200, 528, True)]
    out = []
    for i, (sparse, N, K, lora) in enumerate(shapes):
        W = synth.gaussian_bf16((seed, i, 1), (N, K), 1.0 / np.sqrt(K))
        LA = synth.gaussian_bf16((seed, i, 2), (N, 64), 0.02) if lora else None
        LB = synth.gaussian_bf16((seed, i, 3), (64, K), 0.02) if lora else None
        out.append((sparse, W, LA, LB))
    return out


def _chain(lynx, X, wts):
    """Device layers whose inputs are the previous layers' outputs."""
    layers, x = [], X
    for sparse, W, LA, LB in wts:
        l = lynx.lynx_layer(x, to_dev(W), None if LA is None else to_dev(LA), None if LB is None else to_dev(LB),
                            sparse=sparse)
        layers.append(l)
        x = l["Y"]
    return layers


def _eager(lynx, layers):
    outs, x = [], layers[0]["X"]
    for l in layers:
        if l["sparse"]:
            y = lynx.lynx_linear(x, l["W"], l["LA"], l["LB"])
        else:
            y = lynx.lynx_linear_dense(x, l["W"], l["LA"], l["LB"])
        outs.append(y)
        x = y
    return outs


@pytest.fixture(params=[0, 448], ids=["dense_tile_auto", "dense_tile_448"])
def dense_tile(request, lynx):
    """The dense layers' tile: chosen by shape, or the 448-column collector tile forced on every dense layer."""
    lynx.lynx_debug_force_dense_tile(request.param)
    yield request.param
    lynx.lynx_debug_force_dense_tile(0)


def test_run_layers_and_graph_match_per_call_results(lynx, dense_tile):
    import torch
    wts = _weights(11)
    X = to_dev(synth.act_bf16((M, 512, 11), M, 512, 0.05, 8.0))
    layers = _chain(lynx, X, wts)

    ref = _eager(lynx, layers)
    assert lynx.lynx_sync_status() == 0

    lynx.lynx_run_layers(layers)
    assert lynx.lynx_sync_status() == 0
    for i, (l, r) in enumerate(zip(layers, ref)):
        assert torch.equal(l["Y"], r), f"run_layers layer {i}"

    g = lynx.LynxGraph(layers)
    try:
        for rep in range(2):
            for l in layers:
                l["Y"].zero_()
            g.launch()
            assert lynx.lynx_sync_status() == 0
            for i, (l, r) in enumerate(zip(layers, ref)):
                assert torch.equal(l["Y"], r), f"graph replay {rep} layer {i}"
        # a replay reads the inputs' current contents: a new X gives that X's results
        X.copy_(to_dev(synth.act_bf16((M, 512, 12), M, 512, 0.05, 8.0)))
        g.launch()
        assert lynx.lynx_sync_status() == 0
        ref2 = _eager(lynx, layers)
        assert lynx.lynx_sync_status() == 0
        for i, (l, r) in enumerate(zip(layers, ref2)):
            assert torch.equal(l["Y"], r), f"graph replay with new X, layer {i}"
    finally:
        torch.cuda.synchronize()
        g.close()

    # every layer against the oracle on the inputs it actually read
    x_bits = to_bits(X)
    for i, ((sparse, W, LA, LB), l) in enumerate(zip(wts, layers)):
        want = O.linear(x_bits, W, LA, LB) if sparse else O.linear_dense(x_bits, W, LA, LB)
        assert_y_close(to_bits(l["Y"]), want, f"layer {i}")
        x_bits = to_bits(l["Y"])


def test_graph_rejects_a_bad_layer_without_capturing(lynx):
    import torch
    wts = _weights(13)
    X = to_dev(synth.act_bf16((M, 512, 13), M, 512, 0.05, 8.0))
    layers = _chain(lynx, X, wts)
    layers[2] = dict(layers[2], K=250)  # K % 16 != 0
    with pytest.raises(lynx.LynxError) as e:
        lynx.LynxGraph(layers)
    assert e.value.status == -2 and "layer 2" in str(e.value)
    # the stream is still usable: a valid sequence runs
    lynx.lynx_run_layers(_chain(lynx, X, wts))
    assert lynx.lynx_sync_status() == 0
    torch.cuda.synchronize()
